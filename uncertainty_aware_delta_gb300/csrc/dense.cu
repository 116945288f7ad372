// Dense-covariance (exact) Kalman memory forward, token by token (sm_103a, CUDA cores).
//
// KDN paper Sec. 3.2, Eq. 12-17: per head a mean memory S (d x d, row = key
// channel) and a full key covariance P (d x d); with the diagonal transition
// D_t = diag(a_t), a_t = exp(log_alpha_t), and diagonal process noise
// Omega_t = diag(omega_t), for every token
//     P_hat = D P D + Omega,   u = P_hat k,   z = k^T u,   kappa = u / (r + z)
//     P     = (I - kappa k^T) P_hat = P_hat - kappa u^T      (P_hat symmetric)
//     S_hat = D S,   delta = v - S_hat^T k,   S = S_hat + kappa delta^T
//     o     = S^T q   (read after the write).
// The Diagonal and Isotropic KDN replace P by a diagonal / scalar surrogate;
// this is the filter they approximate, at O(d^2) work and state per token and
// head.  The covariance recurrence is not associative in a closed form that
// chunks, so the tokens of a head run in order on one CTA.
//
// CTA (b, h), 4 d threads: warp w owns rows 8w .. 8w+7 of P and S, lane l the
// columns C l .. C l + C - 1 (C = d / 32); both blocks stay in registers for the
// whole sequence.  Per token: P_hat and its row products with k, and the column
// products of S with a*k, in one local pass; u by a warp reduce-scatter of the
// 8 row sums; z and delta through shared memory (barrier 1, one reduction, barrier
// 2); the local updates of P and S and the column products with q; o through
// shared memory (barrier 3).  The next token's inputs are staged during the
// current one.  fp32 arithmetic throughout.

#include <cuda_bf16.h>

#include "common.cuh"
#include "kdn_internal.h"

namespace kdn {
namespace {

constexpr int kRowsPerWarp = 8;

template <int D, typename TIO>
__global__ void __launch_bounds__(4 * D) dense_forward_kernel(DenseArgs a) {
    constexpr int C = D / 32, W = D / kRowsPerWarp, NT = 4 * D;
    // per-token inputs, double-buffered by token parity: k, q, v, a (decay), omega
    __shared__ __align__(16) float s_in[2][5][D];
    __shared__ float s_r[2];
    __shared__ __align__(16) float s_u[D], s_delta[D];
    __shared__ __align__(16) float s_cpart[W][D], s_opart[W][D];
    __shared__ float s_zpart[W];

    const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i0 = warp * kRowsPerWarp, j0 = lane * C;
    const TIO* q = static_cast<const TIO*>(a.q);
    const TIO* k = static_cast<const TIO*>(a.k);
    const TIO* v = static_cast<const TIO*>(a.v);
    TIO* o = static_cast<TIO*>(a.o);
    const size_t ts = static_cast<size_t>(a.H) * D;   // token stride of [B, T, H, d]
    const size_t row0 = static_cast<size_t>(b) * a.T * ts + static_cast<size_t>(h) * D;
    const size_t sb = static_cast<size_t>(bh) * D * D;

    float P[kRowsPerWarp][C], S[kRowsPerWarp][C];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const size_t e = sb + static_cast<size_t>(i0 + r) * D + j0 + c;
            P[r][c] = a.P0 ? a.P0[e] : (i0 + r == j0 + c ? 1.0f : 0.0f);
            S[r][c] = a.S0 ? a.S0[e] : 0.0f;
        }

    auto stage = [&](int t) {   // inputs of token t into buffer t & 1 (threads 0 .. D-1)
        if (tid < D) {
            const size_t e = row0 + static_cast<size_t>(t) * ts + tid;
            float* buf = &s_in[t & 1][0][0];
            buf[0 * D + tid] = IO<TIO>::load(k, e);
            buf[1 * D + tid] = IO<TIO>::load(q, e);
            buf[2 * D + tid] = IO<TIO>::load(v, e);
            buf[3 * D + tid] = expf(a.log_alpha[e]);
            buf[4 * D + tid] = a.omega[e];
            if (tid == 0) s_r[t & 1] = a.r[(static_cast<size_t>(b) * a.T + t) * a.H + h];
        }
    };
    if (a.T > 0) stage(0);
    __syncthreads();

    for (int t = 0; t < a.T; ++t) {
        const float* kin = s_in[t & 1][0];
        const float* qin = s_in[t & 1][1];
        const float* vin = s_in[t & 1][2];
        const float* ain = s_in[t & 1][3];
        const float* win = s_in[t & 1][4];
        // ---- A: P_hat = D P D + Omega and its row products with k; column products of S with a * k
        float ar[kRowsPerWarp], akr[kRowsPerWarp], ac[C], kc[C];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            ar[r] = ain[i0 + r];
            akr[r] = ar[r] * kin[i0 + r];
        }
#pragma unroll
        for (int c = 0; c < C; ++c) {
            ac[c] = ain[j0 + c];
            kc[c] = kin[j0 + c];
        }
        float rs[kRowsPerWarp], cs[C];
#pragma unroll
        for (int c = 0; c < C; ++c) cs[c] = 0.0f;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            float acc = 0.0f;
#pragma unroll
            for (int c = 0; c < C; ++c) {
                float ph = ar[r] * ac[c] * P[r][c];
                if (i0 + r == j0 + c) ph += win[i0 + r];
                P[r][c] = ph;
                acc = fmaf(ph, kc[c], acc);
                cs[c] = fmaf(akr[r], S[r][c], cs[c]);
            }
            rs[r] = acc;
        }
        // u for the warp's 8 rows: reduce-scatter over the lanes, then full sums over
        // the 4 lanes that share a row (lane bits 4, 3, 2 pick the row)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool hi = lane & 16;
            const float send = hi ? rs[j] : rs[j + 4], keep = hi ? rs[j + 4] : rs[j];
            rs[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const bool hi = lane & 8;
            const float send = hi ? rs[j] : rs[j + 2], keep = hi ? rs[j + 2] : rs[j];
            rs[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
        {
            const bool hi = lane & 4;
            const float send = hi ? rs[0] : rs[1], keep = hi ? rs[1] : rs[0];
            rs[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        rs[0] += __shfl_xor_sync(0xffffffffu, rs[0], 2);
        rs[0] += __shfl_xor_sync(0xffffffffu, rs[0], 1);
        const int rho = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
        float zp = rs[0] * kin[i0 + rho];   // the same on the 4 lanes of a row
        zp += __shfl_xor_sync(0xffffffffu, zp, 4);
        zp += __shfl_xor_sync(0xffffffffu, zp, 8);
        zp += __shfl_xor_sync(0xffffffffu, zp, 16);
        if ((lane & 3) == 0) s_u[i0 + rho] = rs[0];
        if (lane == 0) s_zpart[warp] = zp;
#pragma unroll
        for (int c = 0; c < C; ++c) s_cpart[warp][j0 + c] = cs[c];
        __syncthreads();   // 1
        // ---- B: innovation delta = v - S_hat^T k; next token's inputs
        if (tid < D) {
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < W; ++w) sum += s_cpart[w][tid];
            s_delta[tid] = vin[tid] - sum;
        }
        if (t + 1 < a.T) stage(t + 1);
        __syncthreads();   // 2
        // ---- C: gain, covariance and memory updates, column products with q
        float z = 0.0f;
#pragma unroll
        for (int w = 0; w < W; ++w) z += s_zpart[w];
        const float g = 1.0f / (s_r[t & 1] + z);
        float uc[C], dc[C], os[C];
#pragma unroll
        for (int c = 0; c < C; ++c) {
            uc[c] = s_u[j0 + c];
            dc[c] = s_delta[j0 + c];
            os[c] = 0.0f;
        }
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const float kap = s_u[i0 + r] * g, qr = qin[i0 + r];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                P[r][c] = fmaf(-kap, uc[c], P[r][c]);
                S[r][c] = fmaf(kap, dc[c], ar[r] * S[r][c]);
                os[c] = fmaf(qr, S[r][c], os[c]);
            }
        }
#pragma unroll
        for (int c = 0; c < C; ++c) s_opart[warp][j0 + c] = os[c];
        __syncthreads();   // 3
        // ---- D: o = S^T q
        if (tid < D) {
            float sum = 0.0f;
#pragma unroll
            for (int w = 0; w < W; ++w) sum += s_opart[w][tid];
            IO<TIO>::store(o, row0 + static_cast<size_t>(t) * ts + tid, sum);
        }
    }
    // final state (each thread writes the block it read: in-place resume is safe)
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const size_t e = sb + static_cast<size_t>(i0 + r) * D + j0 + c;
            a.P_T[e] = P[r][c];
            a.S_T[e] = S[r][c];
        }
    (void)NT;
}

template <int D>
cudaError_t launch_d(const DenseArgs& a, cudaStream_t s) {
    const int grid = a.B * a.H;
    if (grid == 0) return cudaSuccess;
    if (a.io == 1)
        dense_forward_kernel<D, __nv_bfloat16><<<grid, 4 * D, 0, s>>>(a);
    else
        dense_forward_kernel<D, float><<<grid, 4 * D, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dense_forward(const DenseArgs& a, cudaStream_t s) {
    switch (a.d) {
        case 32: return launch_d<32>(a, s);
        case 64: return launch_d<64>(a, s);
        case 128: return launch_d<128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kdn
