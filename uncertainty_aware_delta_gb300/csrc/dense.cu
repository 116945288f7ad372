// Dense-covariance (exact) Kalman memory forward (sm_103a).
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
// head.
//
// Two passes.  (1) The covariance recurrence, which is not associative in a
// closed form that chunks, runs token by token, one CTA per head, and writes
// the gains kappa_t.  Given the gains, the mean recurrence S = D S + kappa (v -
// (D S)^T k)^T is the delta rule with write key kappa, so (2) runs it chunkwise:
// the fused tensor-core kernel's given-gains instance (bf16 io, d = 128) or the
// CUDA-core chunk pass (every other case).
//
// The covariance pass keeps the decay out of the per-token work: with G_t the
// running product of the decays since the last renormalisation, P_t =
// G_t Ptil_t G_t, and one token is
//     Ptil_hat = Ptil + diag(omega / g^2),   w = G k,   y = Ptil_hat w,
//     z = w . y,   s = 1 / (r + z),   kappa = s G y,   Ptil <- Ptil_hat - s y y^T
// (G y = P_hat k = u, so G (Ptil_hat - s y y^T) G = P_hat - kappa u^T): one
// matrix-vector product and one rank-1 downdate, 2 d^2 multiply-adds.  When a
// channel's running decay would fall below 2^-20 the token's G is folded into
// Ptil (Ptil <- G Ptil G) and G restarts from 1, so omega / g^2 stays bounded.
// The diagonal increments diag(omega / g^2) are kept in a per-row accumulator
// beside the register block and folded in at the end and at each
// renormalisation.
//
// CTA (b, h), 4 d threads: warp w owns rows 8w .. 8w+7 of Ptil, lane l the
// columns C l .. C l + C - 1 (C = d / 32), in registers for the whole sequence;
// the running decay of each channel is formed once, by the thread that stages
// its inputs, and read from shared memory by the others.
// Per token: the row products with w and their warp reduce-scatter (the four
// lanes of a row end with its sum and keep its diagonal accumulator), z through
// shared memory (the token's one barrier, which also carries the renormalisation
// decision for the next token), the downdate and kappa.  Inputs are loaded from
// global memory kPF tokens ahead into registers (the token loop is unrolled by
// kPF so every register slot has a fixed name) and written to shared memory one
// token ahead, so no global-memory latency sits on a token.  fp32 arithmetic
// throughout.

#include <cuda_bf16.h>

#include "common.cuh"
#include "kdn_internal.h"

namespace kdn {
namespace {

constexpr int kRowsPerWarp = 8;
constexpr float kRenormFloor = 9.5367431640625e-07f;   // 2^-20
constexpr int kPF = 4;   // tokens of inputs in flight (register slots)

// This lane's C consecutive columns from shared memory in one vector load (lane l
// reads words C l .. C l + C - 1: conflict-free, where C scalar loads of stride C
// would hit C-way bank conflicts).
template <int C>
__device__ __forceinline__ void load_cols(const float* p, float (&x)[C]) {
    if constexpr (C == 4) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else if constexpr (C == 2) {
        const float2 v = *reinterpret_cast<const float2*>(p);
        x[0] = v.x; x[1] = v.y;
    } else {
#pragma unroll
        for (int c = 0; c < C; ++c) x[c] = p[c];
    }
}

template <int D, typename TIO>
__global__ void __launch_bounds__(4 * D) dense_cov_kernel(DenseArgs a, float* __restrict__ kappa) {
    constexpr int C = D / 32, W = D / kRowsPerWarp;
    // per-token inputs in three buffers (token t in buffer t % 3): k, the running decay
    // G_{t-1} a_t (before the token's renormalisation, if it has one), omega; y and the
    // warps' partial sums of z in two (token parity).  A buffer is rewritten only after
    // every thread has passed a later barrier than its last read, so one barrier per
    // token suffices.
    __shared__ __align__(16) float s_in[3][3][D];
    __shared__ float s_r[3];
    __shared__ __align__(16) float s_y[2][D];
    __shared__ __align__(16) float s_zpart[2][W];

    const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i0 = warp * kRowsPerWarp, j0 = lane * C;
    // the row whose full sum (and diagonal accumulator) this lane holds after the reduce-scatter
    const int rho = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
    // per-channel duties (staging, running decay, kappa): channel ch = tid on the first D
    // threads (whole warps, so the other warps issue none of this code)
    const bool stager = tid < D;
    const int ch = tid;
    const TIO* k = static_cast<const TIO*>(a.k);
    const size_t ts = static_cast<size_t>(a.H) * D;   // token stride of [B, T, H, d]
    const size_t row0 = static_cast<size_t>(b) * a.T * ts + static_cast<size_t>(h) * D;
    const size_t sb = static_cast<size_t>(bh) * D * D;

    float P[kRowsPerWarp][C];   // Ptil without its diagonal increments
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const size_t e = sb + static_cast<size_t>(i0 + r) * D + j0 + c;
            P[r][c] = a.P0 ? a.P0[e] : (i0 + r == j0 + c ? 1.0f : 0.0f);
        }
    float gs = 1.0f;     // stagers: running decay of channel ch after the current token
    float dacc = 0.0f;   // diagonal increment of row i0 + rho (the same on its four lanes)
    bool folded = false; // the last token renormalised (its G is 1)

    // register slots of the prefetched inputs (stagers): k, log_alpha, omega of channel ch
    // and r (channel 0) of one token each
    float fk[kPF], fl[kPF], fw[kPF], fr[kPF];
    auto fetch = [&](int t, float& k_, float& l_, float& w_, float& r_) {
        if (stager && t < a.T) {
            const size_t e = row0 + static_cast<size_t>(t) * ts + ch;
            k_ = IO<TIO>::load(k, e);
            l_ = a.log_alpha[e];
            w_ = a.omega[e];
            if (ch == 0) r_ = a.r[(static_cast<size_t>(b) * a.T + t) * a.H + h];
        }
    };
    // a token's inputs into buffer t % 3, with the running decay G_{t-1} a_t of channel
    // ch; returns whether it falls below the floor (the token then renormalises)
    auto put = [&](int t, float k_, float l_, float w_, float r_) -> bool {
        bool need = false;
        if (stager) {
            const int bt = t % 3;
            float* buf = &s_in[bt][0][0];
            const float gn = gs * expf(l_);
            buf[0 * D + ch] = k_;
            buf[1 * D + ch] = gn;
            buf[2 * D + ch] = w_;
            if (ch == 0) s_r[bt] = r_;
            need = !(gn >= kRenormFloor);
        }
        return need;
    };
#pragma unroll
    for (int u = 0; u < kPF; ++u) fetch(u, fk[u], fl[u], fw[u], fr[u]);
    bool renorm = __syncthreads_or(a.T > 0 ? put(0, fk[0], fl[0], fw[0], fr[0]) : false);
    fetch(kPF, fk[0], fl[0], fw[0], fr[0]);

#pragma unroll 1
    for (int t0 = 0; t0 < a.T; t0 += kPF)
#pragma unroll
    for (int u = 0; u < kPF; ++u) {
        const int t = t0 + u;
        if (t >= a.T) break;
        const int bt = t % 3, pt = t & 1;
        const float* kin = s_in[bt][0];
        const float* gin = s_in[bt][1];
        const float* win = s_in[bt][2];
        // ---- decay: G_t = G_{t-1} diag(a_t); on renormalisation G_t goes into Ptil and
        //      restarts from 1
        float gc[C], g_rho;
        load_cols<C>(gin + j0, gc);
        if (renorm) {
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const float gi = gin[i0 + r];
#pragma unroll
                for (int c = 0; c < C; ++c) P[r][c] *= gi * gc[c];
            }
            const float gd = gin[i0 + rho];
            dacc *= gd * gd;
#pragma unroll
            for (int c = 0; c < C; ++c) gc[c] = 1.0f;
            g_rho = 1.0f;
            gs = 1.0f;
        } else {
            g_rho = gin[i0 + rho];
            if (stager) gs = gin[ch];
        }
        folded = renorm;
        // ---- Ptil_hat = Ptil + diag(omega / g^2); y = Ptil_hat w, w = G k
        dacc += __fdividef(win[i0 + rho], g_rho * g_rho);
        float wc[C];
        load_cols<C>(kin + j0, wc);
#pragma unroll
        for (int c = 0; c < C; ++c) wc[c] *= gc[c];
        float rs[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            float acc = 0.0f;
#pragma unroll
            for (int c = 0; c < C; ++c) acc = fmaf(P[r][c], wc[c], acc);
            rs[r] = acc;
        }
        // reduce-scatter over the lanes: lane bits 4, 3, 2 pick the row, then full sums
        // over the four lanes that share it
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
        const float w_rho = g_rho * kin[i0 + rho];
        const float y = rs[0] + dacc * w_rho;   // row i0 + rho of Ptil_hat w
        float zp = y * w_rho;                   // the same on the 4 lanes of a row
        zp += __shfl_xor_sync(0xffffffffu, zp, 4);
        zp += __shfl_xor_sync(0xffffffffu, zp, 8);
        zp += __shfl_xor_sync(0xffffffffu, zp, 16);
        if ((lane & 3) == 0) s_y[pt][i0 + rho] = y;
        if (lane == 0) s_zpart[pt][warp] = zp;
        // the next token's inputs (slot (u + 1) % kPF, fetched kPF - 1 tokens ago), whether it
        // renormalises, and the fetch of token t + kPF + 1 into that slot once written
        const int un = (u + 1) % kPF;   // (a constant once the loop over u is unrolled)
        const bool need = t + 1 < a.T ? put(t + 1, fk[un], fl[un], fw[un], fr[un]) : false;
        fetch(t + kPF + 1, fk[un], fl[un], fw[un], fr[un]);
        renorm = __syncthreads_or(need);   // 1
        // ---- gain s = 1 / (r + z), kappa = s G y, downdate Ptil -= s y y^T
        float z4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int w4 = 0; w4 < W / 4; ++w4) {
            const float4 zz = *reinterpret_cast<const float4*>(s_zpart[pt] + 4 * w4);
            z4[0] += zz.x;
            z4[1] += zz.y;
            z4[2] += zz.z;
            z4[3] += zz.w;
        }
        const float z = (z4[0] + z4[1]) + (z4[2] + z4[3]);
        const float sg = __frcp_rn(s_r[bt] + z);
        float yr[kRowsPerWarp], yc[C];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) yr[r] = sg * s_y[pt][i0 + r];
        load_cols<C>(s_y[pt] + j0, yc);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int c = 0; c < C; ++c) P[r][c] = fmaf(-yr[r], yc[c], P[r][c]);
        if (stager) kappa[row0 + static_cast<size_t>(t) * ts + ch] = sg * gs * s_y[pt][ch];
    }
    // final covariance P_T = G (Ptil + diag(dacc)) G with G of the last token (1 when it
    // renormalised, or for T = 0): the register blocks first (each thread writes the
    // block it read, so in-place resume is safe), then the diagonal increments, after
    // a barrier
    const float* gl = s_in[a.T > 0 ? (a.T - 1) % 3 : 0][1];   // the last token's buffer
    const bool unit = a.T == 0 || folded;
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const size_t e = sb + static_cast<size_t>(i0 + r) * D + j0 + c;
            a.P_T[e] = unit ? P[r][c] : P[r][c] * gl[i0 + r] * gl[j0 + c];   // (once)
        }
    __syncthreads();
    if ((lane & 3) == 0) {
        const float gd = unit ? 1.0f : gl[i0 + rho];
        const size_t e = sb + static_cast<size_t>(i0 + rho) * (D + 1);
        a.P_T[e] += dacc * gd * gd;
    }
}

template <int D>
cudaError_t launch_d(const DenseArgs& a, float* kappa, cudaStream_t s) {
    const int grid = a.B * a.H;
    if (grid == 0) return cudaSuccess;
    if (a.io == 1)
        dense_cov_kernel<D, __nv_bfloat16><<<grid, 4 * D, 0, s>>>(a, kappa);
    else
        dense_cov_kernel<D, float><<<grid, 4 * D, 0, s>>>(a, kappa);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dense_covariance(const DenseArgs& a, float* kappa, cudaStream_t s) {
    switch (a.d) {
        case 32: return launch_d<32>(a, kappa, s);
        case 64: return launch_d<64>(a, kappa, s);
        case 128: return launch_d<128>(a, kappa, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kdn
