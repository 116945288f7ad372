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
// channel's running decay would fall below 2^-20 the running G is folded into
// Ptil (Ptil <- G Ptil G) and G restarts from 1, so omega / g^2 stays bounded
// (for any one token's decay a above 2^-20).
// The diagonal increments diag(omega / g^2) are kept in a per-row accumulator
// beside the register block and folded in at the end and at each
// renormalisation.
//
// Tokens go in pairs (t, t+1), so that one pass over the register block of Ptil
// serves two matrix-vector products and one barrier serves two tokens.  With
// y_t = (Ptil + diag(dacc_t)) w_t (Ptil before the pair) is the first token's y,
// and the second token's y is the product with the downdated matrix,
//     y_{t+1} = v - s_t (y_t . w_{t+1}) y_t,   v = (Ptil + diag(dacc_{t+1})) w_{t+1},
//     z_{t+1} = w_{t+1} . v - s_t (y_t . w_{t+1})^2,
// so the three dot products z_t, y_t . w_{t+1} and w_{t+1} . v are reduced together,
// and then Ptil -= s_t y_t y_t^T + s_{t+1} y_{t+1} y_{t+1}^T.  A renormalisation that
// the pair's second token needs happens at the pair's start (folding early is exact).
//
// CTA (b, h), 4 d threads: warp w owns rows 8w .. 8w+7 of Ptil, lane l the
// columns C l .. C l + C - 1 (C = d / 32), in registers for the whole sequence;
// the running decay of each channel is formed once, by the thread that stages
// its inputs, and read from shared memory by the others.
// Per pair: the row products with both w and their warp reduce-scatter (the four
// lanes of a row end with its sums and keep its diagonal accumulator), the three
// dot products through shared memory (the pair's one barrier, which also carries
// the renormalisation decision for the next pair), the rank-2 downdate and the
// two tokens' kappa.  Inputs are loaded from global memory kPP pairs ahead into
// registers (the pair loop is unrolled by kPP so every register slot has a fixed
// name) and written to shared memory one pair ahead, so no global-memory latency
// sits on a pair.  fp32 arithmetic throughout.

#include <cuda_bf16.h>

#include "common.cuh"
#include "kdn_internal.h"
#include "mma_tf32x3.cuh"

namespace kdn {
namespace {

constexpr int kRowsPerWarp = 8;
constexpr float kRenormFloor = 9.5367431640625e-07f;   // 2^-20
constexpr int kPP = 2;   // token pairs of inputs in flight (register slots)

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
    // per-pair inputs in three buffers (pair p in buffer p % 3): k and omega of its two
    // tokens, the running decays G_{t-1} a_t and G_{t-1} a_t a_{t+1} (before the pair's
    // renormalisation, if it has one) and a_{t+1}; y_t, the second token's unreduced
    // product and the warps' partial sums of the three scalars in two (pair parity).  A
    // buffer is rewritten only after every thread has passed a later barrier than its
    // last read, so one barrier per pair suffices.
    __shared__ __align__(16) float s_in[3][7][D];
    __shared__ float s_r[3][2];
    __shared__ __align__(16) float s_u[2][D];
    __shared__ __align__(16) float s_v[2][D];
    __shared__ __align__(16) float s_zpart[2][3][W];
    enum { IK0 = 0, IK1, IW0, IW1, IG0, IG1, IA1 };

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
    const int npairs = (a.T + 1) / 2;

    float P[kRowsPerWarp][C];   // Ptil without its diagonal increments
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) {
            const size_t e = sb + static_cast<size_t>(i0 + r) * D + j0 + c;
            P[r][c] = a.P0 ? a.P0[e] : (i0 + r == j0 + c ? 1.0f : 0.0f);
        }
    float gs = 1.0f;     // stagers: running decay of channel ch after the current pair
    float dacc = 0.0f;   // diagonal increment of row i0 + rho (the same on its four lanes)
    bool folded = false; // the last pair renormalised at its start

    // register slots of the prefetched inputs (stagers): k, log_alpha, omega of channel ch
    // and r (channel 0) of the two tokens of one pair each.  A token past T reads as
    // k = 0, log_alpha = 0, omega = 0, r = 1: it changes nothing (zero gain, no decay,
    // no noise), so an odd T ends on a pair with an empty second token.
    float fk[kPP][2], fl[kPP][2], fw[kPP][2], fr[kPP][2];
    auto fetch = [&](int pp, float (&k_)[2], float (&l_)[2], float (&w_)[2], float (&r_)[2]) {
        if (stager) {
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
                const int t = 2 * pp + e2;
                k_[e2] = 0.0f;
                l_[e2] = 0.0f;
                w_[e2] = 0.0f;
                r_[e2] = 1.0f;
                if (t < a.T) {
                    const size_t e = row0 + static_cast<size_t>(t) * ts + ch;
                    k_[e2] = IO<TIO>::load(k, e);
                    l_[e2] = a.log_alpha[e];
                    w_[e2] = a.omega[e];
                    if (ch == 0) r_[e2] = a.r[(static_cast<size_t>(b) * a.T + t) * a.H + h];
                }
            }
        }
    };
    // a pair's inputs into buffer pp % 3 with the running decays of channel ch; returns
    // whether the second token's falls below the floor (the pair then renormalises at
    // its start: G_{t-1} a_t goes into Ptil and the second token's decay is a_{t+1})
    auto put = [&](int pp, const float (&k_)[2], const float (&l_)[2], const float (&w_)[2],
                   const float (&r_)[2]) -> bool {
        bool need = false;
        if (stager) {
            const int bt = pp % 3;
            const float g0 = gs * expf(l_[0]), a1 = expf(l_[1]), g1 = g0 * a1;
            s_in[bt][IK0][ch] = k_[0];
            s_in[bt][IK1][ch] = k_[1];
            s_in[bt][IW0][ch] = w_[0];
            s_in[bt][IW1][ch] = w_[1];
            s_in[bt][IG0][ch] = g0;
            s_in[bt][IG1][ch] = g1;
            s_in[bt][IA1][ch] = a1;
            if (ch == 0) {
                s_r[bt][0] = r_[0];
                s_r[bt][1] = r_[1];
            }
            need = !(g1 >= kRenormFloor);
        }
        return need;
    };
#pragma unroll
    for (int u = 0; u < kPP; ++u) fetch(u, fk[u], fl[u], fw[u], fr[u]);
    bool renorm = __syncthreads_or(npairs > 0 ? put(0, fk[0], fl[0], fw[0], fr[0]) : false);
    fetch(kPP, fk[0], fl[0], fw[0], fr[0]);

#pragma unroll 1
    for (int p0 = 0; p0 < npairs; p0 += kPP)
#pragma unroll
    for (int u = 0; u < kPP; ++u) {
        const int pp = p0 + u;
        if (pp >= npairs) break;
        const int t = 2 * pp, bt = pp % 3, pt = pp & 1;
        const float* in = &s_in[bt][0][0];
        // ---- decays of the two tokens: G_t = G_{t-1} diag(a_t), G_{t+1} = G_t diag(a_{t+1});
        //      on renormalisation G_t goes into Ptil, and G_t = 1, G_{t+1} = diag(a_{t+1})
        float gc0[C], gc1[C], g0r, g1r;
        load_cols<C>(in + IG0 * D + j0, gc0);
        if (renorm) {
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                const float gi = in[IG0 * D + i0 + r];
#pragma unroll
                for (int c = 0; c < C; ++c) P[r][c] *= gi * gc0[c];
            }
            const float gd = in[IG0 * D + i0 + rho];
            dacc *= gd * gd;
#pragma unroll
            for (int c = 0; c < C; ++c) gc0[c] = 1.0f;
            load_cols<C>(in + IA1 * D + j0, gc1);
            g0r = 1.0f;
            g1r = in[IA1 * D + i0 + rho];
            if (stager) gs = in[IA1 * D + ch];
        } else {
            load_cols<C>(in + IG1 * D + j0, gc1);
            g0r = in[IG0 * D + i0 + rho];
            g1r = in[IG1 * D + i0 + rho];
            if (stager) gs = in[IG1 * D + ch];
        }
        folded = renorm;
        // ---- diagonal increments omega / g^2 of the two tokens; w = G k
        const float dacc0 = dacc + __fdividef(in[IW0 * D + i0 + rho], g0r * g0r);
        const float dacc1 = dacc0 + __fdividef(in[IW1 * D + i0 + rho], g1r * g1r);
        dacc = dacc1;
        float wa[C], wb[C];
        load_cols<C>(in + IK0 * D + j0, wa);
        load_cols<C>(in + IK1 * D + j0, wb);
#pragma unroll
        for (int c = 0; c < C; ++c) {
            wa[c] *= gc0[c];
            wb[c] *= gc1[c];
        }
        // ---- both products with the same Ptil: Ptil w_t and Ptil w_{t+1}
        float ru[kRowsPerWarp], rv[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            float au = 0.0f, av = 0.0f;
#pragma unroll
            for (int c = 0; c < C; ++c) {
                au = fmaf(P[r][c], wa[c], au);
                av = fmaf(P[r][c], wb[c], av);
            }
            ru[r] = au;
            rv[r] = av;
        }
        // reduce-scatter over the lanes: lane bits 4, 3, 2 pick the row, then full sums
        // over the four lanes that share it
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool hi = lane & 16;
            const float su = hi ? ru[j] : ru[j + 4], ku = hi ? ru[j + 4] : ru[j];
            const float sv = hi ? rv[j] : rv[j + 4], kv = hi ? rv[j + 4] : rv[j];
            ru[j] = ku + __shfl_xor_sync(0xffffffffu, su, 16);
            rv[j] = kv + __shfl_xor_sync(0xffffffffu, sv, 16);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const bool hi = lane & 8;
            const float su = hi ? ru[j] : ru[j + 2], ku = hi ? ru[j + 2] : ru[j];
            const float sv = hi ? rv[j] : rv[j + 2], kv = hi ? rv[j + 2] : rv[j];
            ru[j] = ku + __shfl_xor_sync(0xffffffffu, su, 8);
            rv[j] = kv + __shfl_xor_sync(0xffffffffu, sv, 8);
        }
        {
            const bool hi = lane & 4;
            const float su = hi ? ru[0] : ru[1], ku = hi ? ru[1] : ru[0];
            const float sv = hi ? rv[0] : rv[1], kv = hi ? rv[1] : rv[0];
            ru[0] = ku + __shfl_xor_sync(0xffffffffu, su, 4);
            rv[0] = kv + __shfl_xor_sync(0xffffffffu, sv, 4);
        }
        ru[0] += __shfl_xor_sync(0xffffffffu, ru[0], 2);
        rv[0] += __shfl_xor_sync(0xffffffffu, rv[0], 2);
        ru[0] += __shfl_xor_sync(0xffffffffu, ru[0], 1);
        rv[0] += __shfl_xor_sync(0xffffffffu, rv[0], 1);
        // rows i0 + rho of y_t = (Ptil + diag(dacc_t)) w_t and of v = (Ptil + diag(dacc_{t+1}))
        // w_{t+1}; the second token's y is v - s_t (y_t . w_{t+1}) y_t (Ptil after the first
        // token's downdate, applied to w_{t+1}), known once s_t is
        const float wa_r = g0r * in[IK0 * D + i0 + rho], wb_r = g1r * in[IK1 * D + i0 + rho];
        const float yu = ru[0] + dacc0 * wa_r;
        const float yv = rv[0] + dacc1 * wb_r;
        // partial sums (the same on the 4 lanes of a row): z_t = w_t . y_t,
        // y_t . w_{t+1}, w_{t+1} . v
        float zq[3] = {yu * wa_r, yu * wb_r, yv * wb_r};
#pragma unroll
        for (int m = 4; m <= 16; m <<= 1)
#pragma unroll
            for (int e3 = 0; e3 < 3; ++e3) zq[e3] += __shfl_xor_sync(0xffffffffu, zq[e3], m);
        if ((lane & 3) == 0) {
            s_u[pt][i0 + rho] = yu;
            s_v[pt][i0 + rho] = yv;
        }
        if (lane == 0) {
            s_zpart[pt][0][warp] = zq[0];
            s_zpart[pt][1][warp] = zq[1];
            s_zpart[pt][2][warp] = zq[2];
        }
        // the next pair's inputs (slot (u + 1) % kPP, fetched kPP - 1 pairs ago), whether it
        // renormalises, and the fetch of pair pp + kPP + 1 into that slot once written
        const int un = (u + 1) % kPP;   // (a constant once the loop over u is unrolled)
        const bool need = pp + 1 < npairs ? put(pp + 1, fk[un], fl[un], fw[un], fr[un]) : false;
        fetch(pp + kPP + 1, fk[un], fl[un], fw[un], fr[un]);
        renorm = __syncthreads_or(need);   // 1
        // ---- the three scalars, the two gains s = 1 / (r + z), y_{t+1}, and the rank-2
        //      downdate Ptil -= s_t y_t y_t^T + s_{t+1} y_{t+1} y_{t+1}^T
        float zs[3];
#pragma unroll
        for (int e3 = 0; e3 < 3; ++e3) {
            float z4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int w4 = 0; w4 < W / 4; ++w4) {
                const float4 zz = *reinterpret_cast<const float4*>(s_zpart[pt][e3] + 4 * w4);
                z4[0] += zz.x;
                z4[1] += zz.y;
                z4[2] += zz.z;
                z4[3] += zz.w;
            }
            zs[e3] = (z4[0] + z4[1]) + (z4[2] + z4[3]);
        }
        const float s0 = __frcp_rn(s_r[bt][0] + zs[0]);
        const float cb = s0 * zs[1];                        // s_t (y_t . w_{t+1})
        const float z1 = fmaf(-cb, zs[1], zs[2]);           // w_{t+1} . y_{t+1}
        const float s1 = __frcp_rn(s_r[bt][1] + z1);
        float yr0[kRowsPerWarp], yr1[kRowsPerWarp], yc0[C], yc1[C];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const float y0 = s_u[pt][i0 + r];
            yr0[r] = y0;
            yr1[r] = fmaf(-cb, y0, s_v[pt][i0 + r]);
        }
        load_cols<C>(s_u[pt] + j0, yc0);
        load_cols<C>(s_v[pt] + j0, yc1);
#pragma unroll
        for (int c = 0; c < C; ++c) yc1[c] = fmaf(-cb, yc0[c], yc1[c]);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const float f0 = s0 * yr0[r], f1 = s1 * yr1[r];
#pragma unroll
            for (int c = 0; c < C; ++c) P[r][c] = fmaf(-f0, yc0[c], fmaf(-f1, yc1[c], P[r][c]));
        }
        if (stager) {
            // kappa = s G y for each token (G_t of channel ch: 1 after a renormalisation)
            const float y0 = s_u[pt][ch], y1 = fmaf(-cb, y0, s_v[pt][ch]);
            const float g0 = folded ? 1.0f : in[IG0 * D + ch];
            kappa[row0 + static_cast<size_t>(t) * ts + ch] = s0 * g0 * y0;
            if (t + 1 < a.T) kappa[row0 + static_cast<size_t>(t + 1) * ts + ch] = s1 * gs * y1;
        }
    }
    // final covariance P_T = G (Ptil + diag(dacc)) G with G the running decay after the
    // last pair (a_{t+1} when that pair renormalised; 1 for T = 0): the register blocks
    // first (each thread writes the block it read, so in-place resume is safe), then the
    // diagonal increments, after a barrier
    const int lb = npairs > 0 ? (npairs - 1) % 3 : 0;
    const float* gl = s_in[lb][folded ? IA1 : IG1];
    const bool unit = a.T == 0;
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

// ---------------------------------------------------------------- d = 128: token blocks
// The same recurrence over blocks of up to 16 tokens, with the products on tensor
// cores (3xTF32 warp-level MMAs, fp32-level accuracy) and Ptil in shared memory.
// In a block of m tokens with decay factors G_j relative to a per-channel reference
// (Ptil = e^{ref} P e^{ref} at the block start), w_j = G_j k_j and dacc_j = sum_{i<=j}
// omega_i / G_i^2, every token's y is a combination of u_j = (Ptil + diag(dacc_j)) w_j:
//     y_j = u_j - sum_{i<j} s_i (y_i . w_j) y_i,   s_j = 1 / (r_j + w_j . y_j).
// With Gamma(l, j) = u_l . w_j, the elimination H(j, .) = Gamma(j, .) - sum_{i<j} s_i
// H(i, j) H(i, .) gives s_j = 1 / (r_j + H(j, j)) and N(j, i) = s_i H(i, j), and
// (I + N) Y = U.  So a block is: U += W Ptil (Ptil symmetric), Gamma = U W^T, the
// 16 x 16 elimination on one warp, Y by forward substitution per channel, kappa_j =
// s_j G_j y_j, and Ptil += diag(dacc) - Y^T diag(s) Y.  The reference is the middle
// of the block's log decay, and a block ends early where some channel's log decay
// would exceed kBlockLogDecay (one token at least; a single token beyond it takes its
// own decay as the reference), so every factor stays within e^{+-20} and Ptil within
// e^{-40} of P.
constexpr int kTB = 16;                   // tokens per block
constexpr int kLP = 132;                  // row stride (floats) of Ptil in shared memory
constexpr int kLT = 132;                  // row stride of the [16][128] token tiles
constexpr float kBlockLogDecay = 40.0f;
constexpr int kBlockThreads = 512;
constexpr size_t kBlockSmem = sizeof(float) * (128 * kLP + 7 * kTB * kLT + kTB * 17 + 2 * kTB + 128 + 4);

template <typename TIO>
__device__ __forceinline__ void load4(const TIO* p, float (&x)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&x)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[4]) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xffff0000u);
    x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xffff0000u);
}

// C[16][c0 + 8 columns] += f_c (A[16][128] B[128][c0 ..]) for one warp: A given as its
// TF32 high and low parts (rows of stride la), B rows of stride lb split here.  3xTF32
// m16n8k8 MMAs whose three products and two halves of the K steps go to six
// accumulators, so the dependent chains are 8 MMAs long instead of 48.
__device__ __forceinline__ void warp_row16_x_panel(const uint32_t* Ah, const uint32_t* Al, int la, const float* B,
                                                   int lb, float* C, int lc, int c0, const float* f) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    float acc[6][4];
#pragma unroll
    for (int u = 0; u < 6; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[u][e] = 0.0f;
#pragma unroll 4
    for (int ks = 0; ks < 16; ++ks) {
        const int k0 = 8 * ks, hk = 3 * (ks & 1);
        const uint32_t ah[4] = {Ah[g * la + k0 + q], Ah[(g + 8) * la + k0 + q], Ah[g * la + k0 + q + 4],
                                Ah[(g + 8) * la + k0 + q + 4]};
        const uint32_t al[4] = {Al[g * la + k0 + q], Al[(g + 8) * la + k0 + q], Al[g * la + k0 + q + 4],
                                Al[(g + 8) * la + k0 + q + 4]};
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(B[(k0 + q) * lb + c0 + g], bh0, bl0);
        split_tf32(B[(k0 + q + 4) * lb + c0 + g], bh1, bl1);
        mma_m16n8k8_tf32(acc[hk + 0], al, bh0, bh1);
        mma_m16n8k8_tf32(acc[hk + 1], ah, bl0, bl1);
        mma_m16n8k8_tf32(acc[hk + 2], ah, bh0, bh1);
    }
    const float f0 = f[c0 + 2 * q], f1 = f[c0 + 2 * q + 1];
    float* d0 = C + g * lc + c0 + 2 * q;
    float* d1 = d0 + 8 * lc;
    d0[0] += f0 * ((acc[0][0] + acc[3][0]) + (acc[1][0] + acc[4][0]) + (acc[2][0] + acc[5][0]));
    d0[1] += f1 * ((acc[0][1] + acc[3][1]) + (acc[1][1] + acc[4][1]) + (acc[2][1] + acc[5][1]));
    d1[0] += f0 * ((acc[0][2] + acc[3][2]) + (acc[1][2] + acc[4][2]) + (acc[2][2] + acc[5][2]));
    d1[1] += f1 * ((acc[0][3] + acc[3][3]) + (acc[1][3] + acc[4][3]) + (acc[2][3] + acc[5][3]));
}

// The block's update of Ptil for one warp (rows 16 (w >> 1) .., columns 64 (w & 1) ..):
//     Ptil <- F Ptil F - (s Y)^T Y
// (the frame change into this block and its rank-16 downdate in one read-modify-write;
// the diagonal increments follow after a barrier), the product on 3xTF32 m16n8k8 MMAs
// (K = 16 tokens).
__device__ __forceinline__ void warp_block_update(const float* Ys, const float* Y, int lt, float* P, int lp,
                                                  const float* f, int warp) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int r0 = 16 * (warp >> 1), cb = 64 * (warp & 1);
    float acc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[n][e] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const int k0 = 8 * ks;
        uint32_t ah[4], al[4];   // A(r, j) = (s y_j)[r]
        split_tf32(Ys[(k0 + q) * lt + r0 + g], ah[0], al[0]);
        split_tf32(Ys[(k0 + q) * lt + r0 + g + 8], ah[1], al[1]);
        split_tf32(Ys[(k0 + q + 4) * lt + r0 + g], ah[2], al[2]);
        split_tf32(Ys[(k0 + q + 4) * lt + r0 + g + 8], ah[3], al[3]);
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int c = cb + 8 * n + g;
            uint32_t bh0, bl0, bh1, bl1;
            split_tf32(Y[(k0 + q) * lt + c], bh0, bl0);
            split_tf32(Y[(k0 + q + 4) * lt + c], bh1, bl1);
            mma_m16n8k8_tf32(acc[n], al, bh0, bh1);
            mma_m16n8k8_tf32(acc[n], ah, bl0, bl1);
            mma_m16n8k8_tf32(acc[n], ah, bh0, bh1);
        }
    }
    const int ra = r0 + g, rb = ra + 8;
    const float fa = f[ra], fb = f[rb];
#pragma unroll
    for (int n = 0; n < 8; ++n) {
        const int c = cb + 8 * n + 2 * q;
        const float fc0 = f[c], fc1 = f[c + 1];
        float* pa = P + ra * lp + c;
        float* pb = P + rb * lp + c;
        pa[0] = fmaf(fa * fc0, pa[0], -acc[n][0]);
        pa[1] = fmaf(fa * fc1, pa[1], -acc[n][1]);
        pb[0] = fmaf(fb * fc0, pb[0], -acc[n][2]);
        pb[1] = fmaf(fb * fc1, pb[1], -acc[n][3]);
    }
}

template <typename TIO>
__global__ void __launch_bounds__(kBlockThreads, 1) dense_cov_block_kernel(DenseArgs a, float* __restrict__ kappa) {
    constexpr int D = 128;
    extern __shared__ float4 dyn_smem4[];
    float* Pt = reinterpret_cast<float*>(dyn_smem4);   // [128][kLP]
    float* sK = Pt + D * kLP;      // [16][kLT] k, then w = G k
    float* sG = sK + kTB * kLT;    // [16][kLT] log_alpha, then G
    float* sO = sG + kTB * kLT;    // [16][kLT] omega, then dacc
    float* sU = sO + kTB * kLT;    // [16][kLT] u, then s y
    float* sY = sU + kTB * kLT;    // [16][kLT] y
    uint32_t* sWh = reinterpret_cast<uint32_t*>(sY + kTB * kLT);   // [16][kLT] w f, TF32 high part
    uint32_t* sWl = sWh + kTB * kLT;                                 // [16][kLT] and low part
    float* sH = reinterpret_cast<float*>(sWl + kTB * kLT);   // [16][17]  Gamma, then N below the diagonal
    float* sR = sH + kTB * 17;     // [16]      r
    float* sS = sR + kTB;          // [16]      s
    float* sF = sS + kTB;          // [128]     scaling of Ptil at the block start
    int* sM = reinterpret_cast<int*>(sF + D);   // tokens in the block

    const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const TIO* kin = static_cast<const TIO*>(a.k);
    const size_t ts = static_cast<size_t>(a.H) * D;
    const size_t row0 = static_cast<size_t>(b) * a.T * ts + static_cast<size_t>(h) * D;
    const size_t sb = static_cast<size_t>(bh) * D * D;

    for (int e = tid; e < D * D / 4; e += kBlockThreads) {
        const int r = e >> 5, c = (e & 31) * 4;
        float4 v;
        if (a.P0) v = *reinterpret_cast<const float4*>(a.P0 + sb + static_cast<size_t>(r) * D + c);
        else v = make_float4(r == c ? 1.f : 0.f, r == c + 1 ? 1.f : 0.f, r == c + 2 ? 1.f : 0.f, r == c + 3 ? 1.f : 0.f);
        *reinterpret_cast<float4*>(Pt + r * kLP + c) = v;
    }
    // staging: token j = warp of a tile, channels 4 lane .. 4 lane + 3; registers hold
    // the next tile while a block runs
    const int sj = warp, sc = 4 * lane;
    float xk[4], xl[4], xw[4], xr = 1.0f;
    auto load_tile = [&](int t0) {
        const int t = t0 + sj;
        if (t < a.T) {
            const size_t e = row0 + static_cast<size_t>(t) * ts + sc;
            load4<TIO>(kin + e, xk);
            load4<float>(a.log_alpha + e, xl);
            load4<float>(a.omega + e, xw);
            xr = a.r[(static_cast<size_t>(b) * a.T + t) * a.H + h];
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) xk[c] = xl[c] = xw[c] = 0.0f;
            xr = 1.0f;
        }
    };
    float prev_end = 0.0f;   // channel tid >> 2: log decay at the end of the last block, relative to its reference
    float dfold = 0.0f;      // channel tid (< 128): the block's diagonal increment
    int t0 = 0;
    if (a.T > 0) load_tile(0);
    while (t0 < a.T) {
        *reinterpret_cast<float4*>(sK + sj * kLT + sc) = make_float4(xk[0], xk[1], xk[2], xk[3]);
        *reinterpret_cast<float4*>(sG + sj * kLT + sc) = make_float4(xl[0], xl[1], xl[2], xl[3]);
        *reinterpret_cast<float4*>(sO + sj * kLT + sc) = make_float4(xw[0], xw[1], xw[2], xw[3]);
        if (lane == 0) sR[sj] = xr;
        if (tid == 0) *sM = min(kTB, a.T - t0);
        __syncthreads();
        // Per-channel work runs on four threads per channel (channel tid >> 2, tokens
        // 4 p .. 4 p + 3 of the tile for p = tid & 3), the sums over tokens as scans over
        // the four lanes.
        const int ci = tid >> 2, cp = tid & 3;
        auto scan4 = [&](float x) {   // inclusive scan over the four lanes of a channel
            float y = __shfl_up_sync(0xffffffffu, x, 1, 4);
            if (cp >= 1) x += y;
            y = __shfl_up_sync(0xffffffffu, x, 2, 4);
            if (cp >= 2) x += y;
            return x;
        };
        // ---- block length: up to the first token whose log decay from the block start
        //      leaves kBlockLogDecay on some channel (the first token always counts)
        {
            float loc[4], acc = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc += sG[(4 * cp + e) * kLT + ci];
                loc[e] = acc;
            }
            const float off = scan4(acc) - acc;
            int mi = kTB;
#pragma unroll
            for (int e = 3; e >= 0; --e) {
                const int j = 4 * cp + e;
                if (j > 0 && !(fabsf(off + loc[e]) <= kBlockLogDecay)) mi = j;
            }
            mi = __reduce_min_sync(0xffffffffu, mi);
            if (lane == 0) atomicMin(sM, mi);
        }
        __syncthreads();
        const int m = *sM;
        // ---- per channel: decay factors G_j about the reference, w = G k, dacc, u = dacc w,
        //      and the scaling of Ptil into this block's frame
        {
            float loc[4], acc = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (4 * cp + e < m) acc += sG[(4 * cp + e) * kLT + ci];
                loc[e] = acc;
            }
            const float incl = scan4(acc), off = incl - acc;
            const float L = __shfl_sync(0xffffffffu, incl, 3, 4);   // log decay of the block's m tokens
            const float ref = fabsf(L) > kBlockLogDecay ? L : 0.5f * L;
            const float fi = expf(ref + prev_end);
            if (cp == 0) sF[ci] = fi;
            prev_end = L - ref;
            float gq[4], wq[4], tq[4], dacc_loc = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = 4 * cp + e;
                gq[e] = 1.0f;
                wq[e] = 0.0f;
                tq[e] = 0.0f;
                if (j < m) {
                    gq[e] = exp2f((off + loc[e] - ref) * 1.4426950408889634f);
                    wq[e] = gq[e] * sK[j * kLT + ci];
                    dacc_loc += __fdividef(sO[j * kLT + ci], gq[e] * gq[e]);
                }
                tq[e] = dacc_loc;
            }
            const float doff = scan4(dacc_loc) - dacc_loc;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = 4 * cp + e;
                const float dd = doff + tq[e];
                sK[j * kLT + ci] = wq[e];
                sG[j * kLT + ci] = gq[e];
                sO[j * kLT + ci] = dd;
                sU[j * kLT + ci] = dd * wq[e];
                uint32_t wh, wl;   // (w f: the product below reads Ptil before its change of frame)
                split_tf32(wq[e] * fi, wh, wl);
                sWh[j * kLT + ci] = wh;
                sWl[j * kLT + ci] = wl;
            }
        }
        if (tid < kTB && tid >= m) sR[tid] = 1.0f;   // (tokens of the tile not in this block)
        if (m == kTB && t0 + kTB < a.T) load_tile(t0 + kTB);
        __syncthreads();
        // ---- U += W (F Ptil F) (warp w: columns 8 w .. 8 w + 7; Ptil still in the last
        //      block's frame)
        warp_row16_x_panel(sWh, sWl, kLT, Pt, kLP, sU, kLT, 8 * warp, sF);
        __syncthreads();
        {   // ---- Gamma(l, j) = u_l . w_j: two threads per entry, each a half of the channels
            //      (interleaved 4-channel groups, so the two halves sit in different banks)
            const int o = tid >> 1, hh = tid & 1, l = o >> 4, j = o & 15;
            const float* ur = sU + l * kLT + 4 * hh;
            const float* wr = sK + j * kLT + 4 * hh;
            float acc = 0.0f;
#pragma unroll
            for (int v = 0; v < 16; ++v) {
                const float4 x = *reinterpret_cast<const float4*>(ur + 8 * v);
                const float4 y = *reinterpret_cast<const float4*>(wr + 8 * v);
                acc = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc))));
            }
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            if (hh == 0) sH[l * 17 + j] = acc;
        }
        __syncthreads();
        // ---- the elimination (warp 0)
        if (warp == 0) {
            float hc[kTB], rr[kTB];   // lane k: column k of H; r
#pragma unroll
            for (int j = 0; j < kTB; ++j) {
                hc[j] = sH[j * 17 + (lane & 15)];
                rr[j] = sR[j];
            }
            __syncwarp();
            float sv = 0.0f;   // lane j: s_j
#pragma unroll
            for (int j = 0; j < kTB; ++j) {
                const float sj_ = __fdividef(1.0f, rr[j] + __shfl_sync(0xffffffffu, hc[j], j));
                if (lane == j) sv = sj_;
                // lane jp > j: N(jp, j) = s_j H(j, jp), its own H(j, jp) (column jp)
                if (lane > j && lane < kTB) sH[lane * 17 + j] = sj_ * hc[j];
#pragma unroll
                for (int jp = j + 1; jp < kTB; ++jp)
                    hc[jp] = fmaf(-sj_ * __shfl_sync(0xffffffffu, hc[j], jp), hc[j], hc[jp]);
            }
            if (lane < kTB) sS[lane] = sv;
        }
        __syncthreads();
        // ---- Y = (I + N)^{-1} U per channel, kappa, s y; diag(dacc) into Ptil
        if (tid < D) {
            const int c = tid;
            float y[kTB];
#pragma unroll
            for (int j = 0; j < kTB; ++j) {
                float acc = sU[j * kLT + c];
#pragma unroll
                for (int i = 0; i < j; ++i) acc = fmaf(-sH[j * 17 + i], y[i], acc);
                y[j] = acc;
            }
#pragma unroll
            for (int j = 0; j < kTB; ++j) {
                const float s = sS[j];
                sY[j * kLT + c] = y[j];
                sU[j * kLT + c] = s * y[j];
                if (j < m) kappa[row0 + static_cast<size_t>(t0 + j) * ts + c] = s * sG[j * kLT + c] * y[j];
            }
            dfold = sO[(kTB - 1) * kLT + c];
        }
        __syncthreads();
        // ---- Ptil <- F Ptil F - (s Y)^T Y, then + diag(dacc)
        warp_block_update(sU, sY, kLT, Pt, kLP, sF, warp);
        t0 += m;
        if (m < kTB && t0 < a.T) load_tile(t0);   // (the prefetched tile started elsewhere)
        __syncthreads();
        if (tid < D) Pt[tid * kLP + tid] += dfold;
    }
    // P_T = E Ptil E, E = e^{log decay at the end of the last block, relative to its reference}
    if ((tid & 3) == 0) sF[tid >> 2] = expf(prev_end);
    __syncthreads();
    for (int e = tid; e < D * D / 4; e += kBlockThreads) {
        const int r = e >> 5, c = (e & 31) * 4;
        const float4 x = *reinterpret_cast<const float4*>(Pt + r * kLP + c);
        const float fr = sF[r];
        *reinterpret_cast<float4*>(a.P_T + sb + static_cast<size_t>(r) * D + c) =
            make_float4(fr * sF[c] * x.x, fr * sF[c + 1] * x.y, fr * sF[c + 2] * x.z, fr * sF[c + 3] * x.w);
    }
}

template <int D>
cudaError_t launch_d(const DenseArgs& a, float* kappa, cudaStream_t s) {
    const int grid = a.B * a.H;
    if (grid == 0) return cudaSuccess;
    if constexpr (D == 128) {
        // token blocks on tensor cores
        auto kern = a.io == 1 ? dense_cov_block_kernel<__nv_bfloat16> : dense_cov_block_kernel<float>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kBlockSmem));
        kern<<<grid, kBlockThreads, kBlockSmem, s>>>(a, kappa);
        return cudaGetLastError();
    }
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
