// Moebius 2x2 gain scan (CUDA-core path).
//
// KDN paper Sec. 4.1 Eq. 32-37: with information scaling, the per-channel
// posterior variance follows a fractional-linear (Moebius) map
//     p_t = (a_t^2 p_{t-1} + w_t) / (u_t a_t^2 p_{t-1} + 1 + u_t w_t),
//     u_t = mu k_t^2 / r_t,
// i.e. [n; d]_t = M_t [n; d]_{t-1} with M_t = [[a^2, w], [u a^2, 1 + u w]] and
// p = n / d.  Matrix products associate (but do not commute), so the
// recurrence is evaluated as a chunked scan, the structure of the paper's
// App. D gain pass: (A) ordered product of each chunk's matrices,
// (B) exclusive carry over the chunks, (C) replay inside each chunk from its
// carry, emitting the gains
//     p_hat_t = a_t^2 p_{t-1} + w_t,   kappa_t = p_hat_t k_t / (r_t + sum_i p_hat_t,i k_t,i^2).
// All matrix entries are positive, so products have no cancellation; they are
// rescaled by exact powers of two after every token, which leaves n / d
// unchanged (App. D's max-abs renormalisation, done without rounding).
//
// The Isotropic variant (Sec. 4.2 Eq. 40, App. C) runs the same three phases
// on one scalar per head, with a_t = mean_i a_t,i^2 (trace projection) and
// u_t = mu ||k_t||^2 / (d_k r_t); its gain is kappa_t = beta_t k_t.

#include "common.cuh"
#include "kdn_internal.h"

namespace kdn {
namespace {

// Exact power-of-two rescale of a matrix with non-negative entries: the largest
// entry lands in [1, 2) (read from its exponent bits; a zero matrix stays zero).
__device__ __forceinline__ void renorm4(float& m00, float& m01, float& m10, float& m11) {
    const float mx = fmaxf(fmaxf(m00, m01), fmaxf(m10, m11));
    const int ex = min(max((__float_as_int(mx) >> 23) & 0xff, 1), 253);
    const float s = __int_as_float((254 - ex) << 23);   // 2^(127 - ex)
    m00 *= s; m01 *= s; m10 *= s; m11 *= s;
}

// ---------------------------------------------------------------- diagonal
template <typename TIO>
__global__ void mobius_summary_diag(const TIO* __restrict__ k, const float* __restrict__ la,
                                    const float* __restrict__ om, const float* __restrict__ r,
                                    int Tn, int H, int dk, float mu, int Cg, int nG,
                                    float* __restrict__ summary) {
    const int bh = blockIdx.x, c = blockIdx.y, b = bh / H, h = bh % H;
    const int i = threadIdx.x;
    if (i >= dk) return;
    const int t0 = c * Cg, t1 = min(Tn, t0 + Cg);
    float m00 = 1.f, m01 = 0.f, m10 = 0.f, m11 = 1.f;
    // (the loads of a few tokens are independent of the product: unrolled, they
    //  are issued ahead of it)
#pragma unroll 4
    for (int t = t0; t < t1; ++t) {
        const size_t th = ((size_t)b * Tn + t) * H + h;
        const float kv = IO<TIO>::load(k, th * dk + i);
        const float a2 = expf(2.0f * la[th * dk + i]);
        const float w = om[th * dk + i];
        const float u = mu * kv * kv / r[th];
        // P <- M_t P (newest on the left)
        const float n00 = a2 * m00 + w * m10;
        const float n01 = a2 * m01 + w * m11;
        const float n10 = u * a2 * m00 + (1.0f + u * w) * m10;
        const float n11 = u * a2 * m01 + (1.0f + u * w) * m11;
        m00 = n00; m01 = n01; m10 = n10; m11 = n11;
        renorm4(m00, m01, m10, m11);
    }
    float4 out = make_float4(m00, m01, m10, m11);
    reinterpret_cast<float4*>(summary)[((size_t)bh * nG + c) * dk + i] = out;
}

// Four channels of one chunk per thread (16-byte loads of log_alpha and omega,
// 8- or 16-byte loads of k), one warp per (sequence, gain chunk), four chunks per
// block: a quarter of the memory requests of the kernel above, four independent
// products per thread.  Needs d_k % 4 == 0, d_k <= 128 and 16-byte aligned rows.
template <typename TIO>
__device__ __forceinline__ void load_k4(const TIO* k, size_t i, float (&kv)[4]);
template <>
__device__ __forceinline__ void load_k4<float>(const float* k, size_t i, float (&kv)[4]) {
    const float4 x = *reinterpret_cast<const float4*>(k + i);
    kv[0] = x.x; kv[1] = x.y; kv[2] = x.z; kv[3] = x.w;
}
template <>
__device__ __forceinline__ void load_k4<__nv_bfloat16>(const __nv_bfloat16* k, size_t i, float (&kv)[4]) {
    const uint2 x = *reinterpret_cast<const uint2*>(k + i);
    kv[0] = __uint_as_float(x.x << 16); kv[1] = __uint_as_float(x.x & 0xffff0000u);
    kv[2] = __uint_as_float(x.y << 16); kv[3] = __uint_as_float(x.y & 0xffff0000u);
}

template <typename TIO>
__global__ void __launch_bounds__(128, 8) mobius_summary_diag4(const TIO* __restrict__ k, const float* __restrict__ la,
                                                          const float* __restrict__ om, const float* __restrict__ r,
                                                          int Tn, int H, int dk, float mu, int Cg, int nG,
                                                          float* __restrict__ summary) {
    const int bh = blockIdx.x, c = blockIdx.y * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int b = bh / H, h = bh % H;
    if (c >= nG) return;   // (whole warps)
    const int i0 = 4 * lane;
    const bool act = i0 < dk;
    const int t0 = c * Cg, t1 = min(Tn, t0 + Cg);
    float m[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        m[j][0] = 1.f; m[j][1] = 0.f; m[j][2] = 0.f; m[j][3] = 1.f;
    }
    for (int tb = t0; tb < t1; tb += 32) {
        const int nt = min(32, t1 - tb);
        // mu / r of 32 tokens, one per lane
        const float mr = mu / (lane < nt ? r[((size_t)b * Tn + tb + lane) * H + h] : 1.0f);
#pragma unroll 4
        for (int u = 0; u < nt; ++u) {
            const float mu_r = __shfl_sync(0xffffffffu, mr, u);
            if (act) {
                const size_t e = (((size_t)b * Tn + tb + u) * H + h) * dk + i0;
                const float4 l4 = *reinterpret_cast<const float4*>(la + e);
                const float4 w4 = *reinterpret_cast<const float4*>(om + e);
                float kv[4];
                load_k4<TIO>(k, e, kv);
                const float lj[4] = {l4.x, l4.y, l4.z, l4.w}, wj[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float a2 = expf(2.0f * lj[j]), w = wj[j], uc = mu_r * kv[j] * kv[j];
                    // P <- M_t P (newest on the left)
                    const float n00 = a2 * m[j][0] + w * m[j][2];
                    const float n01 = a2 * m[j][1] + w * m[j][3];
                    const float n10 = uc * a2 * m[j][0] + (1.0f + uc * w) * m[j][2];
                    const float n11 = uc * a2 * m[j][1] + (1.0f + uc * w) * m[j][3];
                    m[j][0] = n00; m[j][1] = n01; m[j][2] = n10; m[j][3] = n11;
                    renorm4(m[j][0], m[j][1], m[j][2], m[j][3]);
                }
            }
        }
    }
    if (act) {
        float4* out = reinterpret_cast<float4*>(summary) + ((size_t)bh * nG + c) * dk + i0;
#pragma unroll
        for (int j = 0; j < 4; ++j) out[j] = make_float4(m[j][0], m[j][1], m[j][2], m[j][3]);
    }
}

__global__ void mobius_carry(const float* __restrict__ summary, const float* __restrict__ p0,
                             float p_default, int BH, int nu, int nG, float* __restrict__ carry) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;  // (bh, channel)
    if (e >= BH * nu) return;
    const int bh = e / nu, i = e % nu;
    float p = p0 ? p0[e] : p_default;
    const float4* sm4 = reinterpret_cast<const float4*>(summary);
    // the chunk summaries do not depend on the carry: load eight ahead of the chain
    constexpr int kAhead = 8;
    int c = 0;
    for (; c + kAhead <= nG; c += kAhead) {
        float4 m[kAhead];
#pragma unroll
        for (int u = 0; u < kAhead; ++u) m[u] = sm4[((size_t)bh * nG + c + u) * nu + i];
#pragma unroll
        for (int u = 0; u < kAhead; ++u) {
            carry[((size_t)bh * nG + c + u) * nu + i] = p;
            p = (m[u].x * p + m[u].y) / (m[u].z * p + m[u].w);
        }
    }
    for (; c < nG; ++c) {
        const size_t idx = ((size_t)bh * nG + c) * nu + i;
        carry[idx] = p;
        const float4 m = sm4[idx];
        p = (m.x * p + m.y) / (m.z * p + m.w);
    }
}

constexpr int kReplayGroup = 8;  // tokens whose channel sums are reduced together

template <typename TIO>
__global__ void gain_replay_diag(const TIO* __restrict__ k, const float* __restrict__ la,
                                 const float* __restrict__ om, const float* __restrict__ r,
                                 const float* __restrict__ carry, int Tn, int H, int dk, float mu,
                                 int Cg, int nG, float* __restrict__ kappa, float* __restrict__ p_T) {
    __shared__ float red[4][kReplayGroup];  // per warp partial sums (dk <= 128)
    const int bh = blockIdx.x, c = blockIdx.y, b = bh / H, h = bh % H;
    const int i = threadIdx.x, lane = i & 31, warp = i >> 5, nwarps = blockDim.x >> 5;
    const bool act = i < dk;
    float p = act ? carry[((size_t)bh * nG + c) * dk + i] : 0.f;
    const int t0 = c * Cg, t1 = min(Tn, t0 + Cg);
    for (int tb = t0; tb < t1; tb += kReplayGroup) {
        float ph[kReplayGroup], kv[kReplayGroup], w[kReplayGroup];
#pragma unroll
        for (int j = 0; j < kReplayGroup; ++j) {
            const int t = tb + j;
            ph[j] = 0.f; kv[j] = 0.f; w[j] = 0.f;
            if (act && t < t1) {
                const size_t th = ((size_t)b * Tn + t) * H + h;
                kv[j] = IO<TIO>::load(k, th * dk + i);
                const float a2 = expf(2.0f * la[th * dk + i]);
                ph[j] = a2 * p + om[th * dk + i];
                w[j] = ph[j] * kv[j] * kv[j];
                const float u = mu * kv[j] * kv[j] / r[th];
                p = ph[j] / (1.0f + u * ph[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < kReplayGroup; ++j) {
            const float s = warp_sum(w[j]);
            if (lane == 0) red[warp][j] = s;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kReplayGroup; ++j) {
            const int t = tb + j;
            float z = 0.f;
            for (int q = 0; q < nwarps; ++q) z += red[q][j];
            if (act && t < t1) {
                const size_t th = ((size_t)b * Tn + t) * H + h;
                kappa[th * dk + i] = ph[j] * kv[j] / (r[th] + z);
            }
        }
        __syncthreads();
    }
    if (act && c == nG - 1) p_T[(size_t)bh * dk + i] = p;
}

// ---------------------------------------------------------------- isotropic
// Per-token channel reductions a_bar_t = mean_i exp(2 log_alpha_t,i) and
// ||k_t||^2, one warp per token, into shared memory.
template <typename TIO>
__device__ void iso_token_stats(const TIO* __restrict__ k, const float* __restrict__ la, int b,
                                int h, int Tn, int H, int dk, int t0, int t1, float* abar,
                                float* kn2) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int t = t0 + warp; t < t1; t += nwarps) {
        const size_t th = ((size_t)b * Tn + t) * H + h;
        float sa = 0.f, sk = 0.f;
        for (int i = lane; i < dk; i += 32) {
            sa += expf(2.0f * la[th * dk + i]);
            const float kv = IO<TIO>::load(k, th * dk + i);
            sk += kv * kv;
        }
        sa = warp_sum(sa);
        sk = warp_sum(sk);
        if (lane == 0) {
            abar[t - t0] = sa / (float)dk;
            kn2[t - t0] = sk;
        }
    }
}

template <typename TIO>
__global__ void mobius_summary_iso(const TIO* __restrict__ k, const float* __restrict__ la,
                                   const float* __restrict__ om, const float* __restrict__ r,
                                   int Tn, int H, int dk, float mu, int Cg, int nG,
                                   float* __restrict__ summary) {
    extern __shared__ float sm[];
    float* abar = sm;
    float* kn2 = sm + Cg;
    const int bh = blockIdx.x, c = blockIdx.y, b = bh / H, h = bh % H;
    const int t0 = c * Cg, t1 = min(Tn, t0 + Cg);
    iso_token_stats(k, la, b, h, Tn, H, dk, t0, t1, abar, kn2);
    __syncthreads();
    if (threadIdx.x != 0) return;
    float m00 = 1.f, m01 = 0.f, m10 = 0.f, m11 = 1.f;
    for (int t = t0; t < t1; ++t) {
        const size_t th = ((size_t)b * Tn + t) * H + h;
        const float a = abar[t - t0], w = om[th];
        const float u = mu * kn2[t - t0] / ((float)dk * r[th]);
        const float n00 = a * m00 + w * m10;
        const float n01 = a * m01 + w * m11;
        const float n10 = u * a * m00 + (1.0f + u * w) * m10;
        const float n11 = u * a * m01 + (1.0f + u * w) * m11;
        m00 = n00; m01 = n01; m10 = n10; m11 = n11;
        renorm4(m00, m01, m10, m11);
    }
    reinterpret_cast<float4*>(summary)[(size_t)bh * nG + c] = make_float4(m00, m01, m10, m11);
}

template <typename TIO>
__global__ void gain_replay_iso(const TIO* __restrict__ k, const float* __restrict__ la,
                                const float* __restrict__ om, const float* __restrict__ r,
                                const float* __restrict__ carry, int Tn, int H, int dk, float mu,
                                int Cg, int nG, float* __restrict__ kappa,
                                float* __restrict__ p_T) {
    extern __shared__ float sm[];
    float* abar = sm;
    float* kn2 = sm + Cg;
    float* beta = sm + 2 * Cg;
    const int bh = blockIdx.x, c = blockIdx.y, b = bh / H, h = bh % H;
    const int t0 = c * Cg, t1 = min(Tn, t0 + Cg);
    iso_token_stats(k, la, b, h, Tn, H, dk, t0, t1, abar, kn2);
    __syncthreads();
    if (threadIdx.x == 0) {
        float p = carry[(size_t)bh * nG + c];
        for (int t = t0; t < t1; ++t) {
            const size_t th = ((size_t)b * Tn + t) * H + h;
            const float ph = abar[t - t0] * p + om[th];
            beta[t - t0] = ph / (r[th] + ph * kn2[t - t0]);
            const float u = mu * kn2[t - t0] / ((float)dk * r[th]);
            p = ph / (1.0f + u * ph);
        }
        if (c == nG - 1) p_T[bh] = p;
    }
    __syncthreads();
    const int n = (t1 - t0) * dk;
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
        const int tt = e / dk, i = e % dk;
        const size_t th = ((size_t)b * Tn + t0 + tt) * H + h;
        kappa[th * dk + i] = beta[tt] * IO<TIO>::load(k, th * dk + i);
    }
}

// ---------------------------------------------------------------- PKDA
// Preconditioned DeltaNet (Sec. 2.4 Eq. 9, Sec. 2.6): the per-channel key
// statistic A_t = alpha_p_t A_{t-1} + beta_p_t k_t^2 is affine, i.e. the
// Moebius matrix [[alpha_p, beta_p k^2], [0, 1]], so it rides the same three
// phases; its chunk summary is (prod alpha_p, the chunk's decayed sum), the
// pages' chunk formula for the statistic.  The replay emits the write keys
//     kappa_t = beta_t exp(-log(x) softsign(log max(A_t, floor) - mu_h)) k_t.
constexpr float kStatFloor = 1e-20f;

template <typename TIO>
__global__ void stat_summary_pkda(const TIO* __restrict__ k, const float* __restrict__ alpha_p,
                                  const float* __restrict__ beta_p, int Tn, int H, int dk, int Cg,
                                  int nG, float* __restrict__ summary) {
    const int bh = blockIdx.x, c = blockIdx.y, b = bh / H, h = bh % H;
    const int i = threadIdx.x;
    if (i >= dk) return;
    const int t0 = c * Cg, t1 = min(Tn, t0 + Cg);
    float prod = 1.0f, acc = 0.0f;
#pragma unroll 4
    for (int t = t0; t < t1; ++t) {
        const size_t th = ((size_t)b * Tn + t) * H + h;
        const float kv = IO<TIO>::load(k, th * dk + i);
        const float ap = alpha_p[th];
        acc = fmaf(ap, acc, beta_p[th] * kv * kv);
        prod *= ap;
    }
    reinterpret_cast<float4*>(summary)[((size_t)bh * nG + c) * dk + i] = make_float4(prod, acc, 0.0f, 1.0f);
}

template <typename TIO>
__global__ void gain_replay_pkda(const TIO* __restrict__ k, const float* __restrict__ beta,
                                 const float* __restrict__ alpha_p, const float* __restrict__ beta_p,
                                 const float* __restrict__ center, float neg_log2x,
                                 const float* __restrict__ carry, int Tn, int H, int dk, int Cg,
                                 int nG, float* __restrict__ kappa, float* __restrict__ A_T) {
    const int bh = blockIdx.x, c = blockIdx.y, b = bh / H, h = bh % H;
    const int i = threadIdx.x;
    if (i >= dk) return;
    float A = carry[((size_t)bh * nG + c) * dk + i];
    const float mu = center[h];
    const int t0 = c * Cg, t1 = min(Tn, t0 + Cg);
    for (int t = t0; t < t1; ++t) {
        const size_t th = ((size_t)b * Tn + t) * H + h;
        const float kv = IO<TIO>::load(k, th * dk + i);
        A = fmaf(alpha_p[th], A, beta_p[th] * kv * kv);
        const float rho = logf(fmaxf(A, kStatFloor)) - mu;
        const float sg = rho / (1.0f + fabsf(rho));
        kappa[th * dk + i] = beta[th] * exp2f(neg_log2x * sg) * kv;
    }
    if (c == nG - 1) A_T[(size_t)bh * dk + i] = A;
}

template <typename TIO>
cudaError_t launch_scan_t(const ForwardArgs& a, const ScanWorkspace& w, bool replay, cudaStream_t s) {
    const TIO* k = static_cast<const TIO*>(a.k);
    const int BH = a.B * a.H, Cg = w.chunk_g, nG = w.n_chunks_g;
    const dim3 grid(BH, nG);
    if (a.variant == 2) {
        const int nt = ((a.dk + 31) / 32) * 32;
        stat_summary_pkda<TIO><<<grid, nt, 0, s>>>(k, a.alpha_p, a.beta_p, a.T, a.H, a.dk, Cg, nG, w.summary);
        const int tot = BH * a.dk;
        mobius_carry<<<(tot + 127) / 128, 128, 0, s>>>(w.summary, a.p0, 0.0f, BH, a.dk, nG, w.carry);
        if (replay)
            gain_replay_pkda<TIO><<<grid, nt, 0, s>>>(k, a.beta, a.alpha_p, a.beta_p, a.center, a.neg_log2x,
                                                  w.carry, a.T, a.H, a.dk, Cg, nG, w.kappa, a.p_T);
    } else if (a.variant == 0) {
        const int nt = ((a.dk + 31) / 32) * 32;
        if (a.dk % 4 == 0 && a.dk <= 128)
            mobius_summary_diag4<TIO><<<dim3(BH, (nG + 3) / 4), 128, 0, s>>>(k, a.log_alpha, a.omega, a.r, a.T, a.H,
                                                                            a.dk, a.mu, Cg, nG, w.summary);
        else
            mobius_summary_diag<TIO><<<grid, nt, 0, s>>>(k, a.log_alpha, a.omega, a.r, a.T, a.H, a.dk,
                                                         a.mu, Cg, nG, w.summary);
        const int tot = BH * a.dk;
        mobius_carry<<<(tot + 127) / 128, 128, 0, s>>>(w.summary, a.p0, 1.0f, BH, a.dk, nG, w.carry);
        if (replay)
            gain_replay_diag<TIO><<<grid, nt, 0, s>>>(k, a.log_alpha, a.omega, a.r, w.carry, a.T, a.H,
                                                  a.dk, a.mu, Cg, nG, w.kappa, a.p_T);
    } else {
        mobius_summary_iso<TIO><<<grid, 128, 2 * Cg * sizeof(float), s>>>(
            k, a.log_alpha, a.omega, a.r, a.T, a.H, a.dk, a.mu, Cg, nG, w.summary);
        mobius_carry<<<(BH + 127) / 128, 128, 0, s>>>(w.summary, a.p0, 1.0f, BH, 1, nG, w.carry);
        if (replay)
            gain_replay_iso<TIO><<<grid, 128, 3 * Cg * sizeof(float), s>>>(
            k, a.log_alpha, a.omega, a.r, w.carry, a.T, a.H, a.dk, a.mu, Cg, nG, w.kappa, a.p_T);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gain_scan(const ForwardArgs& a, const ScanWorkspace& w, cudaStream_t s) {
    if (a.io == 1) return launch_scan_t<__nv_bfloat16>(a, w, true, s);
    return launch_scan_t<float>(a, w, true, s);
}

cudaError_t launch_scan_carries(const ForwardArgs& a, const ScanWorkspace& w, cudaStream_t s) {
    if (a.io == 1) return launch_scan_t<__nv_bfloat16>(a, w, false, s);
    return launch_scan_t<float>(a, w, false, s);
}

}  // namespace kdn
