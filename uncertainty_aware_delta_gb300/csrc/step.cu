// Single-token decode (kdn_step): the recurrent form of the KDN mixer
// (KDN paper Sec. 5.1: training scans and token-by-token inference are the
// same recurrence), with the state (S, p) resident in HBM and updated in place.
//
// Per (sequence, head), one token:
//   a = exp(log_alpha);  Diagonal: p_hat = a^2 p + omega,  kappa = p_hat k / (r + sum p_hat k^2)
//                        Isotropic: b_hat = mean(a^2) b + omega, kappa = k b_hat / (r + b_hat ||k||^2)
//   delta = v - (diag(a) S)^T k                               (innovation, Eq. 13-15)
//   S     = diag(a) S + kappa delta^T                         (Eq. 16)
//   o     = S^T q = (diag(a) S)^T q + delta (kappa . q)       (Eq. 17, read after the write)
//   p     = p_hat / (1 + (mu / r) k^2 p_hat)   (Isotropic: u = mu ||k||^2 / (d_k r))   (Eq. 60-65)
// PKDA (Preconditioned DeltaNet Sec. 2.4 Eq. 9, Sec. 2.5) replaces the gain by
// the write key of the preconditioned delta rule and p by the key statistic A:
//   A = alpha_p A + beta_p k^2;  kappa = beta exp(-log(x) softsign(log A - mu_h)) k.
// The two reductions over the key channel (with a*k and a*q) share one read
// of S; the write pass reuses the values held in registers, so S crosses
// HBM exactly once in each direction, with 128-bit accesses.

#include "common.cuh"
#include "kdn_internal.h"

namespace kdn {
namespace {

constexpr int kStepNT = 256;
constexpr int kMaxRegF4 = 16;  // float4 of S per thread for d_k = d_v = 128
constexpr float kStatFloor = 1e-20f;  // PKDA: the key statistic enters the logarithm no smaller

template <typename TIO>
__global__ void __launch_bounds__(kStepNT, 2)
step_kernel(const TIO* __restrict__ q, const TIO* __restrict__ k, const TIO* __restrict__ v,
            const float* __restrict__ la, const float* __restrict__ om, const float* __restrict__ r,
            float* __restrict__ S, float* __restrict__ p, TIO* __restrict__ o, int variant, int DK,
            int DV, float mu, uint32_t* status, const float* __restrict__ beta,
            const float* __restrict__ alpha_p, const float* __restrict__ beta_p,
            const float* __restrict__ center, float neg_log2x, int H) {
    __shared__ float s_a[128], s_ak[128], s_aq[128], s_kap[128];
    __shared__ float s_red[kStepNT / 32][4];
    // per-thread partial column sums: row groups x DV = (256 / (DV / 4)) * DV = 1024
    __shared__ float s_part[2][4 * kStepNT];
    __shared__ float s_scal[4];

    const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (bh == 0 && tid == 0 && status) *status = 0u;
    // -- the one read of this head's S (128-bit loads), issued first so its latency
    //    overlaps the gain computation below
    const int NC4 = DV / 4;                 // float4 columns
    const int NRG = kStepNT / NC4;          // row groups
    const int c4 = tid % NC4, rg = tid / NC4;
    float4* S4 = reinterpret_cast<float4*>(S + (size_t)bh * DK * DV);
    float4 reg[kMaxRegF4];
#pragma unroll
    for (int m = 0; m < kMaxRegF4; ++m) {
        const int i = rg + m * NRG;
        if (i < DK) reg[m] = S4[(size_t)i * NC4 + c4];
    }
    const size_t vec = (size_t)bh * DK;
    const float rt = variant == 2 ? 1.0f : r[bh];

    // -- gain (uses the predictive variance, before the mu-scaled update)
    float kv = 0.f, qv = 0.f, a = 0.f, a2 = 0.f, ph = 0.f;
    if (tid < DK) {
        kv = IO<TIO>::load(k, vec + tid);
        qv = IO<TIO>::load(q, vec + tid);
        a = expf(la[vec + tid]);
        a2 = a * a;
        s_a[tid] = a;
        s_ak[tid] = a * kv;
        s_aq[tid] = a * qv;
    }
    float x0, x1, x2;
    if (variant == 2) {
        x0 = 0.f;            // no reductions: the write key is per channel
        x1 = 0.f;
        x2 = 0.f;
    } else if (variant == 0) {
        if (tid < DK) ph = a2 * p[vec + tid] + om[vec + tid];
        x0 = ph * kv * kv;   // z
        x1 = 0.f;
        x2 = 0.f;
    } else {
        x0 = a2;             // sum a^2
        x1 = kv * kv;        // ||k||^2
        x2 = kv * qv;        // k . q
    }
    x0 = warp_sum(x0); x1 = warp_sum(x1); x2 = warp_sum(x2);
    if (lane == 0) { s_red[warp][0] = x0; s_red[warp][1] = x1; s_red[warp][2] = x2; }
    __syncthreads();
    if (tid == 0) {
        float y0 = 0.f, y1 = 0.f, y2 = 0.f;
        for (int w = 0; w < kStepNT / 32; ++w) { y0 += s_red[w][0]; y1 += s_red[w][1]; y2 += s_red[w][2]; }
        s_scal[0] = y0; s_scal[1] = y1; s_scal[2] = y2;
    }
    __syncthreads();
    float kap = 0.f;
    if (variant == 2) {
        if (tid < DK) {
            const float A = fmaf(alpha_p[bh], p[vec + tid], beta_p[bh] * kv * kv);
            const float rho = logf(fmaxf(A, kStatFloor)) - center[bh % H];
            kap = beta[bh] * exp2f(neg_log2x * (rho / (1.0f + fabsf(rho)))) * kv;
            p[vec + tid] = A;
        }
    } else if (variant == 0) {
        const float z = s_scal[0];
        if (tid < DK) {
            kap = ph * kv / (rt + z);
            const float u = (mu / rt) * kv * kv;
            p[vec + tid] = ph / (1.0f + u * ph);
        }
    } else {
        const float abar = s_scal[0] / (float)DK, kn2 = s_scal[1];
        const float bhat = abar * p[bh] + om[bh];
        const float gain = bhat / (rt + bhat * kn2);
        if (tid < DK) kap = gain * kv;
        __syncthreads();  // every thread has read p[bh] before it is replaced
        if (tid == 0) {
            const float u = mu * kn2 / ((float)DK * rt);
            p[bh] = bhat / (1.0f + u * bhat);
        }
    }
    if (tid < DK) s_kap[tid] = kap;
    // kappa . q
    float kq = warp_sum(kap * qv);
    __syncthreads();
    if (lane == 0) s_red[warp][3] = kq;
    __syncthreads();
    kq = 0.f;
    for (int w = 0; w < kStepNT / 32; ++w) kq += s_red[w][3];

    // -- per column, sum_i (a_i k_i) S_ij and sum_i (a_i q_i) S_ij from the registers
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < kMaxRegF4; ++m) {
        const int i = rg + m * NRG;
        if (i < DK) {
            const float ak = s_ak[i], aq = s_aq[i];
            pk[0] = fmaf(ak, reg[m].x, pk[0]); pk[1] = fmaf(ak, reg[m].y, pk[1]);
            pk[2] = fmaf(ak, reg[m].z, pk[2]); pk[3] = fmaf(ak, reg[m].w, pk[3]);
            pq[0] = fmaf(aq, reg[m].x, pq[0]); pq[1] = fmaf(aq, reg[m].y, pq[1]);
            pq[2] = fmaf(aq, reg[m].z, pq[2]); pq[3] = fmaf(aq, reg[m].w, pq[3]);
        }
    }
    if (rg < DK) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            s_part[0][rg * DV + c4 * 4 + c] = pk[c];
            s_part[1][rg * DV + c4 * 4 + c] = pq[c];
        }
    }
    __syncthreads();
    __shared__ float s_delta[128];
    if (tid < DV) {
        float sk = 0.f, sq = 0.f;
        const int nrg = NRG < DK ? NRG : DK;
        for (int g = 0; g < nrg; ++g) { sk += s_part[0][g * DV + tid]; sq += s_part[1][g * DV + tid]; }
        const float d = IO<TIO>::load(v, (size_t)bh * DV + tid) - sk;
        s_delta[tid] = d;
        IO<TIO>::store(o, (size_t)bh * DV + tid, sq + d * kq);
    }
    __syncthreads();
    // -- write pass from registers
    const float d0 = s_delta[c4 * 4 + 0], d1 = s_delta[c4 * 4 + 1];
    const float d2 = s_delta[c4 * 4 + 2], d3 = s_delta[c4 * 4 + 3];
#pragma unroll
    for (int m = 0; m < kMaxRegF4; ++m) {
        const int i = rg + m * NRG;
        if (i < DK) {
            const float ai = s_a[i], ki = s_kap[i];
            float4 x = reg[m];
            x.x = fmaf(ai, x.x, ki * d0);
            x.y = fmaf(ai, x.y, ki * d1);
            x.z = fmaf(ai, x.z, ki * d2);
            x.w = fmaf(ai, x.w, ki * d3);
            S4[(size_t)i * NC4 + c4] = x;
        }
    }
}

}  // namespace

cudaError_t launch_step(const StepArgs& a, cudaStream_t s) {
    const int BH = a.B * a.H;
    if (BH == 0) return cudaSuccess;
    const int grid = BH;
    if (a.io == 1)
        step_kernel<__nv_bfloat16><<<grid, kStepNT, 0, s>>>(
            static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
            static_cast<const __nv_bfloat16*>(a.v), a.log_alpha, a.omega, a.r, a.S, a.p,
            static_cast<__nv_bfloat16*>(a.o), a.variant, a.dk, a.dv, a.mu, a.status, a.beta,
            a.alpha_p, a.beta_p, a.center, a.neg_log2x, a.H);
    else
        step_kernel<float><<<grid, kStepNT, 0, s>>>(
            static_cast<const float*>(a.q), static_cast<const float*>(a.k),
            static_cast<const float*>(a.v), a.log_alpha, a.omega, a.r, a.S, a.p,
            static_cast<float*>(a.o), a.variant, a.dk, a.dv, a.mu, a.status, a.beta, a.alpha_p,
            a.beta_p, a.center, a.neg_log2x, a.H);
    return cudaGetLastError();
}

}  // namespace kdn
