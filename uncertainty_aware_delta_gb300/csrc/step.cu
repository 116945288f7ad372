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
#include "kdn.h"
#include "kdn_internal.h"
#include "sm100.cuh"

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

// ---------------------------------------------------------------- d_k = d_v = 128
// Streaming form of the same step for the 128 x 128 state: a persistent CTA per SM
// walks heads bh = blockIdx.x + n * gridDim.x.  Each head's S (64 KB) and its
// per-channel vectors arrive by bulk copy into a ring of three shared-memory
// buffers, two heads ahead of the one being updated, and the updated S leaves by
// bulk store, so HBM reads and writes stay in flight while a head is computed.
constexpr int kPD = 128, kPNT = 256, kRing = 3;
constexpr uint32_t kSBytes = kPD * kPD * 4;
// shared-memory map (floats): ring [3][128 * 128]; staged vectors [3][6][128]
// (q, k, v, log_alpha, omega, p); a, a*k, a*q, kappa, delta [5][128]; column partial
// sums [2][8][128]; warp partials [8][4]; per-head scalars [2][4] by head parity;
// mbarriers [3] of the ring and one that nothing completes (timeout probe)
constexpr int PS_VEC = kRing * kPD * kPD, PS_A = PS_VEC + kRing * 6 * kPD, PS_PART = PS_A + 5 * kPD,
              PS_RED = PS_PART + 2 * 8 * kPD, PS_HS = PS_RED + 32, PS_BAR = PS_HS + 8,
              PS_FLOATS = PS_BAR + 2 * (kRing + 1);
constexpr uint32_t kStreamSmem = PS_FLOATS * 4;
static_assert(PS_BAR % 2 == 0, "mbarriers 8-byte aligned");
constexpr uint32_t kStreamWaitLimit = 1u << 20;
// Bound of the timeout probe's wait (KDN_FLAG_TIMEOUT_PROBE): a few milliseconds.
constexpr uint32_t kProbeWaitLimit = 1u << 12;

template <typename TIO, int V>
__global__ void __launch_bounds__(kPNT, 1)
step_stream_kernel(const TIO* __restrict__ q, const TIO* __restrict__ k, const TIO* __restrict__ v,
                   const float* __restrict__ la, const float* __restrict__ om, const float* __restrict__ r,
                   float* S, float* p, TIO* __restrict__ o, float mu, uint32_t* status,
                   const float* __restrict__ beta, const float* __restrict__ alpha_p,
                   const float* __restrict__ beta_p, const float* __restrict__ center, float neg_log2x,
                   int BH, int H, int probe) {
    using namespace sm100;
    constexpr bool DIAG = V == 0, ISO = V == 1, PK = V == 2;
    extern __shared__ __align__(128) float sm[];
    float* ring = sm;
    float* vec = sm + PS_VEC;
    float *s_a = sm + PS_A, *s_ak = s_a + kPD, *s_aq = s_ak + kPD, *s_kap = s_aq + kPD, *s_delta = s_kap + kPD;
    float* s_part = sm + PS_PART;
    float* s_red = sm + PS_RED;
    float* s_hs = sm + PS_HS;
    const uint32_t ring_s = smem_addr(ring), vec_s = smem_addr(vec), bar_s = smem_addr(sm + PS_BAR);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c4 = tid & 31, rg = tid >> 5;   // float4 column group, row group (rows rg + 8 m)
    const int G = gridDim.x, nh = (BH - static_cast<int>(blockIdx.x) + G - 1) / G;
    const uint32_t bar_probe = bar_s + 8 * kRing;   // completed by nothing (timeout probe)
    if (tid == 0) {
        for (int e = 0; e <= kRing; ++e) mbar_init(bar_s + 8 * e, 1);
        mbar_fence_init();
    }
    __syncthreads();
    constexpr uint32_t kVecBytes = 3 * kPD * sizeof(TIO) + kPD * 4 + (DIAG ? 2 * kPD * 4 : PK ? kPD * 4 : 0);
    // bulk loads of this CTA's head n into ring slot n % 3 (one copy in flight per slot)
    auto issue = [&](int n) {
        const size_t bh = static_cast<size_t>(blockIdx.x) + static_cast<size_t>(n) * G;
        const int slot = n % kRing;
        const uint32_t bar = bar_s + 8 * slot, vb = vec_s + slot * 6 * kPD * 4;
        mbar_expect_tx(bar, kSBytes + kVecBytes);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            bulk_load(ring_s + slot * kSBytes + c * 16384, S + bh * kPD * kPD + c * 4096, 16384, bar);
        bulk_load(vb, q + bh * kPD, kPD * sizeof(TIO), bar);
        bulk_load(vb + 512, k + bh * kPD, kPD * sizeof(TIO), bar);
        bulk_load(vb + 1024, v + bh * kPD, kPD * sizeof(TIO), bar);
        bulk_load(vb + 1536, la + bh * kPD, kPD * 4, bar);
        if (DIAG) bulk_load(vb + 2048, om + bh * kPD, kPD * 4, bar);
        if (DIAG || PK) bulk_load(vb + 2560, p + bh * kPD, kPD * 4, bar);
    };
    // per-head scalars: r (KDN); omega and b (isotropic); beta, alpha_p, beta_p, centre (PKDA)
    auto load_scalars = [&](int n, float (&hs)[4]) {
        const size_t bh = static_cast<size_t>(blockIdx.x) + static_cast<size_t>(n) * G;
        if (PK) {
            hs[0] = beta[bh];
            hs[1] = alpha_p[bh];
            hs[2] = beta_p[bh];
            hs[3] = center[bh % H];
        } else {
            hs[0] = r[bh];
            hs[1] = ISO ? om[bh] : 0.0f;
            hs[2] = ISO ? p[bh] : 0.0f;
            hs[3] = 0.0f;
        }
    };
    float hsn[4] = {0.f, 0.f, 0.f, 0.f};
    if (tid == 0) {
        issue(0);
        if (nh > 1) issue(1);
        load_scalars(0, hsn);
#pragma unroll
        for (int e = 0; e < 4; ++e) s_hs[e] = hsn[e];
    }
    __syncthreads();
    int n = 0;
#pragma unroll 1
    for (; n < nh; ++n) {
        const size_t bh = static_cast<size_t>(blockIdx.x) + static_cast<size_t>(n) * G;
        const int slot = n % kRing;
        if (tid == 0 && n + 1 < nh) load_scalars(n + 1, hsn);   // in flight during this head
        // (timeout probe: the first head's wait is on a barrier that nothing completes,
        //  with a short bound, while that head's copies are in flight)
        const bool ok = (probe && n == 0)
                            ? mbar_wait(bar_probe, 0u, kProbeWaitLimit)
                            : mbar_wait(bar_s + 8 * slot, static_cast<uint32_t>(n / kRing) & 1u, kStreamWaitLimit);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) set_status(status, kStatusTimeout);
            break;
        }
        float* Sb = ring + slot * kPD * kPD;
        const float* vb = vec + slot * 6 * kPD;
        const TIO* vq = reinterpret_cast<const TIO*>(vb);
        const TIO* vk = reinterpret_cast<const TIO*>(vb + kPD);
        const TIO* vv = reinterpret_cast<const TIO*>(vb + 2 * kPD);
        float4 reg[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) reg[m] = *reinterpret_cast<const float4*>(Sb + (rg + 8 * m) * kPD + 4 * c4);
        // ---- per key channel i = tid (warps 0-3): decay, predicted variance, reductions
        float kv = 0.f, qv = 0.f, a = 0.f, ph = 0.f, x0 = 0.f, x1 = 0.f, x2 = 0.f;
        if (tid < kPD) {
            kv = IO<TIO>::load(vk, tid);
            qv = IO<TIO>::load(vq, tid);
            a = expf(vb[3 * kPD + tid]);
            s_a[tid] = a;
            s_ak[tid] = a * kv;
            s_aq[tid] = a * qv;
            if (DIAG) {
                ph = a * a * vb[5 * kPD + tid] + vb[4 * kPD + tid];
                x0 = ph * kv * kv;
            } else if (ISO) {
                x0 = a * a;
                x1 = kv * kv;
                x2 = kv * qv;
            }
        }
        if (!PK && warp < 4) {
            x0 = warp_sum(x0);
            if (ISO) {
                x1 = warp_sum(x1);
                x2 = warp_sum(x2);
            }
            if (lane == 0) {
                s_red[warp * 4 + 0] = x0;
                s_red[warp * 4 + 1] = x1;
                s_red[warp * 4 + 2] = x2;
            }
        }
        __syncthreads();
        const float* hs = s_hs + (n & 1) * 4;
        float kap = 0.f;
        if (tid < kPD) {
            if (DIAG) {
                const float z = s_red[0] + s_red[4] + s_red[8] + s_red[12], rt = hs[0];
                kap = ph * kv / (rt + z);
                const float u = (mu / rt) * kv * kv;
                p[bh * kPD + tid] = ph / (1.0f + u * ph);
            } else if (ISO) {
                const float abar = (s_red[0] + s_red[4] + s_red[8] + s_red[12]) * (1.0f / kPD);
                const float kn2 = s_red[1] + s_red[5] + s_red[9] + s_red[13], rt = hs[0];
                const float bhat = abar * hs[2] + hs[1];
                kap = bhat / (rt + bhat * kn2) * kv;
                if (tid == 0) p[bh] = bhat / (1.0f + mu * kn2 / (static_cast<float>(kPD) * rt) * bhat);
            } else {
                const float A = fmaf(hs[1], vb[5 * kPD + tid], hs[2] * kv * kv);
                const float rho = logf(fmaxf(A, kStatFloor)) - hs[3];
                kap = hs[0] * exp2f(neg_log2x * (rho / (1.0f + fabsf(rho)))) * kv;
                p[bh * kPD + tid] = A;
            }
            s_kap[tid] = kap;
        }
        // kappa . q (warps 0-3)
        if (warp < 4) {
            const float kq = warp_sum(kap * qv);
            if (lane == 0) s_red[warp * 4 + 3] = kq;
        }
        // per column j: sum_i (a_i k_i) S_ij and sum_i (a_i q_i) S_ij from the registers
        {
            float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const int i = rg + 8 * m;
                const float ak = s_ak[i], aq = s_aq[i];
                pk.x = fmaf(ak, reg[m].x, pk.x); pk.y = fmaf(ak, reg[m].y, pk.y);
                pk.z = fmaf(ak, reg[m].z, pk.z); pk.w = fmaf(ak, reg[m].w, pk.w);
                pq.x = fmaf(aq, reg[m].x, pq.x); pq.y = fmaf(aq, reg[m].y, pq.y);
                pq.z = fmaf(aq, reg[m].z, pq.z); pq.w = fmaf(aq, reg[m].w, pq.w);
            }
            *reinterpret_cast<float4*>(s_part + rg * kPD + 4 * c4) = pk;
            *reinterpret_cast<float4*>(s_part + 8 * kPD + rg * kPD + 4 * c4) = pq;
        }
        __syncthreads();
        if (tid < kPD) {
            const float kq = s_red[3] + s_red[7] + s_red[11] + s_red[15];
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                sk += s_part[g * kPD + tid];
                sq += s_part[8 * kPD + g * kPD + tid];
            }
            const float d = IO<TIO>::load(vv, tid) - sk;
            s_delta[tid] = d;
            IO<TIO>::store(o, bh * kPD + tid, sq + d * kq);
        }
        __syncthreads();
        // ---- S = diag(a) S + kappa delta^T, back into the ring slot, then out by bulk store
        {
            const float4 d4 = *reinterpret_cast<const float4*>(s_delta + 4 * c4);
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const int i = rg + 8 * m;
                const float ai = s_a[i], ki = s_kap[i];
                float4 x = reg[m];
                x.x = fmaf(ai, x.x, ki * d4.x);
                x.y = fmaf(ai, x.y, ki * d4.y);
                x.z = fmaf(ai, x.z, ki * d4.z);
                x.w = fmaf(ai, x.w, ki * d4.w);
                *reinterpret_cast<float4*>(Sb + i * kPD + 4 * c4) = x;
            }
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
                bulk_store(S + bh * kPD * kPD + c * 4096, ring_s + slot * kSBytes + c * 16384, 16384);
            bulk_commit();
            if (n + 2 < nh) {
                bulk_wait_read1();   // the slot of head n + 2 held head n - 1, whose store has read it
                issue(n + 2);
            }
            if (n + 1 < nh) {
#pragma unroll
                for (int e = 0; e < 4; ++e) s_hs[((n + 1) & 1) * 4 + e] = hsn[e];
            }
        }
    }
    if (tid == 0) {
        if (n < nh) {
            // a copy timed out: let the loads already issued (heads n and n + 1) land
            // before the CTA's shared memory goes away
            for (int m = n; m < nh && m <= n + 1; ++m)
                mbar_wait(bar_s + 8 * (m % kRing), static_cast<uint32_t>(m / kRing) & 1u, kStreamWaitLimit);
        }
        bulk_wait_all();
    }
}

}  // namespace

namespace {
int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

template <typename TIO, int V>
cudaError_t launch_stream(const StepArgs& a, int BH, int nsm, cudaStream_t s) {
    auto kern = step_stream_kernel<TIO, V>;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmem);
    if (e != cudaSuccess) return e;
    const int grid = BH < nsm ? BH : nsm;
    kern<<<grid, kPNT, kStreamSmem, s>>>(static_cast<const TIO*>(a.q), static_cast<const TIO*>(a.k),
                                         static_cast<const TIO*>(a.v), a.log_alpha, a.omega, a.r, a.S, a.p,
                                         static_cast<TIO*>(a.o), a.mu, a.status, a.beta, a.alpha_p, a.beta_p,
                                         a.center, a.neg_log2x, BH, a.H,
                                         (a.flags & KDN_FLAG_TIMEOUT_PROBE) ? 1 : 0);
    return cudaGetLastError();
}

template <typename TIO>
cudaError_t launch_stream_variant(const StepArgs& a, int BH, int nsm, cudaStream_t s) {
    if (a.variant == 0) return launch_stream<TIO, 0>(a, BH, nsm, s);
    if (a.variant == 1) return launch_stream<TIO, 1>(a, BH, nsm, s);
    return launch_stream<TIO, 2>(a, BH, nsm, s);
}
}  // namespace

cudaError_t launch_step(const StepArgs& a, cudaStream_t s) {
    const int BH = a.B * a.H;
    if (BH == 0) return cudaSuccess;
    if (a.dk == kPD && a.dv == kPD) {
        const int nsm = sm_count();
        if (nsm <= 0) return cudaErrorInvalidDevice;
        return a.io == 1 ? launch_stream_variant<__nv_bfloat16>(a, BH, nsm, s)
                         : launch_stream_variant<float>(a, BH, nsm, s);
    }
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
