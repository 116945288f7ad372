// Backward pass of the KDN mixer on CUDA cores (fp32): the gradients of a weighted
// sum  sum(dO * o) + sum(dS_T * S_T) + sum(dp_T * p_T)  with respect to every input
// of kdn_diag_forward / kdn_iso_forward.
//
// The pages define the forward recurrence only (KDN paper Sec. 4.1 Eq. 23-27 and
// 60-65, Sec. 4.2 Eq. 40 and App. C); the gradients are the adjoint of that
// recurrence, evaluated in the chunk form the forward uses (App. D).  With the gains
// kappa_t known, the memory of one chunk of C tokens in its reference frame is
//     S_m   = diag(g_in) S_0,                g_in  = exp(G_ref),
//     (I + L) Delta = X,  X = V - K_bar S_m, L = strict_lower(K_bar K_til^T),
//     O     = Q_bar S_m + A Delta,           A = lower_incl(Q_bar K_til^T),
//     S_out = diag(g_out) (S_m + K_til^T Delta),  g_out = exp(G_C - G_ref),
// with K_bar = k exp(G - G_ref), Q_bar = q exp(G - G_ref), K_til = kappa exp(G_ref - G)
// (G the cumulative log-decay since the chunk start).  Its adjoint, given dO and the
// gradient dS_out of the chunk's end state, is (Gp = diag(g_out) dS_out)
//     dDelta = K_til Gp + A^T dO,     (I + L)^T dX = dDelta,      dV = dX,
//     dK_til = Delta Gp^T + dL^T K_bar + dA^T Q_bar,   dQ_bar = dO S_m^T + dA K_til,
//     dK_bar = -dX S_m^T + dL K_til,   dA = lower_incl(dO Delta^T),
//     dL = strict_lower(-dX Delta^T),  dS_m = Gp + Q_bar^T dO - K_bar^T dX,
//     dS_0 = diag(g_in) dS_m,
// and the decay enters through d/dG of K_bar, Q_bar, K_til and g_out (G_ref cancels
// out of the result, so it is held fixed).  Kernels:
//   mem_adjoint_kernel    one CTA per (b, h): a forward sweep over the chunks that
//                         stores the state at every chunk start, then the reverse
//                         sweep above, writing dq, dv, the memory parts of dk and
//                         d log_alpha, dkappa and dS_0;
//   gain_adjoint_kernel   one CTA per (b, h), one thread per key channel: the
//                         uncertainty recurrence recomputed from checkpoints every
//                         kPB tokens and run backwards token by token (the adjoint of
//                         the gain and of the Moebius update), adding the gain parts of
//                         dk and d log_alpha and writing d omega, dr and dp_0.
// The gains kappa come from the forward's gain scan (scan.cu).

#include <string.h>

#include "common.cuh"
#include "kdn_internal.h"
#include "mma_tf32x3.cuh"

namespace kdn {
namespace {

constexpr int kBC = 16;       // tokens per chunk of the memory adjoint
constexpr int kMNT = 256;     // threads of the memory adjoint
constexpr int kPB = 64;       // tokens per checkpoint block of the gain adjoint
constexpr int kEl = kBC * 128 / kMNT;        // elements of a [kBC][d] tile per thread (d <= 128)

struct MemArgs {
    const void *q, *k, *v, *dO;
    const float *la, *kappa, *S0, *dS_T;
    float *ckpt;                    // [B*H][nch + 1][DK][DV] states at chunk starts
    float *dq, *dk, *dv, *dla, *dkappa, *dS0;
    int T, H, DK, DV;
    uint32_t* status;
};

// Rows of the d-wide operands are padded to d + 4 words: the MMA fragment loads (lane
// 4 g + q reading word g * ld + q, or q * ld + g) then meet at most 2-way bank conflicts.
constexpr int kRowPad = 4;

size_t mem_smem_floats(int DK, int DV) {
    const int LSK = DK + kRowPad, LSV = DV + kRowPad, LCC = kBC + 1;
    return (size_t)2 * DK * LSV + 7 * kBC * LSK + 3 * kBC * LSV + 4 * kBC * LCC + 4 * DK;
}

template <typename TIO>
__global__ void __launch_bounds__(kMNT, 1) mem_adjoint_kernel(const MemArgs P) {
    const int DK = P.DK, DV = P.DV, LSK = DK + kRowPad, LSV = DV + kRowPad, LCC = kBC + 1;
    constexpr int kEPC = 16 / static_cast<int>(sizeof(TIO));   // elements per 16-byte copy
    extern __shared__ float sm[];
    float* Sm = sm;                    // [DK][LSV] chunk-start state, then S_m
    float* dS = Sm + DK * LSV;         // [DK][LSV] gradient of the chunk's end state
    float* Kb = dS + DK * LSV;         // [kBC][LSK]
    float* Qb = Kb + kBC * LSK;
    float* Kt = Qb + kBC * LSK;
    float* dKb = Kt + kBC * LSK;
    float* dQb = dKb + kBC * LSK;
    float* dKt = dQb + kBC * LSK;
    float* Gc = dKt + kBC * LSK;       // [kBC][LSK] cumulative log-decay G_t within the chunk
    float* X = Gc + kBC * LSK;         // [kBC][LSV] V - K_bar S_m, then Delta
    float* dO = X + kBC * LSV;         // [kBC][LSV]
    float* dX = dO + kBC * LSV;        // [kBC][LSV] dDelta, then the adjoint of X
    float* L = dX + kBC * LSV;         // [kBC][LCC]
    float* Am = L + kBC * LCC;
    float* dL = Am + kBC * LCC;
    float* dA = dL + kBC * LCC;
    float* gref = dA + kBC * LCC;      // [DK]
    float* gin = gref + DK;
    float* gout = gin + DK;
    float* eS = gout + DK;             // [DK] sum_j dS_out S_out (dG of the chunk's last token)

    const int bh = blockIdx.x, H = P.H, T = P.T, b = bh / H, h = bh % H, tid = threadIdx.x;
    const int nch = (T + kBC - 1) / kBC;
    const size_t sdd = (size_t)DK * DV;
    float* ck = P.ckpt + (size_t)bh * (nch + 1) * sdd;
    auto row = [&](int t) { return ((size_t)b * T + t) * H + h; };   // token-head index

    // row-wise passes over a [DK][LSV] state tile: a warp per row, 16-byte accesses
    // (LSV and DV are multiples of 4), no index division
    auto scale_rows = [&](float* M, const float* f) {   // M(i, :) *= f[i]
        for (int ri = tid >> 5; ri < DK; ri += kMNT / 32) {
            const float sc = f[ri];
            float4* m4 = reinterpret_cast<float4*>(M + ri * LSV);
            for (int j4 = tid & 31; j4 < DV / 4; j4 += 32) {
                float4 v = m4[j4];
                v.x *= sc; v.y *= sc; v.z *= sc; v.w *= sc;
                m4[j4] = v;
            }
        }
    };
    auto store_state = [&](float* dst) {   // dst[i][j] (dense [DK][DV]) = Sm(i, j)
        for (int ri = tid >> 5; ri < DK; ri += kMNT / 32) {
            const float4* m4 = reinterpret_cast<const float4*>(Sm + ri * LSV);
            float4* d4 = reinterpret_cast<float4*>(dst + (size_t)ri * DV);
            for (int j4 = tid & 31; j4 < DV / 4; j4 += 32) d4[j4] = m4[j4];
        }
    };

    // per-chunk setup: cumulative log-decay G, reference and factors; the operands
    // K_bar, Q_bar, K_til; S_m = diag(g_in) S_0 with S_0 in Sm.  The chunk's inputs are
    // read into registers by one batch of loads per thread before any of them is used.
    auto setup = [&](int n, int nv) {
        const int t0 = n * kBC;
        // log_alpha -> Gc and kappa -> Kt, and k, q (into the dK_bar, dQ_bar tiles, sized
        // by d_k) and v (into the dX tile, sized by d_v) in their storage type, dense rows,
        // by 16-byte async copies, rows past the sequence end zero-filled (those tiles are
        // free until the reverse products)
        const TIO* kg = static_cast<const TIO*>(P.k);
        const TIO* qg = static_cast<const TIO*>(P.q);
        const TIO* vg = static_cast<const TIO*>(P.v);
        TIO* rawK = reinterpret_cast<TIO*>(dKb);
        TIO* rawQ = reinterpret_cast<TIO*>(dQb);
        TIO* rawV = reinterpret_cast<TIO*>(dX);
        for (int e4 = tid; e4 < kBC * DK / 4; e4 += kMNT) {
            const int t = (4 * e4) / DK, i = (4 * e4) % DK;
            const size_t gi = row(t0 + min(t, nv - 1)) * DK + i;
            cp_async16(Gc + t * LSK + i, P.la + gi, t < nv);
            cp_async16(Kt + t * LSK + i, P.kappa + gi, t < nv);
        }
        for (int e = tid * kEPC; e < kBC * DK; e += kMNT * kEPC) {
            const int t = e / DK, i = e % DK;
            const size_t gi = row(t0 + min(t, nv - 1)) * DK + i;
            cp_async16(rawK + e, kg + gi, t < nv);
            cp_async16(rawQ + e, qg + gi, t < nv);
        }
        for (int e = tid * kEPC; e < kBC * DV; e += kMNT * kEPC) {
            const int t = e / DV, j = e % DV;
            cp_async16(rawV + e, vg + row(t0 + min(t, nv - 1)) * DV + j, t < nv);
        }
        cp_async_wait_all();
        __syncthreads();
        for (int e = tid; e < kBC * DV; e += kMNT) X[(e / DV) * LSV + e % DV] = IO<TIO>::load(rawV, e);
        if (tid < DK) {
            float g = 0.f;
            for (int t = 0; t < kBC; ++t) {
                g += Gc[t * LSK + tid];
                Gc[t * LSK + tid] = g;
            }
            const float gr = 0.5f * g;
            gref[tid] = gr;
            gin[tid] = expf(gr);
            gout[tid] = expf(g - gr);
            if (!(fabsf(g) <= kMaxChunkLogDecay)) set_status(P.status, kStatusRange);
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < kEl; ++m) {
            const int e = tid + m * kMNT, t = e / DK, i = e % DK;
            if (e < kBC * DK) {
                const float ef = expf(Gc[t * LSK + i] - gref[i]);
                Kb[t * LSK + i] = IO<TIO>::load(rawK, e) * ef;
                Qb[t * LSK + i] = IO<TIO>::load(rawQ, e) * ef;
                Kt[t * LSK + i] /= ef;   // kappa e^{-(G_t - G_ref)}
                Gc[t * LSK + i] = ef;    // (G itself is not needed again in the chunk)
            }
        }
        scale_rows(Sm, gin);
        __syncthreads();
        // L = strict_lower(K_bar K_til^T), A = lower_incl(Q_bar K_til^T), X = V - K_bar S_m
        smem_gemm<1>(kBC, kBC, DK, Kb, LSK, 1, Kt, 1, LSK, L, LCC, 1.f, false, 2);    // (warps 6-7)
        smem_gemm<1>(kBC, kBC, DK, Qb, LSK, 1, Kt, 1, LSK, Am, LCC, 1.f, false, 4);   // (warps 4-5)
        smem_gemm<2>(kBC, DV, DK, Kb, LSK, 1, Sm, LSV, 1, X, LSV, -1.f, true);
        __syncthreads();
        for (int e = tid; e < kBC * kBC; e += kMNT) {
            const int t = e / kBC, s = e % kBC;
            if (s >= t) L[t * LCC + s] = 0.f;
            if (s > t) Am[t * LCC + s] = 0.f;
        }
        __syncthreads();
        // forward substitution (I + L) Delta = X: a thread per value column, held in
        // registers, which it alone reads and writes (no barrier between rows)
        for (int j = tid; j < DV; j += kMNT) {
            float x[kBC];
#pragma unroll
            for (int t = 0; t < kBC; ++t) x[t] = X[t * LSV + j];
#pragma unroll
            for (int t = 1; t < kBC; ++t) {
                if (t < nv) {
#pragma unroll
                    for (int s = 0; s < t; ++s) x[t] = fmaf(-L[t * LCC + s], x[s], x[t]);
                }
            }
#pragma unroll
            for (int t = 0; t < kBC; ++t) X[t * LSV + j] = x[t];
        }
        __syncthreads();
    };
    // a checkpointed state into Sm: 16-byte async copies, all in flight together (the
    // caller waits and synchronises)
    auto load_state = [&](const float* src) {
        for (int e4 = tid; e4 < DK * DV / 4; e4 += kMNT)
            cp_async16(Sm + ((4 * e4) / DV) * LSV + (4 * e4) % DV, src + 4 * e4, true);
    };

    // ---- forward sweep: the state at every chunk start
    for (int e = tid; e < DK * DV; e += kMNT) {
        const int i = e / DV, j = e % DV;
        Sm[i * LSV + j] = P.S0 ? P.S0[(size_t)bh * sdd + i * DV + j] : 0.f;
    }
    __syncthreads();
    for (int n = 0; n < nch; ++n) {
        const int nv = min(kBC, T - n * kBC);
        store_state(ck + (size_t)n * sdd);
        setup(n, nv);
        // S_out = diag(g_out) (S_m + K_til^T Delta)
        smem_gemm<2>(DK, DV, kBC, Kt, 1, LSK, X, LSV, 1, Sm, LSV, 1.f, true);
        __syncthreads();
        scale_rows(Sm, gout);
        __syncthreads();
    }
    store_state(ck + (size_t)nch * sdd);
    __syncthreads();

    // ---- reverse sweep
    // eS_i = sum_j dS_out(i, j) S_out(i, j) for the chunk about to be processed; for the
    // last chunk from S_T (still in Sm) and dS_T, then at the end of every chunk from its
    // S_m and dS_m (the factors g_in of S_out = diag(g_in)^-1 S_m and dS_out =
    // diag(g_in) dS_m cancel)
    for (int e = tid; e < DK * DV; e += kMNT) {
        const int i = e / DV, j = e % DV;
        dS[i * LSV + j] = P.dS_T ? P.dS_T[(size_t)bh * sdd + i * DV + j] : 0.f;
    }
    __syncthreads();
    for (int ri = tid >> 5; ri < DK; ri += kMNT / 32) {
        float acc = 0.f;
        for (int j = tid & 31; j < DV; j += 32) acc = fmaf(dS[ri * LSV + j], Sm[ri * LSV + j], acc);
        acc = warp_sum(acc);
        if ((tid & 31) == 0) eS[ri] = acc;
    }
    for (int n = nch - 1; n >= 0; --n) {
        const int t0 = n * kBC, nv = min(kBC, T - t0);
        __syncthreads();
        load_state(ck + (size_t)n * sdd);
        // dO in its storage type into the dX tile (sized by d_v, free here), then converted
        {
            const TIO* og = P.dO ? static_cast<const TIO*>(P.dO) : static_cast<const TIO*>(P.q);
            TIO* rawO = reinterpret_cast<TIO*>(dX);
            for (int e = tid * kEPC; e < kBC * DV; e += kMNT * kEPC) {
                const int t = e / DV, j = e % DV;
                cp_async16(rawO + e, og + row(t0 + min(t, nv - 1)) * DV + j, P.dO && t < nv);
            }
            cp_async_wait_all();
            __syncthreads();
            for (int e = tid; e < kBC * DV; e += kMNT) dO[(e / DV) * LSV + e % DV] = IO<TIO>::load(rawO, e);
        }
        __syncthreads();
        setup(n, nv);   // Sm = S_m, X = Delta, operands, L, A
        scale_rows(dS, gout);   // Gp = diag(g_out) dS_out
        __syncthreads();
        // dDelta = K_til Gp + A^T dO;  dK_til = Delta Gp^T;  dQ_bar = dO S_m^T;  dA = dO Delta^T
        smem_gemm<2>(kBC, DV, DK, Kt, LSK, 1, dS, LSV, 1, dX, LSV, 1.f, false);
        smem_gemm<2>(kBC, DK, DV, X, LSV, 1, dS, 1, LSV, dKt, LSK, 1.f, false);
        smem_gemm<2>(kBC, DK, DV, dO, LSV, 1, Sm, 1, LSV, dQb, LSK, 1.f, false);
        smem_gemm<1>(kBC, kBC, DV, dO, LSV, 1, X, 1, LSV, dA, LCC, 1.f, false);
        __syncthreads();
        smem_gemm<2>(kBC, DV, kBC, Am, 1, LCC, dO, LSV, 1, dX, LSV, 1.f, true);
        for (int e = tid; e < kBC * kBC; e += kMNT) {
            const int t = e / kBC, s = e % kBC;
            if (s > t) dA[t * LCC + s] = 0.f;
        }
        __syncthreads();
        // back substitution (I + L)^T dX = dDelta (a thread per value column, in registers;
        // rows past the sequence end are zero in L)
        for (int j = tid; j < DV; j += kMNT) {
            float x[kBC];
#pragma unroll
            for (int t = 0; t < kBC; ++t) x[t] = dX[t * LSV + j];
#pragma unroll
            for (int t = kBC - 2; t >= 0; --t) {
#pragma unroll
                for (int s = t + 1; s < kBC; ++s) x[t] = fmaf(-L[s * LCC + t], x[s], x[t]);
            }
#pragma unroll
            for (int t = 0; t < kBC; ++t) dX[t * LSV + j] = x[t];
        }
        __syncthreads();
        // dL = strict_lower(-dX Delta^T); dK_bar = -dX S_m^T
        smem_gemm<1>(kBC, kBC, DV, dX, LSV, 1, X, 1, LSV, dL, LCC, -1.f, false);
        smem_gemm<2>(kBC, DK, DV, dX, LSV, 1, Sm, 1, LSV, dKb, LSK, -1.f, false);
        __syncthreads();
        for (int e = tid; e < kBC * kBC; e += kMNT) {
            const int t = e / kBC, s = e % kBC;
            if (s >= t) dL[t * LCC + s] = 0.f;
        }
        __syncthreads();
        // dK_bar += dL K_til; dK_til += dL^T K_bar + dA^T Q_bar; dQ_bar += dA K_til;
        // dS_m = Gp + Q_bar^T dO - K_bar^T dX
        smem_gemm<2>(kBC, DK, kBC, dL, LCC, 1, Kt, LSK, 1, dKb, LSK, 1.f, true);
        smem_gemm<2>(kBC, DK, kBC, dL, 1, LCC, Kb, LSK, 1, dKt, LSK, 1.f, true);
        smem_gemm<2>(kBC, DK, kBC, dA, LCC, 1, Kt, LSK, 1, dQb, LSK, 1.f, true);
        smem_gemm<2>(DK, DV, kBC, Qb, 1, LSK, dO, LSV, 1, dS, LSV, 1.f, true);
        __syncthreads();   // (the next two accumulate into dS and dK_til again)
        smem_gemm<2>(DK, DV, kBC, Kb, 1, LSK, dX, LSV, 1, dS, LSV, -1.f, true);
        smem_gemm<2>(kBC, DK, kBC, dA, 1, LCC, Qb, LSK, 1, dKt, LSK, 1.f, true);
        __syncthreads();
        // per-token gradients of the inputs; dS becomes the gradient of the chunk start
        for (int e = tid; e < kBC * DV; e += kMNT) {
            const int t = e / DV, j = e % DV;
            if (t < nv) P.dv[row(t0 + t) * DV + j] = dX[t * LSV + j];
        }
        if (tid < DK) {
            const int i = tid;
            float dG = eS[i];            // d/dG_t, accumulated from the last token backwards
            for (int t = nv - 1; t >= 0; --t) {
                const size_t gi = row(t0 + t) * DK + i;
                const float kb = Kb[t * LSK + i], qb = Qb[t * LSK + i], kt = Kt[t * LSK + i];
                const float dkb = dKb[t * LSK + i], dqb = dQb[t * LSK + i], dkt = dKt[t * LSK + i];
                // K_bar = k f, Q_bar = q f, K_til = kappa / f with f = exp(G_t - G_ref) (in Gc)
                const float f = Gc[t * LSK + i];
                P.dk[gi] = dkb * f;
                P.dq[gi] = dqb * f;
                P.dkappa[gi] = dkt / f;
                dG += dkb * kb + dqb * qb - dkt * kt;
                P.dla[gi] = dG;   // d log_alpha_t = sum over tokens u >= t of dG_u
            }
        }
        __syncthreads();   // (the loop above reads eS)
        // eS of the previous chunk; dS becomes the gradient of the chunk start (a warp
        // per state row)
        for (int ri = tid >> 5; ri < DK; ri += kMNT / 32) {
            float acc = 0.f;
            const float gi = gin[ri];
            for (int j = tid & 31; j < DV; j += 32) {
                const float d = dS[ri * LSV + j];
                acc = fmaf(d, Sm[ri * LSV + j], acc);
                dS[ri * LSV + j] = d * gi;
            }
            acc = warp_sum(acc);
            if ((tid & 31) == 0) eS[ri] = acc;
        }
    }
    __syncthreads();
    for (int e = tid; e < DK * DV; e += kMNT) {
        const int i = e / DV, j = e % DV;
        P.dS0[(size_t)bh * sdd + i * DV + j] = dS[i * LSV + j];
    }
}

// ---------------------------------------------------------------- gain adjoint
struct GainArgs {
    int variant;                       // 0 diagonal, 1 isotropic
    const void* k;
    const float *la, *om, *r, *p0, *dp_T, *dkappa;
    float *pck;                        // [B*H][nblk][nu] variance at every kPB-token block start
    float *dk, *dla, *dom, *dr, *dp0;
    int T, H, DK;
    float mu;
};

template <typename TIO, int V>
__global__ void gain_adjoint_kernel(const GainArgs P) {
    constexpr bool ISO = V == 1;
    // per token of a block: p_prev, p_hat ([kPB][DK]; isotropic [kPB]), den, the
    // isotropic a_bar, ||k||^2, and the token sums s1 (diagonal: sum dkappa p_hat k;
    // isotropic: sum dkappa k); the block's inputs staged by coalesced loads: k,
    // log_alpha (reused for d/du of each channel), dkappa ([kPB][DK]), omega
    // ([kPB][DK]; isotropic [kPB]) and r [kPB].  Every cross-channel sum is taken for
    // the whole block at once (none of them feeds the serial recurrence).
    extern __shared__ float gsm[];
    const int DK = P.DK, T = P.T, H = P.H, bh = blockIdx.x, b = bh / H, h = bh % H;
    const int i = threadIdx.x, lane = i & 31, warp = i >> 5, nwarps = blockDim.x >> 5, nth = blockDim.x;
    const bool act = i < DK;
    const int nblk = (T + kPB - 1) / kPB, nu = ISO ? 1 : DK;
    float* spp = gsm;                           // [kPB][DK] (isotropic: [kPB])
    float* sph = spp + kPB * DK;                // [kPB][DK] (isotropic: [kPB])
    float* sden = sph + kPB * DK;               // [kPB]
    float* sab = sden + kPB;                    // [kPB]
    float* sk2 = sab + kPB;                     // [kPB]
    float* ss1 = sk2 + kPB;                     // [kPB]
    float* xk = ss1 + kPB;                      // [kPB][DK]
    float* xla = xk + kPB * DK;                 // [kPB][DK]
    float* xdk = xla + kPB * DK;                // [kPB][DK]
    float* xom = xdk + kPB * DK;                // [kPB][nu]
    float* xr = xom + kPB * nu;                 // [kPB]
    const TIO* kp = static_cast<const TIO*>(P.k);
    auto row = [&](int t) { return ((size_t)b * T + t) * H + h; };
    float* pck = P.pck + (size_t)bh * nblk * nu;
    const float mu = P.mu;
    // (eight elements per thread per round: the loads of a round are all in flight together)
    auto stage = [&](int t0, int nt, bool with_dkappa) {
        __syncthreads();
        for (int e0 = i; e0 < nt * DK; e0 += 8 * nth) {
            float rk[8], rla[8], rom[8], rdk[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int e = e0 + m * nth;
                const bool ok = e < nt * DK;
                const size_t g = row(t0 + (ok ? e / DK : 0)) * DK + e % DK;
                rk[m] = ok ? IO<TIO>::load(kp, g) : 0.f;
                rla[m] = ok ? P.la[g] : 0.f;
                rom[m] = (ok && !ISO) ? P.om[g] : 0.f;
                rdk[m] = (ok && with_dkappa) ? P.dkappa[g] : 0.f;
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int e = e0 + m * nth;
                if (e < nt * DK) {
                    xk[e] = rk[m];
                    xla[e] = rla[m];
                    if (!ISO) xom[e] = rom[m];
                    if (with_dkappa) xdk[e] = rdk[m];
                }
            }
        }
        for (int e = i; e < nt; e += nth) {
            xr[e] = P.r[row(t0 + e)];
            if (ISO) xom[e] = P.om[row(t0 + e)];
        }
        __syncthreads();
    };
    // out[t] = sum over channels c of f(t, c), for every token of the block (a warp per token)
    auto token_sums = [&](int nt, auto f, float* out) {
        __syncthreads();
        for (int t = warp; t < nt; t += nwarps) {
            float acc = 0.f;
            for (int c = lane; c < DK; c += 32) acc += f(t, c);
            acc = warp_sum(acc);
            if (lane == 0) out[t] = acc;
        }
        __syncthreads();
    };
    auto iso_stats = [&](int nt) {   // a_bar_t = mean exp(2 log_alpha), ||k_t||^2
        token_sums(nt, [&](int t, int c) { return expf(2.f * xla[t * DK + c]); }, sab);
        token_sums(nt, [&](int t, int c) { return xk[t * DK + c] * xk[t * DK + c]; }, sk2);
    };

    // forward over the sequence: the variance at every block start
    float p = P.p0 ? (ISO ? P.p0[bh] : (act ? P.p0[(size_t)bh * DK + i] : 0.f)) : 1.f;
    for (int blk = 0; blk < nblk; ++blk) {
        const int t0 = blk * kPB, nt = min(kPB, T - t0);
        if (ISO ? i == 0 : act) pck[(size_t)blk * nu + (ISO ? 0 : i)] = p;
        stage(t0, nt, false);
        if (ISO) {
            iso_stats(nt);
            for (int tl = 0; tl < nt; ++tl) {   // (every thread runs the scalar recurrence)
                const float ph = sab[tl] / DK * p + xom[tl];
                p = ph / (1.f + mu * sk2[tl] / (DK * xr[tl]) * ph);
            }
        } else if (act) {
            for (int tl = 0; tl < nt; ++tl) {
                const float kv = xk[tl * DK + i];
                const float ph = expf(2.f * xla[tl * DK + i]) * p + xom[tl * DK + i];
                p = ph / (1.f + mu * kv * kv / xr[tl] * ph);
            }
        }
    }
    float dp = P.dp_T ? (ISO ? P.dp_T[bh] : (act ? P.dp_T[(size_t)bh * DK + i] : 0.f)) : 0.f;
    for (int blk = nblk - 1; blk >= 0; --blk) {
        const int t0 = blk * kPB, nt = min(kPB, T - t0);
        stage(t0, nt, true);
        // recompute the block forward, keeping p_prev and p_hat; then den and s1
        p = pck[(size_t)blk * nu + (ISO ? 0 : (act ? i : 0))];
        if (ISO) {
            iso_stats(nt);
            if (i == 0) {
                for (int tl = 0; tl < nt; ++tl) {
                    const float ph = sab[tl] / DK * p + xom[tl];
                    spp[tl] = p;
                    sph[tl] = ph;
                    sden[tl] = xr[tl] + ph * sk2[tl];
                    p = ph / (1.f + mu * sk2[tl] / (DK * xr[tl]) * ph);
                }
            }
            token_sums(nt, [&](int t, int c) { return xdk[t * DK + c] * xk[t * DK + c]; }, ss1);
        } else {
            if (act) {
                for (int tl = 0; tl < nt; ++tl) {
                    const float kv = xk[tl * DK + i];
                    const float ph = expf(2.f * xla[tl * DK + i]) * p + xom[tl * DK + i];
                    spp[tl * DK + i] = p;
                    sph[tl * DK + i] = ph;
                    p = ph / (1.f + mu * kv * kv / xr[tl] * ph);
                }
            }
            token_sums(nt, [&](int t, int c) { return sph[t * DK + c] * xk[t * DK + c] * xk[t * DK + c]; }, sden);
            token_sums(nt, [&](int t, int c) { return xdk[t * DK + c] * sph[t * DK + c] * xk[t * DK + c]; }, ss1);
            for (int t = i; t < nt; t += nth) sden[t] += xr[t];
            __syncthreads();
        }
        // adjoint, newest token first (no cross-channel sums inside)
        for (int tl = nt - 1; tl >= 0; --tl) {
            const size_t th = row(t0 + tl);
            const float rr = xr[tl], den = sden[tl];
            if (ISO) {
                const float ph = sph[tl], pp = spp[tl], ab = sab[tl] / DK, k2 = sk2[tl];
                const float u = mu * k2 / (DK * rr), gq = 1.f + u * ph, beta = ph / den;
                float dph = dp / (gq * gq);
                const float du = -dp * ph * ph / (gq * gq);
                const float dbeta = ss1[tl];
                dph += dbeta / den;
                const float dden = -dbeta * ph / (den * den);
                dph += dden * k2;
                const float dk2 = dden * ph + du * mu / (DK * rr);
                dp = ab * dph;
                if (act) {
                    const float kv = xk[tl * DK + i], a = expf(xla[tl * DK + i]);
                    xdk[tl * DK + i] = beta * xdk[tl * DK + i] + 2.f * dk2 * kv;
                    xla[tl * DK + i] = pp * dph * 2.f * a * a / DK;   // d log a = d a * a
                }
                if (i == 0) {
                    P.dom[th] = dph;
                    P.dr[th] = dden - du * mu * k2 / (DK * rr * rr);
                }
            } else if (act) {
                const float kv = xk[tl * DK + i], a = expf(xla[tl * DK + i]), dkap = xdk[tl * DK + i];
                const float ph = sph[tl * DK + i], pp = spp[tl * DK + i];
                const float u = mu * kv * kv / rr, gq = 1.f + u * ph;
                float dph = dp / (gq * gq);
                const float du = -dp * ph * ph / (gq * gq);
                const float dden = -ss1[tl] / (den * den);
                dph += dkap * kv / den + dden * kv * kv;
                const float gk = dkap * ph / den + 2.f * dden * ph * kv + du * 2.f * mu * kv / rr;
                dp = a * a * dph;
                xdk[tl * DK + i] = gk;                   // (this token's inputs are no longer
                spp[tl * DK + i] = 2.f * a * pp * dph * a;   //  needed: the buffers take its
                xla[tl * DK + i] = du;                   //  gradients)
                P.dom[th * DK + i] = dph;
            }
        }
        if (!ISO) {   // dr_t = dden_t + sum_i -du_i mu k_i^2 / r_t^2
            token_sums(nt, [&](int t, int c) { return xla[t * DK + c] * xk[t * DK + c] * xk[t * DK + c]; }, sab);
            for (int t = i; t < nt; t += nth) {
                const float rr = xr[t], den = sden[t];
                P.dr[row(t0 + t)] = -ss1[t] / (den * den) - mu * sab[t] / (rr * rr);
            }
        }
        __syncthreads();
        const float* gla = ISO ? xla : spp;
        for (int e0 = i; e0 < nt * DK; e0 += 8 * nth) {
            float rk[8], rla[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int e = e0 + m * nth;
                const size_t g = row(t0 + (e < nt * DK ? e / DK : 0)) * DK + e % DK;
                rk[m] = e < nt * DK ? P.dk[g] : 0.f;
                rla[m] = e < nt * DK ? P.dla[g] : 0.f;
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int e = e0 + m * nth;
                if (e < nt * DK) {
                    const size_t g = row(t0 + e / DK) * DK + e % DK;
                    P.dk[g] = rk[m] + xdk[e];
                    P.dla[g] = rla[m] + gla[e];
                }
            }
        }
    }
    if (ISO) {
        if (i == 0) P.dp0[bh] = dp;
    } else if (act) {
        P.dp0[(size_t)bh * DK + i] = dp;
    }
}

}  // namespace

size_t backward_mem_smem_bytes(int dk, int dv) { return mem_smem_floats(dk, dv) * sizeof(float); }

cudaError_t launch_backward(const BackwardArgs& a, const BackwardWorkspace& w, cudaStream_t s) {
    // gains kappa_t from the forward's gain scan
    ForwardArgs f;
    memset(&f, 0, sizeof(f));
    f.variant = a.variant; f.B = a.B; f.T = a.T; f.H = a.H; f.dk = a.dk; f.dv = a.dv; f.chunk = kBC;
    f.mu = a.mu; f.io = a.io; f.q = a.q; f.k = a.k; f.v = a.v; f.log_alpha = a.log_alpha;
    f.omega = a.omega; f.r = a.r; f.S0 = a.S0; f.p0 = a.p0; f.p_T = w.p_scratch; f.status = a.status;
    ScanWorkspace sw;
    sw.kappa = w.kappa;
    sw.summary = w.summary;
    sw.carry = w.carry;
    sw.chunk_g = kGainChunk;
    sw.n_chunks_g = w.n_chunks_g;
    cudaError_t e = launch_gain_scan(f, sw, s);
    if (e != cudaSuccess) return e;

    MemArgs m;
    m.q = a.q; m.k = a.k; m.v = a.v; m.dO = a.dO;
    m.la = a.log_alpha; m.kappa = w.kappa; m.S0 = a.S0; m.dS_T = a.dS_T;
    m.ckpt = w.ckpt;
    m.dq = a.dq; m.dk = a.dk_out; m.dv = a.dv_out; m.dla = a.dla; m.dkappa = w.dkappa; m.dS0 = a.dS0;
    m.T = a.T; m.H = a.H; m.DK = a.dk; m.DV = a.dv; m.status = a.status;
    const size_t smem = backward_mem_smem_bytes(a.dk, a.dv);
    const int BH = a.B * a.H;
    if (a.io == 1) {
        e = cudaFuncSetAttribute(mem_adjoint_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        mem_adjoint_kernel<__nv_bfloat16><<<BH, kMNT, smem, s>>>(m);
    } else {
        e = cudaFuncSetAttribute(mem_adjoint_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        mem_adjoint_kernel<float><<<BH, kMNT, smem, s>>>(m);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    GainArgs g;
    g.variant = a.variant; g.k = a.k; g.la = a.log_alpha; g.om = a.omega; g.r = a.r; g.p0 = a.p0;
    g.dp_T = a.dp_T; g.dkappa = w.dkappa; g.pck = w.pck;
    g.dk = a.dk_out; g.dla = a.dla; g.dom = a.domega; g.dr = a.dr; g.dp0 = a.dp0;
    g.T = a.T; g.H = a.H; g.DK = a.dk; g.mu = a.mu;
    const int nt = ((a.dk + 31) / 32) * 32;
    const int nu = a.variant == 1 ? 1 : a.dk;
    const size_t gsm = sizeof(float) * (5 * kPB * a.dk + 6 * kPB + kPB * nu);
    auto launch_gain = [&](auto kernel) {
        const cudaError_t e2 = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gsm);
        if (e2 != cudaSuccess) return e2;
        kernel<<<BH, nt, gsm, s>>>(g);
        return cudaGetLastError();
    };
    if (a.variant == 1)
        return a.io == 1 ? launch_gain(gain_adjoint_kernel<__nv_bfloat16, 1>) : launch_gain(gain_adjoint_kernel<float, 1>);
    return a.io == 1 ? launch_gain(gain_adjoint_kernel<__nv_bfloat16, 0>) : launch_gain(gain_adjoint_kernel<float, 0>);
}

int backward_chunk() { return kBC; }
int backward_block() { return kPB; }

}  // namespace kdn
