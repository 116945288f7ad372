// Fused tensor-core forward of the KDN mixer (sm_103a): bf16 q/k/v/o,
// d_k = d_v = 128, memory chunk C = 64, fp32 state resident in TMEM.
//
// One CTA owns one (b, h) sequence and walks its chunks in order; per chunk:
//   A1  uncertainty recurrence (KDN paper Sec. 4.1 Eq. 23-27 with the
//       information-scaled update Eq. 60-65, i.e. the Moebius map of Eq. 32-37
//       applied token by token; the chunk carry is the per-channel variance
//       held in a register).  Isotropic variant (Sec. 4.2 Eq. 40, App. C): the
//       scalar map is composed as 2x2 Moebius matrices with a warp-shuffle
//       inclusive scan over the chunk's tokens, then replayed from the carry.
//       Also the cumulative log-decay G_t per channel and the gain
//       denominators r_t + sum_i p_hat_t,i k_t,i^2.
//   A2  decayed operands (bf16, 128-byte-swizzled, tensor-core layouts):
//         K_bar = k e^{G - G_ref}, Q_bar = q e^{G - G_ref}, K_til = kappa e^{G_ref - G},
//       with the per-channel reference G_ref = G_C / 2 (App. D: decay ratios
//       from differences of cumulative log-decay).
//   B   Gram MMA  [K_bar; Q_bar] K_til^T  (M = 128: rows 0-63 give L, rows
//       64-127 the query-write matrix A, diagonal kept).
//   C,D T = (I + strict_lower(L))^{-1}, 16x16 diagonal blocks by forward
//       substitution, merged 16 -> 32 -> 64 (fp32 on CUDA cores).
//   E   W^T = K_bar^T T^T and U^T = V^T T^T (MMA, fp32 in TMEM).
//   G   state: S_m^T = S_in^T diag(e^{G_ref}) (TMEM -> registers -> TMEM, and
//       a bf16 copy as the next MMAs' operand).
//   H   Delta^T = U^T - S_m^T W^T  (innovations), O^T = S_m^T Q_bar^T.
//   J   O^T += Delta^T A^T ; S^T += Delta^T K_til  (state stays in TMEM; the
//       pending factor e^{G_C - G_ref} is folded into the next chunk's scaling).
//   K   o = O (bf16) to global memory.
// This is the compact-WY / UT chunk form of the paper's App. D evaluated with
// per-channel decay; Preconditioned DeltaNet prints the same algebra without
// decay (its Eq. 6 / App. F.2.1).  All MMAs are tcgen05 kind::f16 (bf16
// operands, fp32 accumulation) with M = 128, fed from shared memory; inputs
// arrive by TMA; every wait is bounded and reports KDN_ERR_TIMEOUT.

#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kdn_internal.h"
#include "sm100.cuh"

namespace kdn {
namespace {

using namespace sm100;

constexpr int kC = 64;     // tokens per chunk
constexpr int kD = 128;    // d_k = d_v
constexpr int kNT = 256;   // threads: warps 0-3 own TMEM lanes, warps 4-7 own key channels
constexpr uint32_t kWaitLimit = 1u << 20;

// Shared memory map (bytes from a 1024-aligned base).  Regions reused within
// a chunk are noted; every reuse starts after the previous user finished.
constexpr uint32_t OFF_QIN = 0;        // q tile, 2 TMA boxes of [64 t][64 d] bf16 (SW128)
constexpr uint32_t OFF_KIN = 16384;    // k tile
constexpr uint32_t OFF_VIN = 32768;    // v tile (MN-major A operand of U^T)
constexpr uint32_t OFF_LA = 49152;     // log_alpha [64][128] fp32 -> cumulative G in place
constexpr uint32_t OFF_OM = 81920;     // omega [64][128] fp32 -> p_hat in place (diagonal)
constexpr uint32_t OFF_KQ = 114688;    // [K_bar; Q_bar] 128 rows x 128, two 16 KB K-atoms
constexpr uint32_t OFF_DT = OFF_KQ;    //   later Delta^T [128 j][64 t] bf16, then the o tile
constexpr uint32_t OFF_OST = OFF_KQ;   //   o tile [64 t][128 j] bf16 staged for the TMA store
constexpr uint32_t OFF_KT = 147456;    // K_til [64 s][128 i], two 8 KB K-atoms
constexpr uint32_t OFF_AQ = 163840;    // A [64 t][64 s] bf16
constexpr uint32_t OFF_LF = 172032;    // L fp32 [64][kLDF]
constexpr uint32_t OFF_W = OFF_LF;     //   later W [128 i][64 t] bf16 (MN-major B)
constexpr uint32_t OFF_TT = 189440;    // T [64 t][64 s] bf16
constexpr uint32_t OFF_TF = 197632;    // T fp32 [64][kLDF]
constexpr uint32_t OFF_XT = 215040;    // merge temporaries fp32 [32][kLDX]
constexpr uint32_t OFF_SM = 189440;    //   later S_m^T [128 j][128 i] bf16, two 16 KB K-atoms
constexpr uint32_t OFF_SMALL = 222208;
constexpr int kLDF = 68;
constexpr int kLDX = 36;
// small region, float offsets
constexpr int SM_R = 0, SM_MUR = 64, SM_INVZ = 128, SM_ZP = 192, SM_AP = 448, SM_GREF = 704,
              SM_FOUT = 832, SM_OMI = 960, SM_FLAG = 1024, SM_CF = 1032 /* [2][128] by chunk parity */,
              SM_FLOATS = 1288;
constexpr uint32_t OFF_BAR = OFF_SMALL + SM_FLOATS * 4;
constexpr uint32_t kSmemBytes = OFF_BAR + 64;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(OFF_XT + 32 * kLDX * 4 <= OFF_SM + 32768, "merge scratch inside the S_m^T region");
static_assert(OFF_TF + 64 * kLDF * 4 <= OFF_XT, "T fp32 before the merge scratch");
static_assert(OFF_LF + 64 * kLDF * 4 <= OFF_TT, "L fp32 before T");
static_assert(kSmemAlloc <= 232448, "shared memory per CTA");

// TMEM columns (one CTA per SM, all 512 allocated)
constexpr uint32_t TM_S = 0, TM_D = 128, TM_O = 192, TM_G = 256, TM_W = 320, TM_COLS = 512;

struct TcParams {
    CUtensorMap tq, tk, tv, tla, tom, to;
    const float* r;
    const float* om_iso;
    const float* S0;
    const float* p0;
    __nv_bfloat16* o;
    float* S_T;
    float* p_T;
    uint32_t* status;
    int T, H;
    float mu;
};

// Lane L of a warp returns sum over lanes of v[L] (transpose-reduce, 31 shuffles).
__device__ __forceinline__ float butterfly_sum32(float (&v)[32], int lane) {
#pragma unroll
    for (int n = 16; n >= 1; n >>= 1) {
        const bool up = (lane & n) != 0;
#pragma unroll
        for (int j = 0; j < n; ++j) {
            const float send = up ? v[j] : v[j + n];
            const float keep = up ? v[j + n] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, n);
        }
    }
    return v[0];
}

struct Mob {
    float a, b, c, d;  // [[a, b], [c, d]]
};
__device__ __forceinline__ Mob mob_mul(const Mob& x, const Mob& y) {  // x * y
    return {fmaf(x.a, y.a, x.b * y.c), fmaf(x.a, y.b, x.b * y.d), fmaf(x.c, y.a, x.d * y.c),
            fmaf(x.c, y.b, x.d * y.d)};
}
__device__ __forceinline__ void mob_renorm(Mob& m) {  // exact power-of-two rescale
    const float mx = fmaxf(fmaxf(m.a, m.b), fmaxf(m.c, m.d));
    int e;
    frexpf(mx, &e);
    const float s = ldexpf(1.0f, -e);
    m.a *= s; m.b *= s; m.c *= s; m.d *= s;
}

// ---- warp-level TF32 MMA helpers for the triangular inverse (fp32 row-major tiles in shared memory)
__device__ __forceinline__ uint32_t tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// x[n8 tile][4] = A[16 x 8*k1] (k-steps k0..k1-1) * B[8*k1 x 16]; A, B row-major with strides lda, ldb.
__device__ __forceinline__ void mma_tile_16xN(float (&x)[2][4], const float* A, int lda, const float* B, int ldb,
                                              int k0, int k1) {
    const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[n][e] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
        if (ks < k0 || ks >= k1) continue;
        const float* a = A + 8 * ks;
        const uint32_t a0 = tf32(a[g * lda + q]), a1 = tf32(a[(g + 8) * lda + q]);
        const uint32_t a2 = tf32(a[g * lda + q + 4]), a3 = tf32(a[(g + 8) * lda + q + 4]);
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const float* bp = B + (8 * ks) * ldb + 8 * n;
            mma_tf32(x[n], a0, a1, a2, a3, tf32(bp[q * ldb + g]), tf32(bp[(q + 4) * ldb + g]));
        }
    }
}
__device__ __forceinline__ void mma_tile_16x16(float (&x)[2][4], const float* A, int lda, const float* B, int ldb,
                                               int ksteps) {
    mma_tile_16xN(x, A, lda, B, ldb, 0, ksteps);
}
__device__ __forceinline__ void store_tile_16x16(const float (&x)[2][4], float* D, int ldd, float scale, int g,
                                                 int q) {
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        D[g * ldd + 8 * n + 2 * q] = scale * x[n][0];
        D[g * ldd + 8 * n + 2 * q + 1] = scale * x[n][1];
        D[(g + 8) * ldd + 8 * n + 2 * q] = scale * x[n][2];
        D[(g + 8) * ldd + 8 * n + 2 * q + 1] = scale * x[n][3];
    }
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

template <bool ISO>
__global__ void __launch_bounds__(kNT, 1) kdn_fused_tc_kernel(const __grid_constant__ TcParams P) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(base);
    float* sm = reinterpret_cast<float*>(base + OFF_SMALL);
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + SM_FLAG);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + OFF_BAR + 32);
    const uint32_t bar_in = sb + OFF_BAR, bar_v = bar_in + 8, bar_mma = bar_in + 16;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x, H = P.H, b = bh / H, h = bh % H, T = P.T;
    const int nchunks = (T + kC - 1) / kC;

    if (tid == 0) {
        mbar_init(bar_in, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_mma, 1);
        mbar_fence_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), TM_COLS);
        tc_fence_before();
    }

    auto issue_inputs = [&](int n) {
        const int t0 = n * kC;
        mbar_expect_tx(bar_in, ISO ? 65536u : 98304u);
        tma_load_4d(sb + OFF_QIN, &P.tq, 0, h, t0, b, bar_in);
        tma_load_4d(sb + OFF_QIN + 8192, &P.tq, 64, h, t0, b, bar_in);
        tma_load_4d(sb + OFF_KIN, &P.tk, 0, h, t0, b, bar_in);
        tma_load_4d(sb + OFF_KIN + 8192, &P.tk, 64, h, t0, b, bar_in);
        tma_load_4d(sb + OFF_LA, &P.tla, 0, h, t0, b, bar_in);
        if (!ISO) tma_load_4d(sb + OFF_OM, &P.tom, 0, h, t0, b, bar_in);
    };
    auto issue_v = [&](int n) {
        mbar_expect_tx(bar_v, 16384u);
        tma_load_4d(sb + OFF_VIN, &P.tv, 0, h, n * kC, b, bar_v);
        tma_load_4d(sb + OFF_VIN + 8192, &P.tv, 64, h, n * kC, b, bar_v);
    };
    __syncthreads();
    if (tid == 0 && nchunks > 0) {
        issue_inputs(0);
        issue_v(0);
    }
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);

    // per-thread recurrent state
    float p_reg = 1.0f;   // diagonal: variance of channel tid - 128 (warps 4-7)
    float pend = 0.0f;    // pending log-factor G_C - G_ref of the previous chunk (warps 4-7)
    float b_iso = 1.0f;   // isotropic scalar variance (warp 4)
    if (tid >= 128) {
        const int i = tid - 128;
        if (!ISO && P.p0) p_reg = P.p0[static_cast<size_t>(bh) * kD + i];
    }
    if (ISO && warp == 4 && P.p0) b_iso = P.p0[bh];
    // initial state S^T into TMEM: lane j = value column, columns = key channel
    if (tid < 128) {
        const int j = tid;
        uint32_t r[32];
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const int i = q * 32 + c;
                r[c] = __float_as_uint(P.S0 ? P.S0[(static_cast<size_t>(bh) * kD + i) * kD + j] : 0.0f);
            }
            tmem_st32(lane_base + TM_S + q * 32, r);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    uint32_t ph_in = 0, ph_v = 0, ph_mma = 0;
    int n_in_issued = nchunks > 0 ? 1 : 0, n_v_issued = n_in_issued, n_mma_issued = 0;
    auto wait_or_abort = [&](uint32_t bar, uint32_t parity) {
        if (*s_abort) return;
        if (!mbar_wait(bar, parity, kWaitLimit)) {
            set_status(P.status, kStatusTimeout);
            *s_abort = 1;
        }
    };

    float* LA = reinterpret_cast<float*>(base + OFF_LA);
    float* OM = reinterpret_cast<float*>(base + OFF_OM);
    float* LF = reinterpret_cast<float*>(base + OFF_LF);
    float* TF = reinterpret_cast<float*>(base + OFF_TF);
    float* XT = reinterpret_cast<float*>(base + OFF_XT);

    // Warps 4-7: per-token scalars of chunk c, then (inputs landed) the uncertainty
    // recurrence and cumulative log-decay of chunk c.  Runs one chunk ahead of the
    // memory pass of warps 0-3.
    auto prep_gains = [&](int c) {
        const int t0c = c * kC, nvc = min(kC, T - t0c);
        if (tid < 128 + kC) {
            const int t = tid - 128;
            float rr = 1.0f, om = 0.0f;
            if (t < nvc) {
                const size_t th = (static_cast<size_t>(b) * T + t0c + t) * H + h;
                rr = P.r[th];
                if (ISO) om = P.om_iso[th];
            }
            sm[SM_R + t] = rr;
            sm[SM_MUR + t] = P.mu / rr;
            sm[SM_OMI + t] = om;
        }
        wait_or_abort(bar_in, ph_in);
        named_bar(1, 128);
            if (tid >= 128) {
                const int i = tid - 128, w4 = warp - 4;
                const unsigned char* kin = base + OFF_KIN + (i >> 6) * 8192 + (i & 7) * 2;
                const int kch = (i & 63) >> 3;
                float G = 0.0f;
    #pragma unroll 1
                for (int hf = 0; hf < 2; ++hf) {
                    float w[32], w2[32];
    #pragma unroll
                    for (int qt = 0; qt < 2; ++qt) {
                        // loads and token-local arithmetic first (independent of the carry) ...
                        float a2[16], k2[16], om[16], gq[16];
    #pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const int t = hf * 32 + qt * 16 + u;
                            const float lav = LA[t * kD + i];
                            const float kv = __bfloat162float(
                                *reinterpret_cast<const __nv_bfloat16*>(kin + sw128_off(t, kch)));
                            a2[u] = __expf(2.0f * lav);
                            k2[u] = kv * kv;
                            om[u] = ISO ? 0.0f : OM[t * kD + i];
                            gq[u] = lav;
                        }
    #pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const int t = hf * 32 + qt * 16 + u;
                            if (t < nvc) G += gq[u];
                            gq[u] = G;
                        }
    #pragma unroll
                        for (int u = 0; u < 16; ++u) LA[(hf * 32 + qt * 16 + u) * kD + i] = gq[u];
                        // ... then the serial carry chain
    #pragma unroll
                        for (int u = 0; u < 16; ++u) {
                            const int t = hf * 32 + qt * 16 + u;
                            const bool valid = t < nvc;
                            if (!ISO) {
                                const float ph = fmaf(a2[u], p_reg, om[u]);
                                const float pn = __fdividef(ph, fmaf(sm[SM_MUR + t] * k2[u], ph, 1.0f));
                                p_reg = valid ? pn : p_reg;
                                om[u] = valid ? ph : 0.0f;
                                w[qt * 16 + u] = valid ? ph * k2[u] : 0.0f;
                            } else {
                                w[qt * 16 + u] = valid ? k2[u] : 0.0f;
                                w2[qt * 16 + u] = valid ? a2[u] : 0.0f;
                            }
                        }
                        if (!ISO) {
    #pragma unroll
                            for (int u = 0; u < 16; ++u) OM[(hf * 32 + qt * 16 + u) * kD + i] = om[u];
                        }
                    }
                    sm[SM_ZP + w4 * 64 + hf * 32 + lane] = butterfly_sum32(w, lane);
                    if (ISO) sm[SM_AP + w4 * 64 + hf * 32 + lane] = butterfly_sum32(w2, lane);
                }
                const float gref = 0.5f * G;
                sm[SM_GREF + i] = gref;
                sm[SM_CF + (c & 1) * 128 + i] = __expf(pend + gref);
                pend = G - gref;
                sm[SM_FOUT + i] = __expf(pend);
                if (!(fabsf(G) <= kMaxChunkLogDecay)) set_status(P.status, kStatusRange);
                if (ISO) {
                    named_bar(1, 128);
                    if (w4 == 0) {
                        // Moebius scan of the scalar recurrence over the chunk, 2 tokens per lane
                        float aa[2], uu[2], oo[2], kk[2], rr[2];
                        Mob m[2];
    #pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int t = 2 * lane + e;
                            const float asum = sm[SM_AP + t] + sm[SM_AP + 64 + t] + sm[SM_AP + 128 + t] +
                                               sm[SM_AP + 192 + t];
                            kk[e] = sm[SM_ZP + t] + sm[SM_ZP + 64 + t] + sm[SM_ZP + 128 + t] +
                                    sm[SM_ZP + 192 + t];
                            aa[e] = asum * (1.0f / kD);
                            rr[e] = sm[SM_R + t];
                            oo[e] = sm[SM_OMI + t];
                            uu[e] = P.mu * kk[e] / (kD * rr[e]);
                            if (t < nvc)
                                m[e] = {aa[e], oo[e], uu[e] * aa[e], fmaf(uu[e], oo[e], 1.0f)};
                            else
                                m[e] = {1.0f, 0.0f, 0.0f, 1.0f};
                        }
                        Mob pr = mob_mul(m[1], m[0]);
                        mob_renorm(pr);
    #pragma unroll
                        for (int d = 1; d < 32; d <<= 1) {
                            Mob q;
                            q.a = __shfl_up_sync(0xffffffffu, pr.a, d);
                            q.b = __shfl_up_sync(0xffffffffu, pr.b, d);
                            q.c = __shfl_up_sync(0xffffffffu, pr.c, d);
                            q.d = __shfl_up_sync(0xffffffffu, pr.d, d);
                            if (lane >= d) {
                                pr = mob_mul(pr, q);
                                mob_renorm(pr);
                            }
                        }
                        Mob ex;
                        ex.a = __shfl_up_sync(0xffffffffu, pr.a, 1);
                        ex.b = __shfl_up_sync(0xffffffffu, pr.b, 1);
                        ex.c = __shfl_up_sync(0xffffffffu, pr.c, 1);
                        ex.d = __shfl_up_sync(0xffffffffu, pr.d, 1);
                        if (lane == 0) ex = {1.0f, 0.0f, 0.0f, 1.0f};
                        float bb = (ex.a * b_iso + ex.b) / (ex.c * b_iso + ex.d);
    #pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int t = 2 * lane + e;
                            float beta = 0.0f;
                            if (t < nvc) {
                                const float bhat = fmaf(aa[e], bb, oo[e]);
                                beta = bhat / (rr[e] + bhat * kk[e]);
                                bb = bhat / fmaf(uu[e], bhat, 1.0f);
                            }
                            sm[SM_INVZ + t] = beta;
                        }
                        b_iso = __shfl_sync(0xffffffffu, bb, 31);
                    }
                }
            }

    };

    if (tid >= 128 && nchunks > 0) prep_gains(0);
    ph_in ^= 1u;
    __syncthreads();

#pragma unroll 1
    for (int n = 0; n < nchunks; ++n) {
        const int t0 = n * kC, nv = min(kC, T - t0);
        // ---------------- A2: gain denominators, then decayed bf16 operands (all warps)
        if (tid == 0) bulk_wait_read();  // the previous o tile has left the staging buffer
        if (!ISO && tid < kC) {
            const int t = tid;
            const float z = sm[SM_ZP + t] + sm[SM_ZP + 64 + t] + sm[SM_ZP + 128 + t] + sm[SM_ZP + 192 + t];
            sm[SM_INVZ + t] = t < nv ? 1.0f / (sm[SM_R + t] + z) : 0.0f;
        }
        __syncthreads();
#pragma unroll 1
        for (int m4 = 0; m4 < 4; ++m4) {
            const int idx = tid + kNT * m4, t = idx >> 4, g = idx & 15, box = g >> 3, ch = g & 7;
            const uint4 kr = *reinterpret_cast<const uint4*>(base + OFF_KIN + box * 8192 + sw128_off(t, ch));
            const uint4 qr = *reinterpret_cast<const uint4*>(base + OFF_QIN + box * 8192 + sw128_off(t, ch));
            const float kf[8] = {bf_lo(kr.x), bf_hi(kr.x), bf_lo(kr.y), bf_hi(kr.y),
                                 bf_lo(kr.z), bf_hi(kr.z), bf_lo(kr.w), bf_hi(kr.w)};
            const float qf[8] = {bf_lo(qr.x), bf_hi(qr.x), bf_lo(qr.y), bf_hi(qr.y),
                                 bf_lo(qr.z), bf_hi(qr.z), bf_lo(qr.w), bf_hi(qr.w)};
            const float4 g0 = *reinterpret_cast<const float4*>(LA + t * kD + 8 * g);
            const float4 g1 = *reinterpret_cast<const float4*>(LA + t * kD + 8 * g + 4);
            const float4 r0 = *reinterpret_cast<const float4*>(sm + SM_GREF + 8 * g);
            const float4 r1 = *reinterpret_cast<const float4*>(sm + SM_GREF + 8 * g + 4);
            const float Gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
            const float Rv[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
            float kap[8];
            const float sc = sm[SM_INVZ + t];
            if (!ISO) {
                const float4 p0v = *reinterpret_cast<const float4*>(OM + t * kD + 8 * g);
                const float4 p1v = *reinterpret_cast<const float4*>(OM + t * kD + 8 * g + 4);
                const float Pv[8] = {p0v.x, p0v.y, p0v.z, p0v.w, p1v.x, p1v.y, p1v.z, p1v.w};
#pragma unroll
                for (int c = 0; c < 8; ++c) kap[c] = Pv[c] * kf[c] * sc;
            } else {
#pragma unroll
                for (int c = 0; c < 8; ++c) kap[c] = sc * kf[c];
            }
            uint32_t kb[4], qb[4], kt[4];
#pragma unroll
            for (int c = 0; c < 8; c += 2) {
                const float e1a = __expf(Gv[c] - Rv[c]), e1b = __expf(Gv[c + 1] - Rv[c + 1]);
                const float e2a = __expf(Rv[c] - Gv[c]), e2b = __expf(Rv[c + 1] - Gv[c + 1]);
                kb[c / 2] = pack_bf16(kf[c] * e1a, kf[c + 1] * e1b);
                qb[c / 2] = pack_bf16(qf[c] * e1a, qf[c + 1] * e1b);
                kt[c / 2] = pack_bf16(kap[c] * e2a, kap[c + 1] * e2b);
            }
            *reinterpret_cast<uint4*>(base + OFF_KQ + box * 16384 + sw128_off(t, ch)) =
                make_uint4(kb[0], kb[1], kb[2], kb[3]);
            *reinterpret_cast<uint4*>(base + OFF_KQ + box * 16384 + sw128_off(64 + t, ch)) =
                make_uint4(qb[0], qb[1], qb[2], qb[3]);
            *reinterpret_cast<uint4*>(base + OFF_KT + box * 8192 + sw128_off(t, ch)) =
                make_uint4(kt[0], kt[1], kt[2], kt[3]);
        }
        fence_proxy_async();
        __syncthreads();
        if (*s_abort) break;
        // ---------------- B: prefetch the next chunk's q, k, log_alpha, omega; Gram MMA
        if (tid == 0) {
            if (n + 1 < nchunks) {
                issue_inputs(n + 1);
                ++n_in_issued;
            }
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t ad = sw128_desc(sb + OFF_KQ + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                const uint64_t bd = sw128_desc(sb + OFF_KT + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024);
                mma_bf16(tmem + TM_G, ad, bd, id, ks > 0);
            }
            mma_commit(bar_mma);
            ++n_mma_issued;
        }
        if (tid < 128) {
            // ======== warps 0-3: memory pass of chunk n
            // ---------------- C: Gram rows out of TMEM (L fp32, A bf16)
            {
                wait_or_abort(bar_mma, ph_mma);
                tc_fence_after();
                uint32_t v0[32], v1[32];
                tmem_ld32(lane_base + TM_G, v0);
                tmem_ld32(lane_base + TM_G + 32, v1);
                tmem_wait_ld();
                if (tid < 64) {
                    // L rows as they come: only entries below the diagonal are ever read
                    const int t = tid;
                    float* row = LF + t * kLDF;
    #pragma unroll
                    for (int c4 = 0; c4 < 16; ++c4) {
                        const int s = 4 * c4;
                        *reinterpret_cast<float4*>(row + s) =
                            make_float4(__uint_as_float(s + 0 < 32 ? v0[s + 0] : v1[s + 0 - 32]),
                                        __uint_as_float(s + 1 < 32 ? v0[s + 1] : v1[s + 1 - 32]),
                                        __uint_as_float(s + 2 < 32 ? v0[s + 2] : v1[s + 2 - 32]),
                                        __uint_as_float(s + 3 < 32 ? v0[s + 3] : v1[s + 3 - 32]));
                    }
                } else {
                    const int t = tid - 64;
    #pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint32_t pk[4];
    #pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int s = 8 * ch + 2 * e;
                            const float a0 = (s <= t) ? __uint_as_float(s < 32 ? v0[s] : v1[s - 32]) : 0.0f;
                            const float a1 = (s + 1 <= t) ? __uint_as_float(s + 1 < 32 ? v0[s + 1] : v1[s + 1 - 32]) : 0.0f;
                            pk[e] = pack_bf16(a0, a1);
                        }
                        *reinterpret_cast<uint4*>(base + OFF_AQ + sw128_off(t, ch)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            }

            ph_mma ^= 1u;
            fence_proxy_async();
            named_bar(2, 128);
            // ---------------- D: T = (I + L)^{-1}  (warps 0-3)
            {
                if (tid < 64) {  // 16x16 diagonal blocks: right-looking substitution, one column per thread
                    const int blk = tid >> 4, c = tid & 15, o = 16 * blk;
                    float acc[16];
    #pragma unroll
                    for (int r = 0; r < 16; ++r) acc[r] = (r == c) ? 1.0f : 0.0f;
    #pragma unroll
                    for (int s = 0; s < 16; ++s) {
                        const float xs = acc[s];
    #pragma unroll
                        for (int r = s + 1; r < 16; ++r) acc[r] = fmaf(-LF[(o + r) * kLDF + o + s], xs, acc[r]);
                    }
    #pragma unroll
                    for (int r = 0; r < 16; ++r) TF[(o + r) * kLDF + o + c] = acc[r];
                }
                named_bar(2, 128);
                const int g = lane >> 2, q4 = lane & 3;
                if (warp < 2) {  // 16 -> 32 merges: T_ij = -D_i (L_ij D_j), (i, j) = (1, 0), (3, 2)
                    const int i = 2 * warp + 1, j = 2 * warp;
                    float x[2][4];
                    mma_tile_16x16(x, LF + (16 * i) * kLDF + 16 * j, kLDF, TF + (16 * j) * kLDF + 16 * j, kLDF, 2);
                    float* xs = XT + (16 * warp) * kLDX;
                    store_tile_16x16(x, xs, kLDX, 1.0f, g, q4);
                    __syncwarp();
                    mma_tile_16x16(x, TF + (16 * i) * kLDF + 16 * i, kLDF, xs, kLDX, 2);
                    store_tile_16x16(x, TF + (16 * i) * kLDF + 16 * j, kLDF, -1.0f, g, q4);
                }
                named_bar(2, 128);
                {  // 32 -> 64: X = L[32:64, 0:32] T[0:32, 0:32]; T[32:64, 0:32] = -T[32:64, 32:64] X
                    const int mt = warp >> 1, nt0 = 2 * (warp & 1);
                    float x[2][4];
                    // T[0:16, 16:32] is zero: columns 16-31 take k-steps 2-3 only
                    mma_tile_16xN(x, LF + (32 + 16 * mt) * kLDF, kLDF, TF + 8 * nt0, kLDF, nt0 >= 2 ? 2 : 0, 4);
                    store_tile_16x16(x, XT + (16 * mt) * kLDX + 8 * nt0, kLDX, 1.0f, g, q4);
                    named_bar(2, 128);
                    // T[32:48, 48:64] is zero: rows 32-47 take k-steps 0-1 only
                    mma_tile_16xN(x, TF + (32 + 16 * mt) * kLDF + 32, kLDF, XT + 8 * nt0, kLDX, 0, mt == 0 ? 2 : 4);
                    store_tile_16x16(x, TF + (32 + 16 * mt) * kLDF + 8 * nt0, kLDF, -1.0f, g, q4);
                }
                named_bar(2, 128);
                {  // T (lower triangle incl. diagonal) -> bf16 [t][s]
                    const int t = tid >> 1, hf = tid & 1;
    #pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int ch = 4 * hf + cc;
                        uint32_t pk[4];
    #pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int s = 8 * ch + 2 * e;
                            const float a0 = (s <= t) ? TF[t * kLDF + s] : 0.0f;
                            const float a1 = (s + 1 <= t) ? TF[t * kLDF + s + 1] : 0.0f;
                            pk[e] = pack_bf16(a0, a1);
                        }
                        *reinterpret_cast<uint4*>(base + OFF_TT + sw128_off(t, ch)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
            }
            fence_proxy_async();
            named_bar(2, 128);
            // ---------------- E: W^T = K_bar^T T^T, U^T = V^T T^T
            if (tid == 0) {
                wait_or_abort(bar_v, ph_v);
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 64, 1, 0, 0);
    #pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t bd = sw128_desc(sb + OFF_TT + ks * 32, 16, 1024);
                    mma_bf16(tmem + TM_W, sw128_desc(sb + OFF_KQ + ks * 2048, 16384, 1024), bd, id, ks > 0);
                    mma_bf16(tmem + TM_D, sw128_desc(sb + OFF_VIN + ks * 2048, 8192, 1024), bd, id, ks > 0);
                }
                mma_commit(bar_mma);
                ++n_mma_issued;
            }
            ph_v ^= 1u;
            // ---------------- F: W^T rows -> bf16 W (MN-major B operand); prefetch next v
            {
                wait_or_abort(bar_mma, ph_mma);
                tc_fence_after();
                if (tid == 0 && n + 1 < nchunks) {
                    issue_v(n + 1);
                    ++n_v_issued;
                }
                const int i = tid;
                uint32_t v0[32], v1[32];
                tmem_ld32(lane_base + TM_W, v0);
                tmem_ld32(lane_base + TM_W + 32, v1);
                tmem_wait_ld();
    #pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t pk[4];
    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = 8 * ch + 2 * e;
                        pk[e] = pack_bf16(__uint_as_float(t < 32 ? v0[t] : v1[t - 32]),
                                          __uint_as_float(t + 1 < 32 ? v0[t + 1] : v1[t + 1 - 32]));
                    }
                    *reinterpret_cast<uint4*>(base + OFF_W + sw128_off(i, ch)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                // ---------------- G: state into the chunk's reference frame
                const int j = tid;
    #pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + TM_S + q * 32, r);
                    tmem_wait_ld();
    #pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 f = *reinterpret_cast<const float4*>(sm + SM_CF + (n & 1) * 128 + q * 32 + 4 * c4);
                        r[4 * c4 + 0] = __float_as_uint(__uint_as_float(r[4 * c4 + 0]) * f.x);
                        r[4 * c4 + 1] = __float_as_uint(__uint_as_float(r[4 * c4 + 1]) * f.y);
                        r[4 * c4 + 2] = __float_as_uint(__uint_as_float(r[4 * c4 + 2]) * f.z);
                        r[4 * c4 + 3] = __float_as_uint(__uint_as_float(r[4 * c4 + 3]) * f.w);
                    }
                    tmem_st32(lane_base + TM_S + q * 32, r);
                    const int katom = q >> 1;
    #pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t pk[4];
    #pragma unroll
                        for (int e = 0; e < 4; ++e)
                            pk[e] = pack_bf16(__uint_as_float(r[8 * cc + 2 * e]), __uint_as_float(r[8 * cc + 2 * e + 1]));
                        *reinterpret_cast<uint4*>(base + OFF_SM + katom * 16384 + sw128_off(j, (q & 1) * 4 + cc)) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                }
                tmem_wait_st();
            }

            ph_mma ^= 1u;
            fence_proxy_async();
            tc_fence_before();
            named_bar(2, 128);
            // ---------------- H: Delta^T = U^T - S_m^T W^T ; O^T = S_m^T Q_bar^T
            if (tid == 0) {
                tc_fence_after();
                const uint32_t id_d = idesc_bf16(128, 64, 0, 1, 1);
                const uint32_t id_o = idesc_bf16(128, 64, 0, 0, 0);
    #pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t ad = sw128_desc(sb + OFF_SM + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024);
                    mma_bf16(tmem + TM_D, ad, sw128_desc(sb + OFF_W + ks * 2048, 16, 1024), id_d, 1u);
                    mma_bf16(tmem + TM_O, ad,
                             sw128_desc(sb + OFF_KQ + 8192 + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024), id_o,
                             ks > 0);
                }
                mma_commit(bar_mma);
                ++n_mma_issued;
            }
            // ---------------- I: Delta^T rows -> bf16 (A operand)
            {
                wait_or_abort(bar_mma, ph_mma);
                tc_fence_after();
                const int j = tid;
                uint32_t v0[32], v1[32];
                tmem_ld32(lane_base + TM_D, v0);
                tmem_ld32(lane_base + TM_D + 32, v1);
                tmem_wait_ld();
    #pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t pk[4];
    #pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = 8 * ch + 2 * e;
                        pk[e] = pack_bf16(__uint_as_float(t < 32 ? v0[t] : v1[t - 32]),
                                          __uint_as_float(t + 1 < 32 ? v0[t + 1] : v1[t + 1 - 32]));
                    }
                    *reinterpret_cast<uint4*>(base + OFF_DT + sw128_off(j, ch)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }

            ph_mma ^= 1u;
            fence_proxy_async();
            tc_fence_before();
            named_bar(2, 128);
            // ---------------- J: O^T += Delta^T A^T ; S^T += Delta^T K_til
            if (tid == 0) {
                tc_fence_after();
                const uint32_t id_o = idesc_bf16(128, 64, 0, 0, 0);
                const uint32_t id_s = idesc_bf16(128, 128, 0, 1, 0);
    #pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t ad = sw128_desc(sb + OFF_DT + ks * 32, 16, 1024);
                    mma_bf16(tmem + TM_O, ad, sw128_desc(sb + OFF_AQ + ks * 32, 16, 1024), id_o, 1u);
                    mma_bf16(tmem + TM_S, ad, sw128_desc(sb + OFF_KT + ks * 2048, 8192, 1024), id_s, 1u);
                }
                mma_commit(bar_mma);
                ++n_mma_issued;
            }
            // ---------------- K: outputs, staged as a [64 t][128 j] tile and stored by TMA
            {
                wait_or_abort(bar_mma, ph_mma);
                tc_fence_after();
                const int j = tid;
                uint32_t v0[32], v1[32];
                tmem_ld32(lane_base + TM_O, v0);
                tmem_ld32(lane_base + TM_O + 32, v1);
                tmem_wait_ld();
                __nv_bfloat16* ost = reinterpret_cast<__nv_bfloat16*>(base + OFF_OST) + j;
    #pragma unroll
                for (int t = 0; t < kC; ++t)
                    ost[t * kD] = __float2bfloat16_rn(__uint_as_float(t < 32 ? v0[t] : v1[t - 32]));
                fence_proxy_async();
                named_bar(2, 128);
                if (tid == 0) {
                    tma_store_4d(&P.to, sb + OFF_OST, 0, h, t0, b);  // rows past T are clipped
                    bulk_commit();
                }
            }

            ph_mma ^= 1u;
            tc_fence_before();
        } else if (n + 1 < nchunks) {
            // ======== warps 4-7: gains of chunk n + 1
            prep_gains(n + 1);
        }
        if (n + 1 < nchunks) ph_in ^= 1u;
        __syncthreads();
        if (*s_abort) break;
    }
    if (tid == 0) bulk_wait_all();

    const bool aborted = *s_abort != 0;
    if (!aborted) {
        // final state: S_T = (TMEM state) scaled by the last chunk's pending factor
        if (tid < 128) {
            tc_fence_after();
            const int j = tid;
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t r[32];
                tmem_ld32(lane_base + TM_S + q * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int i = q * 32 + c;
                    const float f = nchunks > 0 ? sm[SM_FOUT + i] : 1.0f;
                    P.S_T[(static_cast<size_t>(bh) * kD + i) * kD + j] = __uint_as_float(r[c]) * f;
                }
            }
        } else if (!ISO) {
            P.p_T[static_cast<size_t>(bh) * kD + tid - 128] = p_reg;
        } else if (tid == 128) {
            P.p_T[bh] = b_iso;
        }
    } else if (tid == 0) {
        // let copies and MMAs already issued land before the CTA's resources go away
        if (n_mma_issued > 0) mbar_wait(bar_mma, (n_mma_issued - 1) & 1, kWaitLimit);
        if (n_in_issued > 0) mbar_wait(bar_in, (n_in_issued - 1) & 1, kWaitLimit);
        if (n_v_issued > 0) mbar_wait(bar_v, (n_v_issued - 1) & 1, kWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TM_COLS);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [B, T, H, 128] tensor, tile of 64 tokens of one (b, h).
bool encode_4d(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int esize, int B, int T, int H,
               uint32_t box0, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kD) * esize, static_cast<cuuint64_t>(H) * kD * esize,
                                   static_cast<cuuint64_t>(T) * H * kD * esize};
    const cuuint32_t box[4] = {box0, 1, static_cast<cuuint32_t>(kC), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, dt, 4, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_path_supported(int io, int dk, int dv, int chunk) {
    return io == 1 && dk == kD && dv == kD && chunk == kC;
}

int tc_kernel_count() { return 1; }

cudaError_t launch_forward_tc(const ForwardArgs& a, cudaStream_t s) {
    TcParams P;
    memset(&P, 0, sizeof(P));
    const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    bool ok = encode_4d(&P.tq, a.q, BF, 2, a.B, a.T, a.H, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_4d(&P.tk, a.k, BF, 2, a.B, a.T, a.H, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_4d(&P.tv, a.v, BF, 2, a.B, a.T, a.H, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_4d(&P.tla, a.log_alpha, F32, 4, a.B, a.T, a.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (ok && a.variant == 0)
        ok = encode_4d(&P.tom, a.omega, F32, 4, a.B, a.T, a.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (ok) ok = encode_4d(&P.to, a.o, BF, 2, a.B, a.T, a.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return cudaErrorInvalidValue;
    P.r = a.r;
    P.om_iso = a.variant == 1 ? a.omega : nullptr;
    P.S0 = a.S0;
    P.p0 = a.p0;
    P.o = static_cast<__nv_bfloat16*>(a.o);
    P.S_T = a.S_T;
    P.p_T = a.p_T;
    P.status = a.status;
    P.T = a.T;
    P.H = a.H;
    P.mu = a.mu;
    const int grid = a.B * a.H;
    cudaError_t e;
    if (a.variant == 0) {
        e = cudaFuncSetAttribute(kdn_fused_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        kdn_fused_tc_kernel<false><<<grid, kNT, kSmemAlloc, s>>>(P);
    } else {
        e = cudaFuncSetAttribute(kdn_fused_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        kdn_fused_tc_kernel<true><<<grid, kNT, kSmemAlloc, s>>>(P);
    }
    return cudaGetLastError();
}

}  // namespace kdn
