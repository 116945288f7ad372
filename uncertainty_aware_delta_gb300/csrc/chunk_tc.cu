// Fused tensor-core forward of the KDN mixer (sm_103a): bf16 q/k/v/o,
// d_k = d_v = 128, memory chunk C = 64, fp32 state resident in TMEM.
//
// One CTA owns one (b, h) sequence and walks its chunks in order; per chunk:
//   A1  uncertainty recurrence (KDN paper Sec. 4.1 Eq. 23-27 with the
//       information-scaled update Eq. 60-65, i.e. the Moebius map of Eq. 32-37
//       applied token by token in projective form (numerator, denominator),
//       which keeps the carry chain free of divisions; the chunk carry is the
//       per-channel variance as that pair, held in registers).  Isotropic variant (Sec. 4.2 Eq. 40, App. C): the
//       per-token channel sums of alpha^2 and k^2 are formed here; the scalar
//       map is composed as 2x2 Moebius matrices with a warp-shuffle inclusive
//       scan over the chunk's tokens (warp 11, beside the Gram MMA), then
//       replayed from the carry.
//       The decay factors relative to the chunk's per-channel reference G_ref
//       (App. D: decay ratios from differences of cumulative log-decay) are
//       running products e1_t = e^{G_t - G_ref}, G_ref = 0 (chunk start) when
//       |G_C| <= 80 and G_C / 2 otherwise; their reciprocals are taken in the
//       operand pass.
//   A2  decayed operands (bf16, 128-byte-swizzled, tensor-core layouts):
//         K_bar = k e1, Q_bar = q e1, K_til' = p_hat k / e1  (isotropic: k / e1;
//       its b_hat enters the triangular system on the diagonal only, as
//       r_t / b_hat_t + ||k_t||^2, and the innovations come out times b_hat_t).
//   B   Gram MMA  [K_bar; Q_bar] K_til'^T  (M = 128: rows 0-63 give the key
//       block, rows 64-127 the query-write matrix A', diagonal kept), and the
//       prediction/query MMA [Z^T | O^T] = S_m^T [K_bar; Q_bar]^T (N = 128).
//   C,D The gains are kappa = p_hat k / z with z_t = r_t + sum_i p_hat_t,i k_t,i^2
//       (Eq. 25).  Since K_bar_t . K_til'_t = sum_i p_hat_t,i k_t,i^2 (the decay
//       factors cancel), the scaled innovations Delta' = diag(1/z) Delta solve
//       M Delta' = V - K_bar S_m  with  M = diag(r) + lower_incl(K_bar K_til'^T),
//       so z comes out of the Gram MMA (and with it, on request, the effective
//       write strength k^T kappa = (z - r) / z of App. B Eq. 58-61).  T = M^{-1}: 16x16 diagonal blocks by
//       forward substitution, merged 16 -> 32 -> 64 (tf32 mma.sync).
//   G   state: S_m^T = S_in^T diag(e^{G_ref}) in TMEM, plus a bf16 copy in TMEM
//       that is the A operand of the prediction/query MMA.  The state is kept with
//       the previous chunk's factor e^{G_C - G_ref} pending, so one factor
//       e^{pending + G_ref} moves it into the frame; after two strongly decaying
//       chunks that product can fall below fp32's normal range, and it is then
//       applied in two parts (warps 4-7 apply e^{G_ref} once the state update of
//       the previous chunk has landed).
//   H   Delta'^T = (V^T - Z^T) T^T = V^T T^T + (-Z^T) T^T (-Z^T in bf16 in TMEM
//       as an A operand).
//   J   S^T += Delta'^T K_til' ; O^T += Delta'^T A'^T (issued at the start of
//       the next chunk)  (Delta'^T in bf16 in TMEM as the A operand; the state
//       stays in TMEM, the pending factor e^{G_C - G_ref} is folded into the next
//       chunk's scaling).
//   K   o = O (bf16) to global memory at the start of the next chunk.
// Schedule per chunk n: warps 0-3 store the outputs of chunk n-1 and move the
// state into the chunk's frame while warps 4-11 build the operands; one thread
// issues the prediction/query MMAs, thread 256 the Gram MMA and thread 160 the
// prefetch of chunk n+1; then
// warps 8-11 read out the Gram matrix and invert the triangular system while
// warps 0-3 convert the prediction and run H-J, and warps 4-7 compute the gains
// of chunk n+1 (A1).
// This is the compact-WY / UT chunk form of the paper's App. D evaluated with
// per-channel decay; Preconditioned DeltaNet prints the same algebra without
// decay (its Eq. 6 / App. F.2.1).  All MMAs are tcgen05 kind::f16 (bf16
// operands, fp32 accumulation) with M = 128; inputs arrive by TMA; every wait
// is bounded and reports KDN_ERR_TIMEOUT.

#include <cuda.h>
#include <cuda_bf16.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kdn.h"
#include "kdn_internal.h"
#include "sm100.cuh"

namespace kdn {
namespace {

using namespace sm100;

constexpr int kC = 64;     // tokens per chunk
constexpr int kD = 128;    // d_k = d_v
// Threads: warps 0-3 hold the state (TMEM lanes = value columns) and issue the
// MMAs and copies; warps 4-7 own the key channels of the uncertainty recurrence
// (one chunk ahead); warps 8-11 read out the Gram matrix and invert the
// triangular system.  Operands are built by warps 4-11.
constexpr int kNT = 384;
// named barriers
constexpr int kBarWG1 = 1, kBarWG0 = 2, kBarTReady = 3, kBarOps = 5, kBarWG2 = 6;
constexpr uint32_t kWaitLimit = 1u << 20;
// Bound of the timeout probe's wait (KDN_FLAG_TIMEOUT_PROBE): a few milliseconds.
constexpr uint32_t kProbeWaitLimit = 1u << 12;
constexpr float kLog2e = 1.4426950408889634f;
// Chunks whose log-decay stays within this bound use the chunk start as the decay
// reference (every factor e^{G_t} and its reciprocal fit in fp32 and bf16); the
// rare chunks beyond it switch to the mid-chunk reference G_C / 2.
constexpr float kStartRefLogDecay = 80.0f;

// Shared memory map (bytes from a 1024-aligned base).  Regions reused within
// a chunk are noted; every reuse starts after the previous user finished.
constexpr uint32_t OFF_QIN = 0;        // q tile, 2 TMA boxes of [64 t][64 d] bf16 (SW128)
constexpr uint32_t OFF_KIN = 16384;    // k tile
constexpr uint32_t OFF_VIN = 32768;    // v tile (MN-major A operand of U^T)
constexpr uint32_t OFF_LA = 49152;     // log_alpha [64][128] fp32 -> e1 in place
constexpr uint32_t OFF_OM = 81920;     // omega [64][128] fp32 -> p_hat in place (diagonal)
constexpr uint32_t OFF_KQ = 114688;    // [K_bar; Q_bar] 128 rows x 128, two 16 KB K-atoms
constexpr uint32_t OFF_KT = 147456;    // K_til' [64 s][128 i], two 8 KB K-atoms
constexpr uint32_t OFF_AQ = 163840;    // A [64 t][64 s] bf16
constexpr uint32_t OFF_LF = 172032;    // M fp32 [64][kLDF]
constexpr uint32_t OFF_TT = 189440;    // T [64 t][64 s] bf16
constexpr uint32_t OFF_TF = 197632;    // T fp32 [64][kLDF]
constexpr uint32_t OFF_XT = 215040;    // merge temporaries fp32 [32][kLDX]
constexpr uint32_t OFF_SMALL = 219648;
constexpr int kLDF = 68;
constexpr int kLDX = 36;
// small region, float offsets
// (buffers marked [2] are indexed by chunk parity; ZP and AP hold the isotropic
//  per-token sums of k^2 and alpha^2 as four per-warp partial sums)
constexpr int SM_R = 0, SM_MUR = 64, SM_OMB = 128 /* [2][64] */, SM_ZP = 256 /* [2][256] */,
              SM_AP = 768 /* [2][256] */, SM_RZ = 1280 /* [2][64] */, SM_FOUT = 1408, SM_OMI = 1536,
              SM_FLAG = 1600, SM_CF = 1608 /* [2][128] */, SM_INVD = 1864, SM_CF2 = 1928 /* [128] */,
              SM_FLOATS = 2056;
constexpr uint32_t OFF_BAR = OFF_SMALL + SM_FLOATS * 4;
constexpr uint32_t kSmemBytes = OFF_BAR + 88;
constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
static_assert(OFF_TF + 64 * kLDF * 4 <= OFF_XT, "T fp32 before the merge scratch");
static_assert(OFF_XT + 32 * kLDX * 4 <= OFF_SMALL, "merge scratch before the small region");
static_assert(OFF_LF + 64 * kLDF * 4 <= OFF_TT, "L fp32 before T");
static_assert(kSmemAlloc <= 232448, "shared memory per CTA");

// TMEM columns (one CTA per SM, 512 allocated): state S^T (fp32); Z^T = S_m^T K_bar^T
// then Delta^T, directly followed by O^T (one N = 128 MMA writes both Z^T and O^T);
// the Gram matrix; the bf16 copy of S_m^T (A operand, two values per column); and
// the bf16 A operand -Z^T, later Delta^T.
constexpr uint32_t TM_S = 0, TM_ZD = 128, TM_O = 192, TM_G = 256, TM_SMB = 320, TM_DB = 384, TM_COLS = 512;

struct TcParams {
    CUtensorMap tq, tk, tv, tla, tom;
    const float* r;
    const float* la;
    const float* om;      // omega: per channel (diagonal) or per token-head (isotropic)
    const float* S0;
    const float* p0;      // initial variances (KDN) or key statistic (PKDA)
    __nv_bfloat16* o;
    float* S_T;
    float* p_T;           // final variances (KDN) or key statistic (PKDA)
    uint32_t* status;
    // PKDA: write strength, statistic decay and weight per token-head, centre per head
    const float* beta;
    const float* alpha_p;
    const float* beta_p;
    const float* center;
    int T, H;
    float mu;
    float neg_log2x;      // PKDA: -log2(x), x the bound of the write scale
    // Sequence split: CTA blockIdx.x = bh * nseg + seg runs tokens
    // [seg * seg_len, min(T, (seg + 1) * seg_len)) of sequence bh (nseg = 1: whole
    // sequences).  seg_len is a multiple of the chunk, so only the last segment has
    // a ragged tail (past T, where the copies read zeros).
    int nseg, seg_len;
    int s0_identity;      // start from S = I (the segment's transition map) instead of S0
    int no_v;             // values read as zero (selects the kernel instance)
    int no_o;             // outputs not written
    int last_only;        // final state of the last segment only, to S_T / p_T at bh;
                          // otherwise every CTA writes its final state to S_T at blockIdx.x
    long long p0_bh, p0_seg;   // p0 element offset of (bh, seg): bh * p0_bh + seg * p0_seg
    int probe;            // timeout probe (KDN_FLAG_TIMEOUT_PROBE): one wait that nothing completes
    float* beta_eff;      // KDN, whole sequences: effective write strength [B,T,H], or null
};

// Kernel variants: the two KDN uncertainty models, the preconditioned delta
// rule with per-channel decay, and the memory pass with given gains (the
// dense-covariance filter's mean: S = diag(a) S + kappa (v - (diag(a) S)^T k)^T
// with kappa read from global memory, a unit-diagonal triangular system).
constexpr int kVarDiag = 0, kVarIso = 1, kVarPkda = 2, kVarGiven = 3;
// PKDA: the statistic enters the logarithm no smaller than this.
constexpr float kStatFloor = 1e-20f;
constexpr float kLn2 = 0.6931471805599453f;

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
__device__ __forceinline__ void mob_renorm(Mob& m) {  // exact power-of-two rescale (entries >= 0)
    const float mx = fmaxf(fmaxf(m.a, m.b), fmaxf(m.c, m.d));
    const int ex = min(max((__float_as_int(mx) >> 23) & 0xff, 1), 253);
    const float s = __int_as_float((254 - ex) << 23);   // 2^(127 - ex): mx * s in [1, 2)
    m.a *= s;
    m.b *= s;
    m.c *= s;
    m.d *= s;
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

// The same tile, scaled, as bf16 pairs into a 128-byte-swizzled [row][col] tile
// (rows r0.., columns c0..; 64 bf16 per row).
__device__ __forceinline__ void store_tile_bf16(const float (&x)[2][4], unsigned char* tile, int r0, int c0,
                                                float scale, int g, int q) {
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        const int col = c0 + 8 * n + 2 * q;
        const uint32_t off = (col & 7) * 2;
        *reinterpret_cast<uint32_t*>(tile + sw128_off(r0 + g, col >> 3) + off) =
            pack_bf16(scale * x[n][0], scale * x[n][1]);
        *reinterpret_cast<uint32_t*>(tile + sw128_off(r0 + g + 8, col >> 3) + off) =
            pack_bf16(scale * x[n][2], scale * x[n][3]);
    }
}

// ---- warp-level bf16 MMA of a 16x16 block of X Y^T, X and Y K-major bf16 tiles in the
// 128-byte-swizzled layout of the tensor-core operands (128-byte rows of 64 channels,
// two K-atoms of 64 channels at atom strides xa and ya bytes)
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_m16n8k16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// x[n8 tile][4] = rows r0..r0+15 of X times rows c0..c0+15 of Y, over 128 channels.
// ldmatrix: lane l addresses row (l & 7) of 8x8 matrix l >> 3; the A matrices are
// (rows 0-7 | 8-15) x (channels 0-7 | 8-15) of each 16-channel step, the B matrices
// (columns 0-7 | 8-15) x (channels 0-7 | 8-15).
__device__ __forceinline__ void gram_block16(float (&x)[2][4], uint32_t X, uint32_t xa, uint32_t Y, uint32_t ya,
                                             int r0, int c0, int lane) {
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[n][e] = 0.0f;
    const int mi = lane >> 3, rr = lane & 7;
    const int ra = r0 + rr + 8 * (mi & 1), rb = c0 + 8 * (mi >> 1) + rr;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        uint32_t a[4], bq[4];
        ldmatrix_x4(X + (ks >> 2) * xa + sw128_off(ra, 2 * (ks & 3) + (mi >> 1)), a);
        ldmatrix_x4(Y + (ks >> 2) * ya + sw128_off(rb, 2 * (ks & 3) + (mi & 1)), bq);
        mma_bf16_m16n8k16(x[0], a, bq[0], bq[1]);
        mma_bf16_m16n8k16(x[1], a, bq[2], bq[3]);
    }
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ float rcp_approx(float x) {   // 1 / x, hardware approximation
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// Packed fp32 pair arithmetic (two lanes per instruction).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{ .reg .b64 ra, rb, rc, rd; mov.b64 ra, {%2, %3}; mov.b64 rb, {%4, %5}; mov.b64 rc, {%6, %7};"
        " fma.rn.f32x2 rd, ra, rb, rc; mov.b64 {%0, %1}, rd; }"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{ .reg .b64 ra, rb, rd; mov.b64 ra, {%2, %3}; mov.b64 rb, {%4, %5}; add.rn.f32x2 rd, ra, rb;"
        " mov.b64 {%0, %1}, rd; }"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{ .reg .b64 ra, rb, rd; mov.b64 ra, {%2, %3}; mov.b64 rb, {%4, %5}; mul.rn.f32x2 rd, ra, rb;"
        " mov.b64 {%0, %1}, rd; }"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float ex2(float x) {   // 2^x, hardware approximation
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float lg2(float x) {   // log2(x), hardware approximation
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Rare path, kept out of line: multiply this thread's TMEM row of the fp32 state
// by per-channel factors f[0..127].
__device__ __noinline__ void rescale_state_rows(uint32_t lane_base, const float* f) {
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
        uint32_t r[32];
        tmem_ld32(lane_base + TM_S + 32 * q, r);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f[32 * q + e]);
        tmem_st32(lane_base + TM_S + 32 * q, r);
    }
}

// Named barrier over `nthreads` threads that also returns the OR of `pred` over them.
__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool pred) {
    uint32_t out;
    asm volatile(
        "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
        : "=r"(out)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return out != 0;
}

// Rare path, kept out of line: a channel whose chunk log-decay exceeds
// kStartRefLogDecay gets its factors e^{G_t - G_ref} and K_til' scales
// (p_hat / e1, 1 / e1 or the PKDA write scale / e1) rewritten with the mid-chunk
// reference G_ref = G_C / 2 (R2 in log2 units), from log_alpha (and omega) in
// global memory and the chunk-start carries, re-running the chunk's recurrence.
template <int V>
__device__ __noinline__ void strong_decay_factors(const TcParams& P, unsigned char* base, int i, int b, int h,
                                                  int t0c, int nvc, float R2, float pns, float pds, float sts,
                                                  float center) {
    constexpr bool ISO = V == kVarIso;
    const int T = P.T, H = P.H;
    float* LA = reinterpret_cast<float*>(base + OFF_LA);
    float* OM = reinterpret_cast<float*>(base + OFF_OM);
    const float* sm = reinterpret_cast<const float*>(base + OFF_SMALL);
    float gg = 0.0f;
    const size_t g0 = (static_cast<size_t>(b) * T + t0c) * H * kD + static_cast<size_t>(h) * kD + i;
    const unsigned char* kin = base + OFF_KIN + (i >> 6) * 8192 + (i & 7) * 2;
    const int kch = (i & 63) >> 3;
#pragma unroll 1
    for (int t = 0; t < kC; ++t) {
        const size_t e = g0 + static_cast<size_t>(t) * H * kD;
        const float l2 = t < nvc ? P.la[e] * kLog2e : 0.0f;
        gg += l2;
        const float kx = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(kin + sw128_off(t, kch)));
        LA[t * kD + i] = ex2(gg - R2);
        float kp;
        if (V == kVarDiag) {
            const float ox = t < nvc ? P.om[e] : 0.0f;
            const float al = ex2(l2), a2 = al * al, cc = sm[SM_MUR + t] * kx * kx;
            const float nn = fmaf(a2, pns, ox * pds);
            const float dd = fmaf(cc * a2, pns, fmaf(cc, ox, 1.0f) * pds);
            kp = nn * rcp_approx(pds) * ex2(R2 - gg);
            pns = nn;
            pds = dd;
            if ((t & 3) == 3) {
                const int ex = min((__float_as_int(pds) >> 23) & 0xff, 253);
                const float sc = __int_as_float((254 - ex) << 23);
                pns *= sc;
                pds *= sc;
            }
        } else if (ISO) {
            kp = ex2(R2 - gg);
        } else if (V == kVarGiven) {
            kp = (t < nvc ? P.om[e] : 0.0f) * ex2(R2 - gg);
        } else {
            const float A = fmaf(sm[SM_OMI + t], sts, sm[SM_MUR + t] * kx * kx);
            sts = A;
            const float rho = fmaf(lg2(fmaxf(A, kStatFloor)), kLn2, -center);
            const float sg = rho * rcp_approx(1.0f + fabsf(rho));
            kp = sm[SM_R + t] * ex2(fmaf(sg, P.neg_log2x, R2 - gg));
        }
        OM[t * kD + i] = kp;
    }
}

template <int V, int MODE>
__global__ void __launch_bounds__(kNT, 1) kdn_fused_tc_kernel(const __grid_constant__ TcParams P) {
    // MODE 0: whole sequences; 1: segments of a split sequence; 2: segments with the
    // values read as zero (a segment's transition map; no v copies)
    constexpr bool SEG = MODE != 0, NOV = MODE == 2;
    constexpr bool ISO = V == kVarIso, PK = V == kVarPkda, GK = V == kVarGiven;
    static_assert(!GK || MODE == 0, "given gains: whole sequences");
    // Measured per variant (A/B on the B8 H16 T4096 workloads): the diagonal blocks of
    // the triangular system by warp-level MMAs while the Gram MMA runs (DB), and the
    // inputs of the chunk after next prefetched into L2 (PF).
    constexpr bool DB = V == kVarPkda || V == kVarGiven;
    constexpr bool PF = V == kVarDiag || V == kVarPkda || V == kVarGiven;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_addr(base);
    float* sm = reinterpret_cast<float*>(base + OFF_SMALL);
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + SM_FLAG);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + OFF_BAR + 64);
    // inputs of a chunk arrive on three barriers: log_alpha (bar_la), k and omega
    // (bar_ko), q (bar_q), in the order the passes need them
    const uint32_t bar_la = sb + OFF_BAR, bar_v = bar_la + 8, bar_mma = bar_la + 16, bar_o = bar_la + 24,
                   bar_oj = bar_la + 32, bar_ops = bar_la + 40, bar_ko = bar_la + 48, bar_q = bar_la + 56,
                   bar_js = bar_la + 72,   // state update of a chunk (once per chunk, parity n & 1)
                   bar_probe = bar_la + 80;   // completed by nothing (timeout probe)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool wg0 = tid < 128, wg1 = tid >= 128 && tid < 256, wg2 = tid >= 256;
    const int vs = blockIdx.x, nseg = SEG ? P.nseg : 1;
    const int bh = SEG ? vs / nseg : vs, seg = SEG ? vs % nseg : 0, H = P.H, b = bh / H, h = bh % H;
    const int Tall = P.T, tb = SEG ? seg * P.seg_len : 0;   // sequence length, first token of the segment
    const int T = SEG ? min(P.seg_len, Tall - tb) : Tall;    // tokens of this CTA's segment
    const int nchunks = (T + kC - 1) / kC;

    if (tid == 0) {
        mbar_init(bar_la, 1);
        mbar_init(bar_ko, 1);
        mbar_init(bar_q, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_oj, 1);
        mbar_init(bar_ops, 1);
        mbar_init(bar_js, 1);
        mbar_init(bar_probe, 1);
        mbar_fence_init();
        *s_abort = 0;
    }
    if (warp == 0) {
        tmem_alloc(smem_addr(tmem_slot), TM_COLS);
        tc_fence_before();
    }

    auto issue_inputs = [&](int n) {
        const int t0 = n * kC;
        mbar_expect_tx(bar_la, 32768u);
        tma_load_4d(sb + OFF_LA, &P.tla, 0, h, tb + t0, b, bar_la);
        // (diagonal: omega; given gains: kappa, into the omega tile)
        mbar_expect_tx(bar_ko, (V == kVarDiag || GK) ? 49152u : 16384u);
        if (V == kVarDiag || GK) tma_load_4d(sb + OFF_OM, &P.tom, 0, h, tb + t0, b, bar_ko);
        tma_load_4d(sb + OFF_KIN, &P.tk, 0, h, tb + t0, b, bar_ko);
        tma_load_4d(sb + OFF_KIN + 8192, &P.tk, 64, h, tb + t0, b, bar_ko);
        mbar_expect_tx(bar_q, 16384u);
        tma_load_4d(sb + OFF_QIN, &P.tq, 0, h, tb + t0, b, bar_q);
        tma_load_4d(sb + OFF_QIN + 8192, &P.tq, 64, h, tb + t0, b, bar_q);
    };
    auto issue_v = [&](int n) {
        mbar_expect_tx(bar_v, 16384u);
        tma_load_4d(sb + OFF_VIN, &P.tv, 0, h, tb + n * kC, b, bar_v);
        tma_load_4d(sb + OFF_VIN + 8192, &P.tv, 64, h, tb + n * kC, b, bar_v);
    };
    // The tiles of chunk n into L2 (no shared memory written): issued while the copy
    // engine is idle, a chunk before their copy to shared memory, which then reads L2.
    auto prefetch_inputs = [&](int n) {
        const int t0 = tb + n * kC;
        tma_prefetch_4d(&P.tla, 0, h, t0, b);
        if (V == kVarDiag || GK) tma_prefetch_4d(&P.tom, 0, h, t0, b);
        tma_prefetch_4d(&P.tk, 0, h, t0, b);
        tma_prefetch_4d(&P.tk, 64, h, t0, b);
        tma_prefetch_4d(&P.tq, 0, h, t0, b);
        tma_prefetch_4d(&P.tq, 64, h, t0, b);
        if (!NOV) {
            tma_prefetch_4d(&P.tv, 0, h, t0, b);
            tma_prefetch_4d(&P.tv, 64, h, t0, b);
        }
    };
    __syncthreads();
    // copies and MMA commits issued so far (thread 0: v, MMAs; thread 256: the Gram MMAs;
    // thread 160: q, k, log_alpha, omega)
    int n_in_issued = 0, n_v_issued = 0, n_mma_issued = 0, n_o_issued = 0, n_oj_issued = 0, n_gram_issued = 0,
        n_js_issued = 0;
    if (tid == 0 && nchunks > 0 && !NOV) {
        issue_v(0);
        n_v_issued = 1;
    }
    if (tid == 160 && nchunks > 0) {
        issue_inputs(0);
        n_in_issued = 1;
    }
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);

    // per-thread recurrent state
    // diagonal: variance of channel tid - 128 (warps 4-7) in projective form p = pn / pd,
    // pd renormalised to [1, 2) by powers of two
    float pn = 1.0f, pd = 1.0f;
    float pend2 = 0.0f;   // pending log2-factor of the previous chunk, (G_C - G_ref) log2(e) (warps 4-7)
    float b_iso = 1.0f;   // isotropic scalar variance (warp 11)
    // PKDA: key statistic of channel tid - 128 (warps 4-7), and the head's centre
    float stat = 0.0f;
    const float center = PK ? P.center[h] : 0.0f;
    const float* p0v = !P.p0 ? nullptr
                       : SEG ? P.p0 + bh * P.p0_bh + seg * P.p0_seg
                             : P.p0 + static_cast<size_t>(bh) * (ISO ? 1 : kD);
    if (wg1 && V == kVarDiag && p0v) pn = p0v[tid - 128];
    if (wg1 && PK && p0v) stat = p0v[tid - 128];
    if (ISO && warp == 11 && p0v) b_iso = p0v[0];
    // initial state S^T into TMEM: lane j = value column, columns = key channel
    if (wg0) {
        const int j = tid;
        uint32_t r[32];
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const int i = q * 32 + c;
                r[c] = __float_as_uint((SEG && P.s0_identity) ? (i == j ? 1.0f : 0.0f)
                                       : P.S0 ? P.S0[(static_cast<size_t>(vs) * kD + i) * kD + j] : 0.0f);
            }
            tmem_st32(lane_base + TM_S + q * 32, r);
        }
        tmem_wait_st();
    } else {
        // blocks of T above the diagonal are never written: zero its bf16 tile once
        uint4* tt4 = reinterpret_cast<uint4*>(base + OFF_TT);
        for (int e = tid - 128; e < 8192 / 16; e += 256) tt4[e] = make_uint4(0u, 0u, 0u, 0u);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    uint32_t ph_in = 0, ph_v = 0;
    // bar_mma completes three phases per chunk n: Gram (parity n & 1, committed by
    // thread 256), innovations ((n + 1) & 1), state update (n & 1).  bar_o (prediction
    // and query MMA), bar_oj (output update) and bar_ops (operands built, an arrive by
    // thread 256) complete once per chunk, parity n & 1.
    auto wait_or_abort = [&](uint32_t bar, uint32_t parity) {
        if (*s_abort) return;
        if (!mbar_wait(bar, parity, kWaitLimit)) {
            set_status(P.status, kStatusTimeout);
            *s_abort = 1;
        }
    };
    auto tmem_ld64 = [&](uint32_t col, uint32_t (&v0)[32], uint32_t (&v1)[32]) {
        tmem_ld32(lane_base + col, v0);
        tmem_ld32(lane_base + col + 32, v1);
        tmem_wait_ld();
    };

    float* LA = reinterpret_cast<float*>(base + OFF_LA);
    float* OM = reinterpret_cast<float*>(base + OFF_OM);
    float* LF = reinterpret_cast<float*>(base + OFF_LF);
    float* TF = reinterpret_cast<float*>(base + OFF_TF);
    float* XT = reinterpret_cast<float*>(base + OFF_XT);

    // ------------------------------------------------------------------ warps 4-7
    // Per-token scalars of chunk c, then (inputs landed) the chunk's log-decay, the
    // uncertainty recurrence and the decay factors, written over the inputs in place.
    // Runs one chunk ahead of the memory pass.  Rows past the end of the sequence
    // arrive as zeros (TMA fill): log_alpha = omega = k = 0 leaves the variance and
    // the decay factor unchanged and zeroes those rows' operands.
    // Returns true when this channel's frame factor for chunk c is kept in two parts.
    auto prep_gains = [&](int c) -> bool {
        bool split = false;
        const int t0c = c * kC, nvc = min(kC, T - t0c);
        if (tid < 128 + kC) {
            const int t = tid - 128;
            if (PK) {
                // write strength, statistic weight and decay (rows past T leave the
                // statistic unchanged and write nothing)
                float be = 0.0f, bp = 0.0f, ap = 1.0f;
                if (t < nvc) {
                    const size_t th = (static_cast<size_t>(b) * Tall + tb + t0c + t) * H + h;
                    be = P.beta[th];
                    bp = P.beta_p[th];
                    ap = P.alpha_p[th];
                }
                sm[SM_R + t] = be;
                sm[SM_MUR + t] = bp;
                sm[SM_OMI + t] = ap;
            } else if (!GK) {
                float rr = 1.0f, om = 0.0f;
                if (t < nvc) {
                    const size_t th = (static_cast<size_t>(b) * Tall + tb + t0c + t) * H + h;
                    rr = P.r[th];
                    if (ISO) om = P.om[th];
                }
                sm[SM_R + t] = rr;
                sm[SM_RZ + (c & 1) * 64 + t] = rr;
                sm[SM_MUR + t] = P.mu / rr;
                sm[SM_OMI + t] = om;
                if (ISO) sm[SM_OMB + (c & 1) * 64 + t] = om;
            }
        }
        wait_or_abort(bar_la, ph_in);
        named_bar(kBarWG1, 128);
        const int i = tid - 128, w4 = warp - 4;
        wait_or_abort(bar_ko, ph_in);   // k and omega of chunk c
        // decay factors relative to the chunk start (reference checked after the chunk)
        const float pn0 = pn, pd0 = pd, stat0 = stat;
        float e1 = 1.0f, gr = 0.0f;   // e^{G_t}, and G_t log2(e) (PKDA)
        float2 g2 = make_float2(0.0f, 0.0f);   // chunk log-decay, log2 units, two partial sums
        const unsigned char* kin = base + OFF_KIN + (i >> 6) * 8192 + (i & 7) * 2;
        const int kch = (i & 63) >> 3;
        // Tokens per loop body: one short body (8 tokens for KDN, 16 for PKDA, each
        // measured fastest) keeps the code small; the isotropic variant unrolls the
        // bodies of a half for its per-half reductions.
        constexpr int kGB = PK ? 16 : 8, kGQ = 32 / kGB;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
            float w[32], w2[32];
#pragma unroll (ISO ? kGQ : 1)
            for (int qt = 0; qt < kGQ; ++qt) {
                const int tb = hf * 32 + qt * kGB;
                // loads first (independent of the carry) ...
                float la[kGB], kv[kGB], om[kGB], mr[kGB];
#pragma unroll
                for (int u = 0; u < kGB; ++u) {
                    const int t = tb + u;
                    la[u] = LA[t * kD + i];
                    kv[u] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(kin + sw128_off(t, kch)));
                    om[u] = (V == kVarDiag || GK) ? OM[t * kD + i] : 0.0f;
                }
#pragma unroll
                for (int u4 = 0; u4 < kGB / 4; ++u4) {
                    const float4 m4 = *reinterpret_cast<const float4*>(sm + SM_MUR + tb + 4 * u4);
                    mr[4 * u4 + 0] = m4.x;
                    mr[4 * u4 + 1] = m4.y;
                    mr[4 * u4 + 2] = m4.z;
                    mr[4 * u4 + 3] = m4.w;
                }
                // ... then the carries: variance and decay factors.  The variance map
                // p -> a^2 p + omega -> p_hat / (1 + c p_hat), c = mu k^2 / r, is the
                // Moebius matrix [[a^2, omega], [c a^2, 1 + c omega]] acting on (pn, pd):
                // two independent multiply-adds per token, p_hat_t = pn_t / pd_{t-1}.
                // Token-local factors are formed two tokens at a time (packed fp32 pairs).
                if (PK) {
                    // key statistic A = alpha_p A + beta_p k^2 (this token included), then
                    // the write scale exp(-log(x) s), s = softsign(log A - mu), times beta:
                    // the coefficient of the write key (Preconditioned DeltaNet Eq. 9)
                    float bp[kGB], ap[kGB], be[kGB];
#pragma unroll
                    for (int u4 = 0; u4 < kGB / 4; ++u4) {
                        const float4 b4 = *reinterpret_cast<const float4*>(sm + SM_MUR + tb + 4 * u4);
                        const float4 a4 = *reinterpret_cast<const float4*>(sm + SM_OMI + tb + 4 * u4);
                        const float4 w4 = *reinterpret_cast<const float4*>(sm + SM_R + tb + 4 * u4);
                        bp[4 * u4 + 0] = b4.x; bp[4 * u4 + 1] = b4.y; bp[4 * u4 + 2] = b4.z; bp[4 * u4 + 3] = b4.w;
                        ap[4 * u4 + 0] = a4.x; ap[4 * u4 + 1] = a4.y; ap[4 * u4 + 2] = a4.z; ap[4 * u4 + 3] = a4.w;
                        be[4 * u4 + 0] = w4.x; be[4 * u4 + 1] = w4.y; be[4 * u4 + 2] = w4.z; be[4 * u4 + 3] = w4.w;
                    }
#pragma unroll
                    for (int u = 0; u < kGB; u += 2) {
                        const int t = tb + u;
                        const float2 l2 = fmul2(make_float2(la[u], la[u + 1]), make_float2(kLog2e, kLog2e));
                        const float gr0 = gr + l2.x, gr1 = gr0 + l2.y;
                        gr = gr1;
                        const float al0 = ex2(l2.x), al1 = ex2(l2.y);
                        e1 *= al0;
                        LA[t * kD + i] = e1;
                        e1 *= al1;
                        LA[(t + 1) * kD + i] = e1;
                        const float2 kk = make_float2(kv[u], kv[u + 1]);
                        const float2 bk = fmul2(make_float2(bp[u], bp[u + 1]), fmul2(kk, kk));
                        const float A0 = fmaf(ap[u], stat, bk.x);
                        const float A1 = fmaf(ap[u + 1], A0, bk.y);
                        stat = A1;
                        const float2 rho = ffma2(make_float2(lg2(fmaxf(A0, kStatFloor)), lg2(fmaxf(A1, kStatFloor))),
                                                 make_float2(kLn2, kLn2), make_float2(-center, -center));
                        const float2 sg = fmul2(rho, make_float2(rcp_approx(1.0f + fabsf(rho.x)),
                                                                 rcp_approx(1.0f + fabsf(rho.y))));
                        // divided by the decay factor e1 = 2^{G_t log2 e} (the operand pass
                        // multiplies k by this directly)
                        const float2 ex = ffma2(sg, make_float2(P.neg_log2x, P.neg_log2x), make_float2(-gr0, -gr1));
                        OM[t * kD + i] = be[u] * ex2(ex.x);
                        OM[(t + 1) * kD + i] = be[u + 1] * ex2(ex.y);
                    }
                } else if (GK) {
                    // given gains: decay factors, and kappa / e1 over kappa in place
#pragma unroll
                    for (int u = 0; u < kGB; u += 2) {
                        const int t = tb + u;
                        const float2 l2 = fmul2(make_float2(la[u], la[u + 1]), make_float2(kLog2e, kLog2e));
                        g2 = fadd2(g2, l2);
                        e1 *= ex2(l2.x);
                        LA[t * kD + i] = e1;
                        OM[t * kD + i] = om[u] * rcp_approx(e1);
                        e1 *= ex2(l2.y);
                        LA[(t + 1) * kD + i] = e1;
                        OM[(t + 1) * kD + i] = om[u + 1] * rcp_approx(e1);
                    }
                } else if (!ISO) {
#pragma unroll
                    for (int u = 0; u < kGB; u += 2) {
                        const int t = tb + u;
                        const float2 l2 = fmul2(make_float2(la[u], la[u + 1]), make_float2(kLog2e, kLog2e));
                        g2 = fadd2(g2, l2);
                        const float al0 = ex2(l2.x), al1 = ex2(l2.y);
                        const float2 a2 = fmul2(make_float2(al0, al1), make_float2(al0, al1));
                        const float2 kk = make_float2(kv[u], kv[u + 1]);
                        const float2 cc = fmul2(make_float2(mr[u], mr[u + 1]), fmul2(kk, kk));
                        const float2 ca2 = fmul2(cc, a2);
                        const float2 ee = ffma2(cc, make_float2(om[u], om[u + 1]), make_float2(1.0f, 1.0f));
                        e1 *= al0;
                        LA[t * kD + i] = e1;
                        float rd = rcp_approx(pd * e1);
                        float2 nd = ffma2(make_float2(a2.x, ca2.x), make_float2(pn, pn),
                                          fmul2(make_float2(om[u], ee.x), make_float2(pd, pd)));
                        OM[t * kD + i] = nd.x * rd;   // p_hat_t / e1_t
                        pn = nd.x;
                        pd = nd.y;
                        e1 *= al1;
                        LA[(t + 1) * kD + i] = e1;
                        rd = rcp_approx(pd * e1);
                        nd = ffma2(make_float2(a2.y, ca2.y), make_float2(pn, pn),
                                   fmul2(make_float2(om[u + 1], ee.y), make_float2(pd, pd)));
                        OM[(t + 1) * kD + i] = nd.x * rd;
                        pn = nd.x;
                        pd = nd.y;
                        if ((u & 3) == 2) {   // exact rescale: pd back to [1, 2)
                            const int eb = min(__float_as_int(pd) & 0x7f800000, 253 << 23);
                            const float sc = __int_as_float(0x7f000000 - eb);   // 2^(127 - exponent)
                            pn *= sc;
                            pd *= sc;
                        }
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < kGB; ++u) {
                        const int t = tb + u;
                        const float l2 = la[u] * kLog2e;
                        g2.x += l2;
                        const float al = ex2(l2), a2 = al * al, k2 = kv[u] * kv[u];
                        e1 *= al;
                        LA[t * kD + i] = e1;
                        w[qt * kGB + u] = k2;
                        w2[qt * kGB + u] = t < nvc ? a2 : 0.0f;
                    }
                }
            }
            if (ISO) {
                sm[SM_ZP + (c & 1) * 256 + w4 * 64 + hf * 32 + lane] = butterfly_sum32(w, lane);
                sm[SM_AP + (c & 1) * 256 + w4 * 64 + hf * 32 + lane] = butterfly_sum32(w2, lane);
            }
        }
        {
            const float G2C = PK ? gr : g2.x + g2.y;
            if (!(fabsf(G2C) <= kMaxChunkLogDecay * kLog2e)) set_status(P.status, kStatusRange);
            float R2 = 0.0f;
            if (fabsf(G2C) > kStartRefLogDecay * kLog2e) {
                // rare: strong decay in this channel, recompute its factors with G_ref = G_C / 2
                // from log_alpha (and omega) in global memory (the tiles now hold the
                // factors), re-running the variance (statistic) recurrence of the chunk
                R2 = 0.5f * G2C;
                strong_decay_factors<V>(P, base, i, b, h, tb + t0c, nvc, R2, pn0, pd0, stat0, center);
            }
            // The frame factor 2^(pend2 + R2) of the state: each part is at least
            // 2^-116 (|G_C| <= 160), but after two strongly decaying chunks their sum
            // can leave the normal range, and ex2.approx.ftz would flush it to zero.
            // Such chunks keep the two parts apart and the state is scaled twice
            // (2^pend2 brings it to its true scale, 2^R2 into the chunk's frame).
            split = pend2 + R2 < -120.0f;
            sm[SM_CF + (c & 1) * 128 + i] = split ? ex2(pend2) : ex2(pend2 + R2);
            sm[SM_CF2 + i] = ex2(R2);
            pend2 = G2C - R2;
            sm[SM_FOUT + i] = ex2(pend2);
        }
        return split;
    };

    // Isotropic: the scalar variance recurrence of chunk c (warp 11, after the operand
    // pass, beside the Gram MMA).  The write keys K_til' = k / e1 carry no b_hat, so
    // b_hat_s scales column s of the Gram matrix; dividing row t of the triangular
    // system by b_hat_t instead gives the diagonal z_t / b_hat_t = r_t / b_hat_t +
    // ||k_t||^2 (the Gram diagonal is ||k_t||^2) and innovations multiplied by b_hat_t,
    // which the update and query-write products then take with the unscaled keys.
    // So b_hat enters only as r_t / b_hat_t in the diagonal, written here.
    auto iso_scan = [&](int c, int nvc) {
        const float* zp = sm + SM_ZP + (c & 1) * 256;
        const float* ap = sm + SM_AP + (c & 1) * 256;
        float* rz = sm + SM_RZ + (c & 1) * 64;
        // Moebius scan over the chunk, 2 tokens per lane
        float aa[2], uu[2], oo[2], rr[2];
        Mob m[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int t = 2 * lane + e;
            const float kk = zp[t] + zp[64 + t] + zp[128 + t] + zp[192 + t];
            aa[e] = (ap[t] + ap[64 + t] + ap[128 + t] + ap[192 + t]) * (1.0f / kD);
            rr[e] = rz[t];
            oo[e] = sm[SM_OMB + (c & 1) * 64 + t];
            uu[e] = __fdividef(P.mu * kk, kD * rr[e]);
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
        float bb = __fdividef(fmaf(ex.a, b_iso, ex.b), fmaf(ex.c, b_iso, ex.d));
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int t = 2 * lane + e;
            if (t < nvc) {
                const float bhat = fmaf(aa[e], bb, oo[e]);
                bb = __fdividef(bhat, fmaf(uu[e], bhat, 1.0f));
                // b_hat = 0 (no prior variance, no process noise): a large finite
                // diagonal gives a zero innovation, the zero gain
                rz[t] = __fdividef(rr[e], fmaxf(bhat, 1e-30f));
            }
        }
        b_iso = __shfl_sync(0xffffffffu, bb, 31);
    };

    // ------------------------------------------------------------------ warps 0-3
    // Outputs of a finished chunk: thread j holds column j of the [64 t][128 j] tile
    // (its O^T row in TMEM) and stores it directly; a warp writes 64 contiguous bytes
    // per token.  Rows past T are skipped.
    auto emit_outputs = [&](int c) {
        uint32_t v0[32], v1[32];
        tc_fence_after();
        tmem_ld64(TM_O, v0, v1);
        const int t0c = c * kC, nvc = min(kC, T - t0c);
        __nv_bfloat16* og =
            P.o + (static_cast<size_t>(b) * Tall + tb + t0c) * H * kD + static_cast<size_t>(h) * kD + tid;
        const size_t ts = static_cast<size_t>(H) * kD;
        if (nvc == kC) {
#pragma unroll
            for (int t = 0; t < kC; ++t) og[t * ts] = __float2bfloat16_rn(__uint_as_float(t < 32 ? v0[t] : v1[t - 32]));
        } else {
#pragma unroll
            for (int t = 0; t < kC; ++t)
                if (t < nvc) og[t * ts] = __float2bfloat16_rn(__uint_as_float(t < 32 ? v0[t] : v1[t - 32]));
        }
    };
    // State of chunk c into its reference frame: S_m^T = S^T diag(cf) in TMEM, and
    // its bf16 copy (A operand of the query and prediction MMA) in TMEM.
    auto scale_state = [&](int c) {
        tc_fence_after();
#pragma unroll 1
        for (int q2 = 0; q2 < 2; ++q2) {
            uint32_t r0[32], r1[32], pk[32];
            tmem_ld64(TM_S + 64 * q2, r0, r1);
            // (two channels per packed multiply)
            auto scale4 = [](uint32_t* r, const float4 f) {
                const float2 a = fmul2(make_float2(__uint_as_float(r[0]), __uint_as_float(r[1])), make_float2(f.x, f.y));
                const float2 b = fmul2(make_float2(__uint_as_float(r[2]), __uint_as_float(r[3])), make_float2(f.z, f.w));
                r[0] = __float_as_uint(a.x);
                r[1] = __float_as_uint(a.y);
                r[2] = __float_as_uint(b.x);
                r[3] = __float_as_uint(b.y);
            };
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                scale4(r0 + 4 * c4, *reinterpret_cast<const float4*>(sm + SM_CF + (c & 1) * 128 + 64 * q2 + 4 * c4));
                scale4(r1 + 4 * c4, *reinterpret_cast<const float4*>(sm + SM_CF + (c & 1) * 128 + 64 * q2 + 32 + 4 * c4));
            }
            tmem_st32(lane_base + TM_S + 64 * q2, r0);
            tmem_st32(lane_base + TM_S + 64 * q2 + 32, r1);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                pk[e] = pack_bf16(__uint_as_float(r0[2 * e]), __uint_as_float(r0[2 * e + 1]));
                pk[16 + e] = pack_bf16(__uint_as_float(r1[2 * e]), __uint_as_float(r1[2 * e + 1]));
            }
            tmem_st32(lane_base + TM_SMB + 32 * q2, pk);
        }
        tmem_wait_st();
    };

    // O^T += Delta'^T A'^T of a finished chunk (thread 0; Delta' in TMEM and A' stay
    // intact until the next chunk's prediction readout and Gram readout)
    auto issue_output_update = [&]() {
        tc_fence_after();
        const uint32_t id_o = idesc_bf16(128, 64, 0, 0, 0);
        const uint64_t d_aq = sw128_desc(sb + OFF_AQ, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            mma_bf16_tmem_a(tmem + TM_O, tmem + TM_DB + 8 * ks, desc_add(d_aq, ks * 32), id_o, 1u);
        mma_commit(bar_oj);
        ++n_oj_issued;
    };

    // Timeout probe (a test of the bounded-wait path): the gains warps wait, with a
    // short bound, on a barrier that nothing completes while chunk 0's copies are in
    // flight; the wait gives up, records KDN_ERR_TIMEOUT and the CTA takes its abort
    // path (no MMA issued, copies in flight drained before exit).
    if (P.probe && wg1 && !*s_abort && !mbar_wait(bar_probe, 0u, kProbeWaitLimit)) {
        set_status(P.status, kStatusTimeout);
        *s_abort = 1;
    }
    if (wg1 && nchunks > 0) prep_gains(0);   // chunk 0 never splits: pend2 = 0
    ph_in ^= 1u;
    tc_fence_before();
    __syncthreads();

#pragma unroll 1
    for (int n = 0; n < nchunks; ++n) {
        const int t0 = n * kC, nv = min(kC, T - t0);
        const uint32_t pb = static_cast<uint32_t>(n) & 1u;
        // ================= step 1: state frame, outputs of chunk n-1, prediction/query MMA
        //                   || operands, Gram MMA, prefetch of chunk n+1
        if (wg0) {
            if (tid == 0 && n > 0 && !*s_abort) issue_output_update();   // of chunk n-1
            scale_state(n);
            if (n > 0) {
                wait_or_abort(bar_oj, pb ^ 1u);   // output update of chunk n-1 has landed
                if (!(SEG && P.no_o)) emit_outputs(n - 1);
            }
            tc_fence_before();
            named_bar(kBarWG0, 128);
            // [Z^T | O^T] = S_m^T [K_bar; Q_bar]^T  (N = 128: prediction and query together)
            if (tid == 0 && !*s_abort) {
                wait_or_abort(bar_ops, pb);   // operands built (warps 4-11)
                tc_fence_after();
                const uint32_t id_zo = idesc_bf16(128, 128, 0, 0, 0);
                const uint64_t d_kq = sw128_desc(sb + OFF_KQ, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_tmem_a(tmem + TM_ZD, tmem + TM_SMB + 8 * ks,
                                    desc_add(d_kq, (ks >> 2) * 16384 + (ks & 3) * 32), id_zo,
                                    ks > 0);
                mma_commit(bar_o);
                ++n_o_issued;
            }
        } else {
            // decayed bf16 operands (warps 4-11): thread -> 4 channels in each K-atom
            // (8-byte pieces of the swizzled rows), 16 threads (half a warp) per token row.
            // K_til' = p_hat k / e1 (isotropic: k / e1); the gain denominator enters
            // through the diagonal of the triangular system.
            const int u = tid - 128, g = u & 15, tr = u >> 4;
            wait_or_abort(bar_q, pb);   // q of chunk n
#pragma unroll 2
            for (int m4 = 0; m4 < 4; ++m4) {
                const int t = tr + 16 * m4;
                const uint32_t sw = sw128_off(t, g >> 1) + (g & 1) * 8;
                float kb[8], qb[8], kt[8];
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    const uint2 kr = *reinterpret_cast<const uint2*>(base + OFF_KIN + a * 8192 + sw);
                    const uint2 qr = *reinterpret_cast<const uint2*>(base + OFF_QIN + a * 8192 + sw);
                    const float4 e = *reinterpret_cast<const float4*>(LA + t * kD + 64 * a + 4 * g);
                    // p_hat / e1 (PKDA: write scale / e1; given gains: kappa / e1), formed by
                    // warps 4-7; isotropic: 1 / e1
                    float4 kp;
                    if (ISO) {
                        kp = make_float4(rcp_approx(e.x), rcp_approx(e.y), rcp_approx(e.z), rcp_approx(e.w));
                    } else {
                        kp = *reinterpret_cast<const float4*>(OM + t * kD + 64 * a + 4 * g);
                    }
                    const float k0 = bf_lo(kr.x), k1 = bf_hi(kr.x), k2 = bf_lo(kr.y), k3 = bf_hi(kr.y);
                    kb[4 * a + 0] = k0 * e.x;
                    kb[4 * a + 1] = k1 * e.y;
                    kb[4 * a + 2] = k2 * e.z;
                    kb[4 * a + 3] = k3 * e.w;
                    qb[4 * a + 0] = bf_lo(qr.x) * e.x;
                    qb[4 * a + 1] = bf_hi(qr.x) * e.y;
                    qb[4 * a + 2] = bf_lo(qr.y) * e.z;
                    qb[4 * a + 3] = bf_hi(qr.y) * e.w;
                    // (given gains: the tile holds kappa / e1, the write key itself)
                    kt[4 * a + 0] = GK ? kp.x : k0 * kp.x;
                    kt[4 * a + 1] = GK ? kp.y : k1 * kp.y;
                    kt[4 * a + 2] = GK ? kp.z : k2 * kp.z;
                    kt[4 * a + 3] = GK ? kp.w : k3 * kp.w;
                }
#pragma unroll
                for (int a = 0; a < 2; ++a) {
                    *reinterpret_cast<uint2*>(base + OFF_KQ + a * 16384 + sw) =
                        make_uint2(pack_bf16(kb[4 * a], kb[4 * a + 1]), pack_bf16(kb[4 * a + 2], kb[4 * a + 3]));
                    *reinterpret_cast<uint2*>(base + OFF_KQ + a * 16384 + 8192 + sw) =
                        make_uint2(pack_bf16(qb[4 * a], qb[4 * a + 1]), pack_bf16(qb[4 * a + 2], qb[4 * a + 3]));
                    *reinterpret_cast<uint2*>(base + OFF_KT + a * 8192 + sw) =
                        make_uint2(pack_bf16(kt[4 * a], kt[4 * a + 1]), pack_bf16(kt[4 * a + 2], kt[4 * a + 3]));
                }
            }
            fence_proxy_async();
            tc_fence_before();
            named_bar(kBarOps, 256);
            // Gram MMA (thread 256, whose warps read it out next) and the next inputs (thread 160)
            if (tid == 256 && !*s_abort) {
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 64, 0, 0, 0);
                const uint64_t d_kq = sw128_desc(sb + OFF_KQ, 16, 1024), d_kt = sw128_desc(sb + OFF_KT, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t ad = desc_add(d_kq, (ks >> 2) * 16384 + (ks & 3) * 32);
                    const uint64_t bd = desc_add(d_kt, (ks >> 2) * 8192 + (ks & 3) * 32);
                    mma_bf16(tmem + TM_G, ad, bd, id, ks > 0);
                }
                mma_commit(bar_mma);
                ++n_gram_issued;
                mbar_arrive(bar_ops);
            }
            if (tid == 160 && !*s_abort && n + 1 < nchunks) {   // the operand pass has consumed the inputs
                issue_inputs(n + 1);
                ++n_in_issued;
            }
        }
        // ================= step 3
        if (wg2) {
            const int lt = tid - 256, lw = warp - 8;
            unsigned char* tt = base + OFF_TT;
            const int g8 = lane >> 2, q4 = lane & 3;
            // ---- T = M^{-1}, first its 16x16 diagonal blocks; each finished block also
            //      goes to the bf16 tile T [t][s] (its blocks above the diagonal stay zero
            //      from the start)
            auto invert_diagonal_blocks = [&]() {
                if (lt < 64) {  // 16x16 diagonal blocks: right-looking substitution, one column per thread
                    const int blk = lt >> 4, c = lt & 15, o = 16 * blk;
                    float acc[16], inv[16];
#pragma unroll
                    for (int r4 = 0; r4 < 4; ++r4) {
                        const float4 d4 = *reinterpret_cast<const float4*>(sm + SM_INVD + o + 4 * r4);
                        inv[4 * r4 + 0] = d4.x;
                        inv[4 * r4 + 1] = d4.y;
                        inv[4 * r4 + 2] = d4.z;
                        inv[4 * r4 + 3] = d4.w;
                    }
#pragma unroll
                    for (int r = 0; r < 16; ++r) acc[r] = (r == c) ? 1.0f : 0.0f;
#pragma unroll
                    for (int s4 = 0; s4 < 16; s4 += 4) {
                        // columns s4..s4+3 of the rows below, one 16-byte load per row
                        float4 lq[16];
#pragma unroll
                        for (int r = s4 + 1; r < 16; ++r)
                            lq[r] = *reinterpret_cast<const float4*>(LF + (o + r) * kLDF + o + s4);
#pragma unroll
                        for (int s = s4; s < s4 + 4; ++s) {
                            const float xs = acc[s] * inv[s];
                            acc[s] = xs;
#pragma unroll
                            for (int r = s + 1; r < 16; ++r) {
                                const float4 q = lq[r];
                                const float l = (s & 3) == 0 ? q.x : (s & 3) == 1 ? q.y : (s & 3) == 2 ? q.z : q.w;
                                acc[r] = fmaf(-l, xs, acc[r]);
                            }
                        }
                    }
                    __nv_bfloat16* tcol = reinterpret_cast<__nv_bfloat16*>(tt + ((o + c) & 7) * 2);
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        TF[(o + r) * kLDF + o + c] = acc[r];
                        *reinterpret_cast<__nv_bfloat16*>(reinterpret_cast<unsigned char*>(tcol) +
                                                           sw128_off(o + r, (o + c) >> 3)) = __float2bfloat16_rn(acc[r]);
                    }
                }
            };
            // M = diag(r) + lower_incl(K_bar K_til'^T) (KDN): its diagonal is the gain
            // denominator z_t = r_t + sum_i p_hat_t,i k_t,i^2 (the decay factors cancel).
            // Isotropic: M'' = diag(r / b_hat) + lower_incl(K_bar K_til''^T), its diagonal
            // r_t / b_hat_t + ||k_t||^2.  PKDA and given gains: M = I + strict_lower(K_bar K_til^T).
            auto set_diagonal = [&](int t) {   // z_t on the diagonal of row t, 1 / z_t, beta_eff
                float* row = LF + t * kLDF;
                if (PK || GK) {
                    row[t] = 1.0f;
                    sm[SM_INVD + t] = 1.0f;
                } else {
                    const float g = row[t];
                    const float z = sm[SM_RZ + pb * 64 + t] + g;
                    row[t] = z;
                    sm[SM_INVD + t] = rcp_approx(z);
                    // effective write strength k^T kappa = (z - r) / z: the Gram diagonal
                    // over z (isotropic: both divided by b_hat)
                    if (!SEG && P.beta_eff && t < nv)
                        P.beta_eff[(static_cast<size_t>(b) * Tall + t0 + t) * H + h] = g / z;
                }
            };
            if (ISO && lw == 3) iso_scan(n, nv);   // gain denominators of chunk n (r / b_hat)
            if (DB) {
                // The diagonal blocks of M straight from the operand tiles (warp-level bf16
                // MMAs, warp lw -> block lw), inverted while the Gram MMA runs; the Gram's
                // readout then only fills the blocks below them.
                float x[2][4];
                gram_block16(x, sb + OFF_KQ, 16384u, sb + OFF_KT, 8192u, 16 * lw, 16 * lw, lane);
                store_tile_16x16(x, LF + (16 * lw) * kLDF + 16 * lw, kLDF, 1.0f, g8, q4);
                if (ISO) named_bar(kBarWG2, 128);   // the scan's r / b_hat
                else __syncwarp();
                if (lane < 16) set_diagonal(16 * lw + lane);
                named_bar(kBarWG2, 128);
                invert_diagonal_blocks();
            } else if (ISO) {
                named_bar(kBarWG2, 128);
            }
            // ---- Gram rows out of TMEM: M (fp32), query-write matrix A' (bf16)
            {
                wait_or_abort(bar_mma, pb);
                if (n > 0) wait_or_abort(bar_oj, pb ^ 1u);   // A' of chunk n-1 has been read
                tc_fence_after();
                uint32_t v0[32], v1[32];
                tmem_ld64(TM_G, v0, v1);
                if (lt < 64) {
                    // the whole row, or the blocks left of the diagonal block
                    float* row = LF + lt * kLDF;
                    const int nc4 = DB ? 4 * (lt >> 4) : 16;
#pragma unroll
                    for (int c4 = 0; c4 < 16; ++c4) {
                        const int s = 4 * c4;
                        if (c4 < nc4)
                            *reinterpret_cast<float4*>(row + s) =
                                make_float4(__uint_as_float(s + 0 < 32 ? v0[s + 0] : v1[s + 0 - 32]),
                                            __uint_as_float(s + 1 < 32 ? v0[s + 1] : v1[s + 1 - 32]),
                                            __uint_as_float(s + 2 < 32 ? v0[s + 2] : v1[s + 2 - 32]),
                                            __uint_as_float(s + 3 < 32 ? v0[s + 3] : v1[s + 3 - 32]));
                    }
                    if (!DB) set_diagonal(lt);   // (its own row, read back)
                } else {
                    const int t = lt - 64;
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
            tc_fence_before();
            named_bar(kBarWG2, 128);
            if (!DB) {
                invert_diagonal_blocks();
                named_bar(kBarWG2, 128);
            }
            if (lw < 2) {  // 16 -> 32 merges: T_ij = -T_ii (M_ij T_jj), (i, j) = (1, 0), (3, 2)
                const int i = 2 * lw + 1, j = 2 * lw;
                float x[2][4];
                mma_tile_16x16(x, LF + (16 * i) * kLDF + 16 * j, kLDF, TF + (16 * j) * kLDF + 16 * j, kLDF, 2);
                float* xs = XT + (16 * lw) * kLDX;
                store_tile_16x16(x, xs, kLDX, 1.0f, g8, q4);
                __syncwarp();
                mma_tile_16x16(x, TF + (16 * i) * kLDF + 16 * i, kLDF, xs, kLDX, 2);
                store_tile_16x16(x, TF + (16 * i) * kLDF + 16 * j, kLDF, -1.0f, g8, q4);
                store_tile_bf16(x, tt, 16 * i, 16 * j, -1.0f, g8, q4);
            }
            named_bar(kBarWG2, 128);
            {  // 32 -> 64: X = M[32:64, 0:32] T[0:32, 0:32]; T[32:64, 0:32] = -T[32:64, 32:64] X
                const int mt = lw >> 1, nt0 = 2 * (lw & 1);
                float x[2][4];
                // T[0:16, 16:32] is zero: columns 16-31 take k-steps 2-3 only
                mma_tile_16xN(x, LF + (32 + 16 * mt) * kLDF, kLDF, TF + 8 * nt0, kLDF, nt0 >= 2 ? 2 : 0, 4);
                store_tile_16x16(x, XT + (16 * mt) * kLDX + 8 * nt0, kLDX, 1.0f, g8, q4);
                named_bar(kBarWG2, 128);
                // T[32:48, 48:64] is zero: rows 32-47 take k-steps 0-1 only
                mma_tile_16xN(x, TF + (32 + 16 * mt) * kLDF + 32, kLDF, XT + 8 * nt0, kLDX, 0, mt == 0 ? 2 : 4);
                store_tile_bf16(x, tt, 32 + 16 * mt, 8 * nt0, -1.0f, g8, q4);
            }
            fence_proxy_async();
            named_bar(kBarTReady, 256);   // -> warps 0-3 issue the innovation MMAs
        } else if (wg0) {
            // ---- Y^T = V^T - Z^T (innovation before the triangular solve; Z^T = S_m^T K_bar^T
            //      is the prediction) -> bf16 A operand in TMEM
            {
                wait_or_abort(bar_o, pb);
                if (!NOV) wait_or_abort(bar_v, ph_v);
                tc_fence_after();
                uint32_t v0[32], v1[32], pk[32];
                tmem_ld64(TM_ZD, v0, v1);
                // column j = tid of the v tile (two [64 t][64 j] swizzled boxes)
                const unsigned char* vcol = base + OFF_VIN + (tid >> 6) * 8192 + (tid & 7) * 2;
                const int jc = (tid & 63) >> 3;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int t = 2 * e;
                    // (no_v: the segment's transition map, values zero)
                    const float va = NOV ? 0.0f : __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(vcol + sw128_off(t, jc)));
                    const float vb = NOV ? 0.0f : __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(vcol + sw128_off(t + 1, jc)));
                    const float za = __uint_as_float(t < 32 ? v0[t] : v1[t - 32]);
                    const float zb = __uint_as_float(t + 1 < 32 ? v0[t + 1] : v1[t + 1 - 32]);
                    pk[e] = pack_bf16(va - za, vb - zb);
                }
                tmem_st32(lane_base + TM_DB, pk);
                tmem_wait_st();
            }
            ph_v ^= 1u;
            fence_proxy_async();   // v has been read: the next chunk's copy may overwrite it
            // (chunk n + 1's tiles landed before the gains pass; chunk n + 2's copies are
            //  issued after chunk n + 1's operand pass)
            if (PF && tid == 32 && n + 2 < nchunks) prefetch_inputs(n + 2);
            tc_fence_before();
            // ---- Delta'^T = Y^T T^T
            named_bar(kBarTReady, 256);
            if (tid == 0 && !*s_abort) {
                tc_fence_after();
                const uint32_t id_y = idesc_bf16(128, 64, 0, 0, 0);
                const uint64_t d_tt = sw128_desc(sb + OFF_TT, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_tmem_a(tmem + TM_ZD, tmem + TM_DB + 8 * ks, desc_add(d_tt, ks * 32),
                                    id_y, ks > 0);
                mma_commit(bar_mma);
                ++n_mma_issued;
                if (n + 1 < nchunks && !NOV) {
                    issue_v(n + 1);
                    ++n_v_issued;
                }
            }
            // ---- Delta'^T -> bf16 in TMEM (A operand)
            {
                wait_or_abort(bar_mma, pb ^ 1u);
                tc_fence_after();
                uint32_t v0[32], v1[32], pk[32];
                tmem_ld64(TM_ZD, v0, v1);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    pk[e] = pack_bf16(__uint_as_float(v0[2 * e]), __uint_as_float(v0[2 * e + 1]));
                    pk[16 + e] = pack_bf16(__uint_as_float(v1[2 * e]), __uint_as_float(v1[2 * e + 1]));
                }
                tmem_st32(lane_base + TM_DB, pk);
                tmem_wait_st();
            }
            tc_fence_before();
            named_bar(kBarWG0, 128);
            // ---- S^T += Delta'^T K_til' (the next chunk starts from it); the output part
            //      O^T += Delta'^T A'^T is issued at the start of the next chunk
            if (tid == 0 && !*s_abort) {
                tc_fence_after();
                const uint32_t id_s = idesc_bf16(128, 128, 0, 1, 0);
                const uint64_t d_ktm = sw128_desc(sb + OFF_KT, 8192, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16_tmem_a(tmem + TM_S, tmem + TM_DB + 8 * ks, desc_add(d_ktm, ks * 2048),
                                    id_s, 1u);
                mma_commit(bar_mma);
                mma_commit(bar_js);
                ++n_mma_issued;
                ++n_js_issued;
            }
        } else if (n + 1 < nchunks) {
            // ---- warps 4-7: gains of chunk n + 1
            const bool split = prep_gains(n + 1);
            if (bar_red_or(kBarWG1, 128, split)) {
                // rare: some channel's frame factor for chunk n + 1 is kept in two parts;
                // once this chunk's state update has landed, these warps (the same TMEM
                // lanes) apply the second part; the first comes with the next chunk's
                // scaling, after the barrier that ends this chunk
                wait_or_abort(bar_js, pb);
                tc_fence_after();
                rescale_state_rows(lane_base, sm + SM_CF2);
                tmem_wait_st();
                tc_fence_before();
            }
        }
        if (n + 1 < nchunks) ph_in ^= 1u;
        // the next chunk starts from the updated state (and overwrites K_til')
        if (wg0) wait_or_abort(bar_mma, pb);
        tc_fence_before();
        __syncthreads();
        if (*s_abort) break;
    }

    if (tid == 0 && nchunks > 0 && !*s_abort) issue_output_update();   // of the last chunk
    const bool aborted = *s_abort != 0;
    if (!aborted && nchunks > 0) {
        wait_or_abort(bar_mma, static_cast<uint32_t>(nchunks - 1) & 1u);   // update of the last chunk has landed
        wait_or_abort(bar_oj, static_cast<uint32_t>(nchunks - 1) & 1u);
        if (wg0 && !(SEG && P.no_o)) emit_outputs(nchunks - 1);
    }
    if (!*s_abort) {
        // final state: S_T = (TMEM state) scaled by the last chunk's pending factor
        // (sequence split: only the last segment writes the sequence's final state,
        //  unless every segment's final state is wanted, at its CTA index; the
        //  final variances come from the last segment when p_T is given)
        const bool last = seg == nseg - 1, last_only = !SEG || P.last_only;
        const size_t st_idx = last_only ? static_cast<size_t>(bh) : static_cast<size_t>(vs);
        if (wg0 && (last || !last_only)) {
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
                    P.S_T[(st_idx * kD + i) * kD + j] = __uint_as_float(r[c]) * f;
                }
            }
        } else if (wg1 && last && P.p_T) {
            if (V == kVarDiag) P.p_T[static_cast<size_t>(bh) * kD + tid - 128] = pn / pd;
            else if (PK) P.p_T[static_cast<size_t>(bh) * kD + tid - 128] = stat;
        } else if (ISO && tid == 352 && last && P.p_T) {
            P.p_T[bh] = b_iso;
        }
    }
    int* s_ngram = reinterpret_cast<int*>(sm + SM_FLAG + 1);
    if (tid == 256) *s_ngram = n_gram_issued;
    tc_fence_before();
    __syncthreads();
    if (*s_abort) {
        // let copies and MMAs already issued land before the CTA's resources go away
        if (tid == 0) {
            const int nm = n_mma_issued + *s_ngram;
            if (nm > 0) mbar_wait(bar_mma, (nm - 1) & 1, kWaitLimit);
            if (n_o_issued > 0) mbar_wait(bar_o, (n_o_issued - 1) & 1, kWaitLimit);
            if (n_oj_issued > 0) mbar_wait(bar_oj, (n_oj_issued - 1) & 1, kWaitLimit);
            if (n_v_issued > 0) mbar_wait(bar_v, (n_v_issued - 1) & 1, kWaitLimit);
            if (n_js_issued > 0) mbar_wait(bar_js, (n_js_issued - 1) & 1, kWaitLimit);
        }
        if (tid == 160 && n_in_issued > 0) {
            mbar_wait(bar_la, (n_in_issued - 1) & 1, kWaitLimit);
            mbar_wait(bar_ko, (n_in_issued - 1) & 1, kWaitLimit);
            mbar_wait(bar_q, (n_in_issued - 1) & 1, kWaitLimit);
        }
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

// The split runs on one wave of CTAs (one per SM of the current device; 152 on
// GB300, also taken when no device can be queried), with segments of at least
// kMinSegTokens tokens.
constexpr int kDefaultSMs = 152, kMinSegTokens = 1024;

int split_ctas() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();   // no device here: keep the GB300 plan
        return kDefaultSMs;
    }
    return n;
}

TcSplit tc_split_plan(int B, int T, int H, uint32_t flags) {
    TcSplit sp;
    sp.seg_len = T;
    const long long BH = static_cast<long long>(B) * H;
    const int ctas = split_ctas();
    if ((flags & KDN_FLAG_NO_SPLIT) || BH <= 0 || 2 * BH > ctas) return sp;
    long long nseg = ctas / BH;
    if (nseg > T / kMinSegTokens) nseg = T / kMinSegTokens;
    if (nseg < 2) return sp;
    const int G = kGainChunk;   // a multiple of the chunk: segments start on gain-chunk carries
    const long long per = (T + nseg - 1) / nseg;
    const int seg_len = static_cast<int>((per + G - 1) / G * G);
    const int n = (T + seg_len - 1) / seg_len;
    if (n < 2) return sp;
    sp.nseg = n;
    sp.seg_len = seg_len;
    return sp;
}

// carries (2 launches), segment maps (2), chaining (1), output correction (1)
int tc_kernel_count(int nseg) { return nseg > 1 ? 6 : 1; }

cudaError_t launch_forward_tc(const ForwardArgs& a, const TcSplit& sp, cudaStream_t s) {
    TcParams P;
    memset(&P, 0, sizeof(P));
    const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    bool ok = encode_4d(&P.tq, a.q, BF, 2, a.B, a.T, a.H, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_4d(&P.tk, a.k, BF, 2, a.B, a.T, a.H, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_4d(&P.tv, a.v, BF, 2, a.B, a.T, a.H, 64, CU_TENSOR_MAP_SWIZZLE_128B) &&
              encode_4d(&P.tla, a.log_alpha, F32, 4, a.B, a.T, a.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (ok && (a.variant == kVarDiag || a.variant == kVarGiven))   // omega, or the given kappa
        ok = encode_4d(&P.tom, a.omega, F32, 4, a.B, a.T, a.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return cudaErrorInvalidValue;
    if (a.variant == kVarGiven && sp.nseg > 1) return cudaErrorInvalidValue;   // whole sequences only
    P.r = a.r;
    P.la = a.log_alpha;
    P.om = a.omega;
    P.beta = a.beta;
    P.alpha_p = a.alpha_p;
    P.beta_p = a.beta_p;
    P.center = a.center;
    P.neg_log2x = a.neg_log2x;
    P.S0 = a.S0;
    P.p0 = a.p0;
    P.o = static_cast<__nv_bfloat16*>(a.o);
    P.S_T = a.S_T;
    P.p_T = a.p_T;
    P.status = a.status;
    P.T = a.T;
    P.H = a.H;
    P.mu = a.mu;
    const int nu = a.variant == kVarIso ? 1 : kD;
    P.nseg = 1;
    P.seg_len = a.T;
    P.last_only = 1;
    P.p0_bh = nu;
    P.p0_seg = 0;
    P.probe = (a.flags & KDN_FLAG_TIMEOUT_PROBE) ? 1 : 0;
    // (the split path never writes the effective write strength: its callers keep
    //  one CTA per sequence when they want it)
    P.beta_eff = (sp.nseg > 1 || a.variant == kVarPkda || a.variant == kVarGiven) ? nullptr : a.beta_eff;
    int grid = a.B * a.H;
    auto launch = [&](auto kernel) {
        const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
        if (e != cudaSuccess) return e;
        kernel<<<grid, kNT, kSmemAlloc, s>>>(P);
        return cudaGetLastError();
    };
    // kernel instance: whole sequences, segments, or segments without values
    auto run = [&]() {
        if (P.nseg <= 1) {
            if (a.variant == kVarGiven) return launch(kdn_fused_tc_kernel<kVarGiven, 0>);
            if (a.variant == kVarDiag) return launch(kdn_fused_tc_kernel<kVarDiag, 0>);
            if (a.variant == kVarIso) return launch(kdn_fused_tc_kernel<kVarIso, 0>);
            return launch(kdn_fused_tc_kernel<kVarPkda, 0>);
        }
        if (P.no_v) {
            if (a.variant == kVarDiag) return launch(kdn_fused_tc_kernel<kVarDiag, 2>);
            if (a.variant == kVarIso) return launch(kdn_fused_tc_kernel<kVarIso, 2>);
            return launch(kdn_fused_tc_kernel<kVarPkda, 2>);
        }
        if (a.variant == kVarDiag) return launch(kdn_fused_tc_kernel<kVarDiag, 1>);
        if (a.variant == kVarIso) return launch(kdn_fused_tc_kernel<kVarIso, 1>);
        return launch(kdn_fused_tc_kernel<kVarPkda, 1>);
    };
    if (sp.nseg <= 1) return run();

    // ---- sequence split: every segment's initial uncertainty (statistic) from the scan
    ScanWorkspace w;
    w.kappa = nullptr;
    w.summary = sp.summary;
    w.carry = sp.carry;
    w.chunk_g = kGainChunk;
    w.n_chunks_g = sp.n_chunks_g;
    cudaError_t e = launch_scan_carries(a, w, s);
    if (e != cudaSuccess) return e;
    P.nseg = sp.nseg;
    P.seg_len = sp.seg_len;
    P.p0 = sp.carry;
    P.p0_bh = static_cast<long long>(sp.n_chunks_g) * nu;
    P.p0_seg = static_cast<long long>(sp.seg_len / kGainChunk) * nu;
    grid = a.B * a.H * sp.nseg;
    // ---- each segment's affine state map: S_loc (and the outputs o_loc) from S = 0,
    //      Phi (and q~_t = Phi_t^T q_t) from S = I with zero values; the last
    //      segment's pass from S = 0 also gives the final variances
    P.S0 = nullptr;
    P.last_only = 0;
    P.S_T = sp.S_loc;
    P.p_T = a.p_T;
    if ((e = run()) != cudaSuccess) return e;
    P.s0_identity = 1;
    P.no_v = 1;
    P.S_T = sp.Phi;
    P.p_T = nullptr;
    P.o = static_cast<__nv_bfloat16*>(sp.qt);
    if ((e = run()) != cudaSuccess) return e;
    // ---- chained initial states and the final state, then o += S_in^T q~
    if ((e = launch_segment_states(a, sp, s)) != cudaSuccess) return e;
    return launch_segment_correction(a, sp, s);
}

}  // namespace kdn
