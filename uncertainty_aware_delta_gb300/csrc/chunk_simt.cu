// Chunkwise memory pass on CUDA cores (fp32 FFMA).
//
// With the gains kappa_t known (from the gain scan), the memory follows the
// affine recurrence of the KDN paper Eq. 38-39,
//     S_t = diag(a_t) S_{t-1} + kappa_t (v_t - (diag(a_t) S_{t-1})^T k_t)^T,
// read out as o_t = S_t^T q_t after the write.  Inside a chunk of C tokens,
// with G_t the cumulative log-decay since the chunk start (per channel) and a
// per-channel reference G_ref = G_C / 2 (half the chunk total, which bounds
// every exponential factor by exp(|G_C| / 2)), the recurrence unrolls to
//     K_bar_t = k_t * exp(G_t - G_ref),   Q_bar_t = q_t * exp(G_t - G_ref),
//     K_til_s = kappa_s * exp(G_ref - G_s),
//     S_m     = diag(exp(G_ref)) S_in,
//     (I + L) Delta = V - K_bar S_m,      L = strict_lower(K_bar K_til^T),
//     O       = Q_bar S_m + lower_incl_diag(Q_bar K_til^T) Delta,
//     S_out   = diag(exp(G_C - G_ref)) (S_m + K_til^T Delta),
// the compact-WY / UT chunk form of the paper's App. D with the decay ratios
// taken from differences of cumulative log-decay, and the query-write matrix
// keeping its diagonal so each token reads its own write.  Delta holds the
// innovations v_t - S_hat_t^T k_t.  (The no-decay form of the same algebra is
// printed by Preconditioned DeltaNet, Eq. 6 / App. F.2.1.)
//
// One CTA owns one (b, h) and one slice of VS value columns (the columns are
// independent given kappa) and walks the chunks in order, keeping its slice
// of S in shared memory in fp32.  The products (Gram matrices, the state's
// predictions and reads, the output and state updates) run as warp-level
// m16n8k8 TF32 tensor-core MMAs in the 3xTF32 split, which keeps fp32-level
// accuracy.  The triangular system is solved blockwise: each 16-row diagonal
// block by substitution (a thread per value column, in registers), then the rows
// below it updated by one product.

#include "common.cuh"
#include "kdn_internal.h"
#include "mma_tf32x3.cuh"

namespace kdn {
namespace {

constexpr int kNT = 256;
constexpr int kPadW = 4;   // row padding (words) of the d-wide and VS-wide tiles
constexpr int kSB = 16;    // rows of a diagonal block of the triangular solve

template <typename TIO>
__global__ void __launch_bounds__(kNT, 1)
chunk_simt_kernel(const TIO* __restrict__ q, const TIO* __restrict__ k, const TIO* __restrict__ v,
                  const float* __restrict__ la, const float* __restrict__ kappa,
                  const float* __restrict__ S0, TIO* __restrict__ o, float* __restrict__ S_T,
                  int Tn, int H, int DK, int dv, int C, int VS, uint32_t* status) {
    const int LD = DK + kPadW, LS = VS + kPadW, LC = C + 1;
    extern __shared__ float sm[];
    float* Kb = sm;                 // [C][LD]
    float* Qb = Kb + C * LD;        // [C][LD]
    float* Kt = Qb + C * LD;        // [C][LD]  (cumulative log-decay G first)
    float* S = Kt + C * LD;         // [DK][LS]
    float* L = S + DK * LS;         // [C][LC]
    float* A = L + C * LC;          // [C][LC]
    float* X = A + C * LC;          // [C][LS]  V - K_bar S_m, then Delta
    float* O = X + C * LS;          // [C][LS]
    float* gref = O + C * LS;       // [DK]
    float* gin = gref + DK;         // [DK] exp(G_ref)
    float* gout = gin + DK;         // [DK] exp(G_C - G_ref)
    float* G = gout + DK;           // [C][DK] log_alpha, then the cumulative log-decay
    // (every region starts on a 16-byte boundary: all sizes above are multiples of 4 words)

    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int j0 = blockIdx.y * VS;
    const int tid = threadIdx.x;

    for (int e = tid; e < DK * VS; e += kNT) {
        const int i = e / VS, j = e % VS;
        S[i * LS + j] = S0 ? S0[((size_t)bh * DK + i) * dv + j0 + j] : 0.f;
    }

    const int nchunks = (Tn + C - 1) / C;
    for (int n = 0; n < nchunks; ++n) {
        const int t0 = n * C, nv = min(C, Tn - t0);
        // 1. the chunk's inputs: log_alpha, kappa and, for fp32 inputs, k, q, v by 16-byte
        //    async copies (rows past the sequence end zero-filled); bf16 k, q, v through
        //    loads unrolled by eight
        const size_t tok0 = ((size_t)b * Tn + t0) * H + h;   // token-head index of the chunk's first token
        for (int e4 = tid; e4 < C * DK / 4; e4 += kNT) {
            const int t = (4 * e4) / DK, i = (4 * e4) % DK;
            const size_t gi = (tok0 + (size_t)min(t, nv - 1) * H) * DK + i;
            cp_async16(G + t * DK + i, la + gi, t < nv);
            cp_async16(Kt + t * LD + i, kappa + gi, t < nv);
            if constexpr (sizeof(TIO) == 4) {
                cp_async16(Kb + t * LD + i, k + gi, t < nv);
                cp_async16(Qb + t * LD + i, q + gi, t < nv);
            }
        }
        if constexpr (sizeof(TIO) == 4) {
            for (int e4 = tid; e4 < C * VS / 4; e4 += kNT) {
                const int t = (4 * e4) / VS, j = (4 * e4) % VS;
                cp_async16(X + t * LS + j, v + (tok0 + (size_t)min(t, nv - 1) * H) * dv + j0 + j, t < nv);
            }
        } else {
#pragma unroll 8
            for (int e = tid; e < C * DK; e += kNT) {
                const int t = e / DK, i = e % DK;
                const size_t gi = (tok0 + (size_t)t * H) * DK + i;
                Kb[t * LD + i] = t < nv ? IO<TIO>::load(k, gi) : 0.f;
                Qb[t * LD + i] = t < nv ? IO<TIO>::load(q, gi) : 0.f;
            }
#pragma unroll 8
            for (int e = tid; e < C * VS; e += kNT) {
                const int t = e / VS, j = e % VS;
                X[t * LS + j] = t < nv ? IO<TIO>::load(v, (tok0 + (size_t)t * H) * dv + j0 + j) : 0.f;
            }
        }
        cp_async_wait_all();
        __syncthreads();
        // cumulative log-decay per channel, its reference and factors
        if (tid < DK) {
            float g = 0.f;
            for (int t = 0; t < C; ++t) {
                g += G[t * DK + tid];
                G[t * DK + tid] = g;
            }
            const float gr = 0.5f * g;
            gref[tid] = gr;
            gin[tid] = expf(gr);
            gout[tid] = expf(g - gr);
            if (!(fabsf(g) <= kMaxChunkLogDecay)) set_status(status, kStatusRange);
        }
        __syncthreads();
        // 2. decayed operands (in place); state into the chunk's reference frame
        for (int e = tid; e < C * DK; e += kNT) {
            const int t = e / DK, i = e % DK;
            const float g = G[t * DK + i];
            Kb[t * LD + i] *= expf(g - gref[i]);
            Qb[t * LD + i] *= expf(g - gref[i]);
            Kt[t * LD + i] *= expf(gref[i] - g);
        }
        for (int e = tid; e < DK * VS; e += kNT) {
            const int i = e / VS, j = e % VS;
            S[i * LS + j] *= gin[i];
        }
        __syncthreads();
        // 3. Gram matrices L = K_bar K_til^T, A = Q_bar K_til^T (triangles taken below) and
        // 4. state products X = V - K_bar S_m, O = Q_bar S_m
        smem_gemm<2>(C, C, DK, Kb, LD, 1, Kt, 1, LD, L, LC, 1.f, false);
        smem_gemm<2>(C, C, DK, Qb, LD, 1, Kt, 1, LD, A, LC, 1.f, false);
        smem_gemm<2>(C, VS, DK, Kb, LD, 1, S, LS, 1, X, LS, -1.f, true);
        smem_gemm<2>(C, VS, DK, Qb, LD, 1, S, LS, 1, O, LS, 1.f, false);
        __syncthreads();
        for (int e = tid; e < C * C; e += kNT) {
            const int t = e / C, s = e % C;
            if (s >= t) L[t * LC + s] = 0.f;
            if (s > t) A[t * LC + s] = 0.f;
        }
        __syncthreads();
        // 5. forward substitution (I + L) Delta = X, blockwise: each 16-row diagonal block
        //    by substitution (a thread per value column, in registers), then the rows
        //    below it updated by one product
        for (int r0 = 0; r0 < C; r0 += kSB) {
            for (int j = tid; j < VS; j += kNT) {
                float x[kSB];
#pragma unroll
                for (int t = 0; t < kSB; ++t) x[t] = X[(r0 + t) * LS + j];
#pragma unroll
                for (int t = 1; t < kSB; ++t)
#pragma unroll
                    for (int s2 = 0; s2 < t; ++s2) x[t] = fmaf(-L[(r0 + t) * LC + r0 + s2], x[s2], x[t]);
#pragma unroll
                for (int t = 0; t < kSB; ++t) X[(r0 + t) * LS + j] = x[t];
            }
            __syncthreads();
            if (r0 + kSB < C) {
                smem_gemm<2>(C - r0 - kSB, VS, kSB, L + (r0 + kSB) * LC + r0, LC, 1, X + r0 * LS, LS, 1,
                             X + (r0 + kSB) * LS, LS, -1.f, true);
                __syncthreads();
            }
        }
        // 6. output rows O += A Delta and 7. state update S = diag(g_out) (S_m + K_til^T Delta)
        smem_gemm<2>(C, VS, C, A, LC, 1, X, LS, 1, O, LS, 1.f, true);
        smem_gemm<2>(DK, VS, C, Kt, 1, LD, X, LS, 1, S, LS, 1.f, true);
        __syncthreads();
        for (int e = tid; e < C * VS; e += kNT) {
            const int t = e / VS, j = e % VS;
            if (t < nv) IO<TIO>::store(o, (((size_t)b * Tn + t0 + t) * H + h) * dv + j0 + j, O[t * LS + j]);
        }
        for (int e = tid; e < DK * VS; e += kNT) {
            const int i = e / VS, j = e % VS;
            S[i * LS + j] *= gout[i];
        }
        __syncthreads();
    }
    for (int e = tid; e < DK * VS; e += kNT) {
        const int i = e / VS, j = e % VS;
        S_T[((size_t)bh * DK + i) * dv + j0 + j] = S[i * LS + j];
    }
}

size_t simt_smem_bytes(int DK, int C, int VS) {
    const size_t LD = DK + kPadW, LS = VS + kPadW, LC = C + 1;
    return sizeof(float) * (3 * C * LD + DK * LS + 2 * C * LC + 2 * C * LS + 3 * DK + C * DK);
}

template <typename TIO>
cudaError_t launch_chunk_t(const ForwardArgs& a, const float* kappa, cudaStream_t s) {
    const int VS = a.dv < 32 ? a.dv : 32;
    const size_t smem = simt_smem_bytes(a.dk, a.chunk, VS);
    cudaError_t e = cudaFuncSetAttribute(chunk_simt_kernel<TIO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(a.B * a.H, a.dv / VS);
    chunk_simt_kernel<TIO><<<grid, kNT, smem, s>>>(
        static_cast<const TIO*>(a.q), static_cast<const TIO*>(a.k), static_cast<const TIO*>(a.v),
        a.log_alpha, kappa, a.S0, static_cast<TIO*>(a.o), a.S_T, a.T, a.H, a.dk, a.dv, a.chunk, VS,
        a.status);
    return cudaGetLastError();
}

__global__ void state_copy_kernel(const float* __restrict__ S0, const float* __restrict__ p0,
                                  float* __restrict__ S_T, float* __restrict__ p_T, size_t nS,
                                  size_t np, float p_default) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < nS; e += stride)
        S_T[e] = S0 ? S0[e] : 0.f;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < np; e += stride)
        p_T[e] = p0 ? p0[e] : p_default;
}

}  // namespace

cudaError_t launch_chunk_simt(const ForwardArgs& a, const float* kappa, cudaStream_t s) {
    if (a.io == 1) return launch_chunk_t<__nv_bfloat16>(a, kappa, s);
    return launch_chunk_t<float>(a, kappa, s);
}

cudaError_t launch_state_copy(const ForwardArgs& a, cudaStream_t s) {
    const size_t nS = (size_t)a.B * a.H * a.dk * a.dv;
    // per-channel state for the diagonal variant and PKDA, one scalar for isotropic;
    // defaults: variance 1 (KDN), key statistic 0 (PKDA)
    const size_t np = (size_t)a.B * a.H * (a.variant == 1 ? 1 : a.dk);
    if (nS == 0) return cudaSuccess;
    int blocks = (int)((nS + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    state_copy_kernel<<<blocks, 256, 0, s>>>(a.S0, a.p0, a.S_T, a.p_T, nS, np, a.variant == 2 ? 0.f : 1.f);
    return cudaGetLastError();
}

}  // namespace kdn
