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
// of S in shared memory in fp32.  The triangular system is solved by forward
// substitution.

#include "common.cuh"
#include "kdn_internal.h"

namespace kdn {
namespace {

constexpr int kNT = 256;

template <typename TIO>
__global__ void __launch_bounds__(kNT)
chunk_simt_kernel(const TIO* __restrict__ q, const TIO* __restrict__ k, const TIO* __restrict__ v,
                  const float* __restrict__ la, const float* __restrict__ kappa,
                  const float* __restrict__ S0, TIO* __restrict__ o, float* __restrict__ S_T,
                  int Tn, int H, int DK, int dv, int C, int VS, uint32_t* status) {
    const int LD = DK + 1, LS = VS + 1, LC = C + 1;
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
        // 1. cumulative log-decay per channel
        if (tid < DK) {
            float g = 0.f;
            for (int t = 0; t < C; ++t) {
                if (t < nv) g += la[(((size_t)b * Tn + t0 + t) * H + h) * DK + tid];
                Kt[t * LD + tid] = g;
            }
            const float gr = 0.5f * g;
            gref[tid] = gr;
            gin[tid] = expf(gr);
            gout[tid] = expf(g - gr);
            if (!(fabsf(g) <= kMaxChunkLogDecay)) set_status(status, kStatusRange);
        }
        __syncthreads();
        // 2. decayed operands; state into the chunk's reference frame
        for (int e = tid; e < C * DK; e += kNT) {
            const int t = e / DK, i = e % DK;
            if (t < nv) {
                const size_t gi = (((size_t)b * Tn + t0 + t) * H + h) * DK + i;
                const float g = Kt[t * LD + i];
                const float ef = expf(g - gref[i]);
                const float eb = expf(gref[i] - g);
                Kb[t * LD + i] = IO<TIO>::load(k, gi) * ef;
                Qb[t * LD + i] = IO<TIO>::load(q, gi) * ef;
                Kt[t * LD + i] = kappa[gi] * eb;
            } else {
                Kb[t * LD + i] = 0.f;
                Qb[t * LD + i] = 0.f;
                Kt[t * LD + i] = 0.f;
            }
        }
        for (int e = tid; e < DK * VS; e += kNT) {
            const int i = e / VS, j = e % VS;
            S[i * LS + j] *= gin[i];
        }
        __syncthreads();
        // 3. Gram matrices (lower triangles) and 4. state products
        for (int e = tid; e < C * C; e += kNT) {
            const int t = e / C, s = e % C;
            float l = 0.f, aq = 0.f;
            if (s <= t) {
                for (int i = 0; i < DK; ++i) {
                    const float kt = Kt[s * LD + i];
                    l = fmaf(Kb[t * LD + i], kt, l);
                    aq = fmaf(Qb[t * LD + i], kt, aq);
                }
            }
            L[t * LC + s] = (s < t) ? l : 0.f;
            A[t * LC + s] = (s <= t) ? aq : 0.f;
        }
        for (int e = tid; e < C * VS; e += kNT) {
            const int t = e / VS, j = e % VS;
            float x = 0.f, oo = 0.f;
            for (int i = 0; i < DK; ++i) {
                const float sv = S[i * LS + j];
                x = fmaf(Kb[t * LD + i], sv, x);
                oo = fmaf(Qb[t * LD + i], sv, oo);
            }
            const float vv = (t < nv)
                ? IO<TIO>::load(v, (((size_t)b * Tn + t0 + t) * H + h) * dv + j0 + j) : 0.f;
            X[t * LS + j] = vv - x;
            O[t * LS + j] = oo;
        }
        __syncthreads();
        // 5. forward substitution (I + L) Delta = X, one row at a time;
        //    8 threads share a column's sum over earlier rows.
        {
            const int j = tid >> 3, g8 = tid & 7;
            for (int t = 1; t < nv; ++t) {
                float part = 0.f;
                if (j < VS)
                    for (int s = g8; s < t; s += 8) part = fmaf(L[t * LC + s], X[s * LS + j], part);
                part += __shfl_xor_sync(0xffffffffu, part, 4);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                if (j < VS && g8 == 0) X[t * LS + j] -= part;
                __syncthreads();
            }
        }
        // 6. output rows and 7. state update
        for (int e = tid; e < C * VS; e += kNT) {
            const int t = e / VS, j = e % VS;
            if (t < nv) {
                float acc = O[t * LS + j];
                for (int s = 0; s <= t; ++s) acc = fmaf(A[t * LC + s], X[s * LS + j], acc);
                IO<TIO>::store(o, (((size_t)b * Tn + t0 + t) * H + h) * dv + j0 + j, acc);
            }
        }
        for (int e = tid; e < DK * VS; e += kNT) {
            const int i = e / VS, j = e % VS;
            float acc = S[i * LS + j];
            for (int s = 0; s < nv; ++s) acc = fmaf(Kt[s * LD + i], X[s * LS + j], acc);
            S[i * LS + j] = acc * gout[i];
        }
        __syncthreads();
    }
    for (int e = tid; e < DK * VS; e += kNT) {
        const int i = e / VS, j = e % VS;
        S_T[((size_t)bh * DK + i) * dv + j0 + j] = S[i * LS + j];
    }
}

size_t simt_smem_bytes(int DK, int C, int VS) {
    const size_t LD = DK + 1, LS = VS + 1, LC = C + 1;
    return sizeof(float) * (3 * C * LD + DK * LS + 2 * C * LC + 2 * C * LS + 3 * DK);
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
