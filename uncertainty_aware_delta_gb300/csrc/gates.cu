// Gate prologue of the KDN layer (log alpha, omega and r from the layer's gate
// pre-activations, for the forward paths), and the effective write strength from
// the gain scan's gains.
//
// KDN reading notes Sec. 5.1: the end-to-end network produces alpha_t =
// sigma(a_t), omega_t = softplus(w_t) (one scalar per token-head for Isotropic
// KDN) and r_t = r_min + softplus(rho_t) from the projections a, w, rho of the
// layer input.  The mixer consumes log alpha = log sigma(a) = -softplus(-a).
// Both branches are evaluated with the exponential's argument kept non-positive:
//   log sigma(x) = min(x, 0) - log1p(e^{-|x|}),   softplus(x) = max(x, 0) + log1p(e^{-|x|}).
// bf16 logits (the tensor-core path): 16-byte loads of eight logits, the hardware
// exponential and logarithm, and log1p(u) for u < 1/16 from its Taylor series
// u - u^2/2 + u^3/3 - u^4/4 (remainder below u^5/5 < 1e-6 u); fp32 logits use the
// accurate expf / log1pf.  Evaluating the branches here, over every SM, keeps their
// transcendental work off the forward kernels' serial gain pass.
//
// Effective write strength (reading notes Sec. 3.2; the paper's App. B, Eq. 58-61):
// beta_eff_t = k_t^T kappa_t, one warp per token-head.

#include "common.cuh"
#include "kdn_internal.h"

namespace kdn {
namespace {

__device__ __forceinline__ float log_sigmoid(float x) { return fminf(x, 0.0f) - log1pf(expf(-fabsf(x))); }
__device__ __forceinline__ float softplus(float x) { return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x))); }

// log(1 + e^{-|x|}) with the hardware exponential and logarithm (bf16 logits)
__device__ __forceinline__ float log1p_exp_neg_abs(float x) {
    const float u = __expf(-fabsf(x));
    return u < 0.0625f ? u * (1.0f - u * (0.5f - u * (0.33333334f - 0.25f * u))) : __logf(1.0f + u);
}

// Eight bf16 logits per step: a grid-stride walk over the 8-element groups of log
// alpha, then omega, then r (mode 0: log sigma, 1: softplus, 2: r_min + softplus);
// the groups that do not fill eight elements (omega and r with B*T*H % 8 != 0) are
// taken one element per thread at the end.
__global__ void gate_expand_bf16_kernel(const __nv_bfloat16* __restrict__ al, const __nv_bfloat16* __restrict__ wl,
                                        const __nv_bfloat16* __restrict__ rl, float r_min, size_t n_la, size_t n_om,
                                        size_t n_r, float* __restrict__ la, float* __restrict__ om,
                                        float* __restrict__ r) {
    const size_t g_la = n_la / 8, g_om = n_om / 8, g_r = n_r / 8, ng = g_la + g_om + g_r;
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x, stride = (size_t)gridDim.x * blockDim.x;
    for (size_t e = tid; e < ng; e += stride) {
        const __nv_bfloat16* src;
        float* dst;
        size_t j;
        int mode;
        if (e < g_la) {
            src = al; dst = la; j = e; mode = 0;
        } else if (e < g_la + g_om) {
            src = wl; dst = om; j = e - g_la; mode = 1;
        } else {
            src = rl; dst = r; j = e - g_la - g_om; mode = 2;
        }
        const uint4 raw = *reinterpret_cast<const uint4*>(src + 8 * j);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        float y[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float x0 = __uint_as_float(w[q] << 16), x1 = __uint_as_float(w[q] & 0xffff0000u);
            const float l0 = log1p_exp_neg_abs(x0), l1 = log1p_exp_neg_abs(x1);
            if (mode == 0) {
                y[2 * q] = fminf(x0, 0.0f) - l0;
                y[2 * q + 1] = fminf(x1, 0.0f) - l1;
            } else {
                const float c = mode == 2 ? r_min : 0.0f;
                y[2 * q] = c + fmaxf(x0, 0.0f) + l0;
                y[2 * q + 1] = c + fmaxf(x1, 0.0f) + l1;
            }
        }
        float4* d4 = reinterpret_cast<float4*>(dst + 8 * j);
        d4[0] = make_float4(y[0], y[1], y[2], y[3]);
        d4[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
    if (tid < n_om - 8 * g_om) {
        const size_t j = 8 * g_om + tid;
        const float x = __bfloat162float(wl[j]);
        om[j] = fmaxf(x, 0.0f) + log1p_exp_neg_abs(x);
    }
    if (tid < n_r - 8 * g_r) {
        const size_t j = 8 * g_r + tid;
        const float x = __bfloat162float(rl[j]);
        r[j] = r_min + fmaxf(x, 0.0f) + log1p_exp_neg_abs(x);
    }
}

// One grid-stride pass over the three tensors (n_la = B*T*H*dk elements of log alpha,
// n_om of omega, n_r of r; the index ranges are walked one after the other).
template <typename TIO>
__global__ void gate_expand_kernel(const TIO* __restrict__ al, const TIO* __restrict__ wl,
                                   const TIO* __restrict__ rl, float r_min, size_t n_la, size_t n_om,
                                   size_t n_r, float* __restrict__ la, float* __restrict__ om,
                                   float* __restrict__ r) {
    const size_t n = n_la + n_om + n_r;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
        if (e < n_la) {
            la[e] = log_sigmoid(IO<TIO>::load(al, e));
        } else if (e < n_la + n_om) {
            const size_t j = e - n_la;
            om[j] = softplus(IO<TIO>::load(wl, j));
        } else {
            const size_t j = e - n_la - n_om;
            r[j] = r_min + softplus(IO<TIO>::load(rl, j));
        }
    }
}

template <typename TIO>
__global__ void beta_from_kappa_kernel(const TIO* __restrict__ k, const float* __restrict__ kappa, size_t ntok,
                                       int dk, float* __restrict__ beta) {
    const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
    const int lane = threadIdx.x & 31;
    for (size_t th = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); th < ntok; th += warps) {
        float acc = 0.0f;
        for (int i = lane; i < dk; i += 32) acc = fmaf(IO<TIO>::load(k, th * dk + i), kappa[th * dk + i], acc);
        acc = warp_sum(acc);
        if (lane == 0) beta[th] = acc;
    }
}

int grid_for(size_t work, int per_block) {
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess) {
        (void)cudaGetLastError();
        sms = 152;
    }
    const size_t want = (work + per_block - 1) / per_block;
    const size_t cap = (size_t)sms * 8;   // grid-stride beyond eight blocks per SM
    return (int)(want < cap ? (want > 0 ? want : 1) : cap);
}

}  // namespace

cudaError_t launch_gate_expand(int variant, int B, int T, int H, int dk, int io, float r_min,
                               const void* alpha_logit, const void* omega_logit, const void* r_logit,
                               float* log_alpha, float* omega, float* r, cudaStream_t s) {
    const size_t ntok = (size_t)B * T * H, n_la = ntok * dk, n_om = variant == 1 ? ntok : ntok * dk;
    const size_t n = n_la + n_om + ntok;
    if (n == 0) return cudaSuccess;
    if (io == 1) {
        const int grid = grid_for(n / 8 + 8, 256);   // (at least one block for the tails)
        gate_expand_bf16_kernel<<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(alpha_logit), static_cast<const __nv_bfloat16*>(omega_logit),
            static_cast<const __nv_bfloat16*>(r_logit), r_min, n_la, n_om, ntok, log_alpha, omega, r);
    } else {
        gate_expand_kernel<float><<<grid_for(n, 256), 256, 0, s>>>(
            static_cast<const float*>(alpha_logit), static_cast<const float*>(omega_logit),
            static_cast<const float*>(r_logit), r_min, n_la, n_om, ntok, log_alpha, omega, r);
    }
    return cudaGetLastError();
}

cudaError_t launch_beta_from_kappa(int B, int T, int H, int dk, int io, const void* k, const float* kappa,
                                   float* beta_eff, cudaStream_t s) {
    const size_t ntok = (size_t)B * T * H;
    if (ntok == 0) return cudaSuccess;
    const int grid = grid_for(ntok, 8);   // 8 warps (token-heads) per block
    if (io == 1)
        beta_from_kappa_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(k), kappa,
                                                                   ntok, dk, beta_eff);
    else
        beta_from_kappa_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(k), kappa, ntok, dk, beta_eff);
    return cudaGetLastError();
}

}  // namespace kdn
