// Device helpers shared by the KDN kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kdn {

// Device status codes (same values as kdn_status in include/kdn.h).
constexpr uint32_t kStatusTimeout = 8u;
constexpr uint32_t kStatusRange = 9u;

// A chunk whose per-channel cumulative log-decay magnitude exceeds this is
// reported as out of range: the factored decay exp(G_t - G_ref) * exp(G_ref - G_s)
// uses the chunk's half-way reference, so each factor stays below exp(kMaxChunkLogDecay / 2)
// = exp(80) ~ 5.5e34, inside the fp32 and bf16 exponent range.
constexpr float kMaxChunkLogDecay = 160.0f;

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t code) {
    if (status) atomicCAS(status, 0u, code);  // the first condition seen wins
}

template <typename T> struct IO;
template <> struct IO<float> {
    __device__ __forceinline__ static float load(const float* p, size_t i) { return p[i]; }
    __device__ __forceinline__ static void store(float* p, size_t i, float x) { p[i] = x; }
};
template <> struct IO<__nv_bfloat16> {
    __device__ __forceinline__ static float load(const __nv_bfloat16* p, size_t i) {
        return __bfloat162float(p[i]);
    }
    __device__ __forceinline__ static void store(__nv_bfloat16* p, size_t i, float x) {
        p[i] = __float2bfloat16_rn(x);
    }
};

// Sum over a warp (all 32 lanes participate).
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

}  // namespace kdn
