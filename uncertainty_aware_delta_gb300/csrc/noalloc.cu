// kdn_forward_noalloc: the forward mixer for callers that cannot allocate
// device memory when they run it.  The scratch the forward needs lives in a
// library-owned static device array instead of a caller workspace.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kdn.h"

namespace {

// One array per GPU that loads the library, held until the process exits.
__device__ __align__(256) unsigned char g_kdn_static_scratch[KDN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices];  // device address of the array, per device, once looked up

// In host code `g_kdn_static_scratch` names a host-side stand-in, not device
// memory, so kernels must be given the address the runtime reports for the
// current device.  Looked up once per device, with that device current.
kdn_status scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kdn_static_scratch) != cudaSuccess || p == nullptr)
            return KDN_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KDN_OK;
}

}  // namespace

extern "C" kdn_status kdn_forward_noalloc(int variant, int B, int T, int H, int dk, int dv,
                                          int chunk, float mu, int io_dtype, uint32_t flags,
                                          const void* q, const void* k, const void* v,
                                          const float* log_alpha, const float* omega,
                                          const float* r, const float* S0, const float* p0,
                                          void* o, float* S_T, float* p_T, uint32_t* status_out,
                                          kdn_stream_t stream) {
    if (variant != KDN_DIAG && variant != KDN_ISO) return KDN_ERR_SHAPE;
    auto forward = variant == KDN_DIAG ? kdn_diag_forward : kdn_iso_forward;
    const size_t need = kdn_workspace_size(variant, B, T, H, dk, dv, chunk, io_dtype, flags);
    if (need == 0)  // rejected sizes: let the regular entry point name the reason
        return forward(B, T, H, dk, dv, chunk, mu, io_dtype, flags, q, k, v, log_alpha, omega, r,
                       S0, p0, o, S_T, p_T, nullptr, 0, stream);
    if (need > (size_t)KDN_STATIC_SCRATCH_BYTES) return KDN_ERR_WORKSPACE;
    if (status_out && (reinterpret_cast<uintptr_t>(status_out) & 3u)) return KDN_ERR_ALIGN;
    void* scratch = nullptr;
    kdn_status st = scratch_for_current_device(&scratch);
    if (st != KDN_OK) return st;
    // The regular forward zeroes the status word at the start of the scratch;
    // everything else it reads from the scratch it writes first in the same call.
    st = forward(B, T, H, dk, dv, chunk, mu, io_dtype, flags, q, k, v, log_alpha, omega, r, S0, p0,
                 o, S_T, p_T, scratch, (size_t)KDN_STATIC_SCRATCH_BYTES, stream);
    if (st != KDN_OK || status_out == nullptr) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(status_out, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess)
        return KDN_ERR_CUDA;
    return KDN_OK;
}
