// Fused tensor-core forward (sm_103a): not built yet; the CUDA-core path runs.
#include "kdn_internal.h"

namespace kdn {

bool tc_path_supported(int, int, int, int) { return false; }

cudaError_t launch_forward_tc(const ForwardArgs&, cudaStream_t) { return cudaErrorNotSupported; }

int tc_kernel_count() { return 1; }

}  // namespace kdn
