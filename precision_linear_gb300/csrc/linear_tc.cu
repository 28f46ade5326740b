// tcgen05 tensor-core NVFP4 + LoRA linear (placeholder: not yet enabled).
#include "common.cuh"

namespace pl {
bool tc_supported(int64_t, int64_t, int64_t, int) { return false; }
size_t tc_workspace_bytes(int64_t, int64_t, int64_t, int) { return 0; }
cudaError_t launch_linear_tc(const LinearArgs&, cudaStream_t) { return cudaErrorNotSupported; }
uint32_t tc_read_and_clear_status() { return 0; }
}  // namespace pl
