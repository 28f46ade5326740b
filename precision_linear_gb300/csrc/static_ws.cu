// pl_nvfp4_lora_linear_static_ws: the linear with its scratch in a device array
// owned by this library, for callers that cannot allocate device memory.
//
// The scratch is one file-scope __device__ array of PL_STATIC_WORKSPACE_BYTES.  Every
// device that loads the library holds it until the process exits.  Host code never
// passes the array's name to a kernel -- on the host that name is only a stand-in
// symbol -- but the device address that cudaGetSymbolAddress returns for the current
// device.  That lookup is made on every call (it is cheap once the module is loaded), so
// an address never outlives a device reset or a context torn down and created again.
#include "../../include/precision_linear.h"
#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[PL_STATIC_WORKSPACE_BYTES];

// Device address of the scratch array on the current device.
pl_status static_ws_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);
  if (e != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return PL_ERR_CUDA;
  }
  *out = p;
  return PL_OK;
}

}  // namespace

extern "C" pl_status pl_nvfp4_lora_linear_static_ws(
    const void* x, int64_t M, int64_t d_i, int64_t d_o, const uint8_t* codes, const uint8_t* scales,
    const float* s_g, const void* A, const void* B, int r, float lambda, const float* w_norm, const float* z,
    float eps, void* y, int y_dtype, pl_stream_t stream) {
  const size_t need = pl_workspace_bytes(M, d_i, d_o, r);
  if (need > static_cast<size_t>(PL_STATIC_WORKSPACE_BYTES)) return PL_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need != 0) {  // need == 0: invalid shape, reported by the call below
    // on a device this library does not support the symbol has no image: report that
    // device as unsupported, as the workspace entry point does
    if (!pl::device_supported()) return PL_ERR_DEVICE;
    const pl_status st = static_ws_address(&ws);
    if (st != PL_OK) return st;
  }
  // Nothing in the scratch has to start at zero: the kernels write every byte of it
  // that they later read, within the same call.
  return pl_nvfp4_lora_linear(x, M, d_i, d_o, codes, scales, s_g, A, B, r, lambda, w_norm, z, 0, eps, y, y_dtype,
                              ws, static_cast<size_t>(PL_STATIC_WORKSPACE_BYTES), stream);
}
