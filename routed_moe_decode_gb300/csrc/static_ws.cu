// Whole-layer entry point whose scratch lives in a fixed device array of this library,
// for callers that cannot allocate device memory themselves (see moe.h,
// moe_layer_static_workspace).
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "moe_kernels.cuh"

// The scratch: one fixed array per device that loads the library, held until exit.
constexpr size_t kStaticWorkspaceBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

namespace {

constexpr int kMaxDevices = 64;
void* g_static_ptr[kMaxDevices] = {};
std::mutex g_static_mutex;

// Device address of the array on the current device, looked up once per device.  In host
// code `g_static_workspace` only names a host-side stand-in; kernels must be given this
// address instead.  The cached address belongs to the device's primary context as the
// first call found it: a process that resets the device (cudaDeviceReset) or drives it
// through another context must not use this entry point afterwards.
int static_workspace_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    moe::set_last_error_message("moe_layer_static_workspace: cudaGetDevice failed");
    return MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    moe::set_last_error_message("moe_layer_static_workspace: device ordinal beyond the library's table of 64");
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || !p) {
      moe::set_last_error_message("moe_layer_static_workspace: cudaGetSymbolAddress failed");
      return MOE_ERR_CUDA;
    }
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_layer_static_workspace(const moe_shape* shape, const float* logits, const void* hidden,
                               const uint8_t* w13_codes, const uint8_t* w13_scales, float w13_scale,
                               const uint8_t* w2_codes, const uint8_t* w2_scales, float w2_scale,
                               const void* residual, void* out, int32_t* ids, float* weights,
                               moe_stream_t stream) {
  const int rc = moe_check_shape(shape);
  if (rc != MOE_OK) return rc;
  const size_t need = moe_workspace_bytes(shape);
  if (need > kStaticWorkspaceBytes) {
    char msg[160];
    snprintf(msg, sizeof msg, "moe_layer_static_workspace: this shape needs %zu bytes of scratch, more than the %zu-byte static array",
             need, kStaticWorkspaceBytes);
    moe::set_last_error_message(msg);
    return MOE_ERR_WORKSPACE;
  }
  if (shape->T == 0) return MOE_OK;
  void* ws = nullptr;
  const int arc = static_workspace_address(&ws);
  if (arc != MOE_OK) return arc;
  // the status block and the decode kernel's counter sets must start at zero; every other
  // field is rewritten by the call
  if (cudaMemsetAsync(ws, 0, std::min(need, moe::kZeroedPrefix), stream) != cudaSuccess) {
    moe::set_last_error_message("moe_layer_static_workspace: clearing the status block failed");
    return MOE_ERR_CUDA;
  }
  return moe_layer(shape, logits, hidden, w13_codes, w13_scales, w13_scale, w2_codes, w2_scales, w2_scale,
                   residual, out, ids, weights, ws, need, stream);
}

int moe_static_workspace_read_status(int clear, uint32_t* status_bits, moe_stream_t stream) {
  if (!status_bits) return MOE_ERR_INVALID_ARG;
  void* ws = nullptr;
  const int arc = static_workspace_address(&ws);
  if (arc != MOE_OK) return arc;
  return moe_read_device_status(ws, clear, status_bits, stream);
}

}  // extern "C"
