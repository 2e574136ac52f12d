// dcn_noalloc.cu -- dcn_core_bwd_noalloc: the backward with its float32
// grad_input accumulator in a static device array of this library instead of
// a caller-provided workspace, for callers that cannot allocate device memory
// (see include/dcn_core.h).
#include <mutex>

#include "../../include/dcn_core.h"
#include <cuda_runtime.h>

namespace {

// The scratch array.  In host code this name is only a host-side handle: its
// device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char dcn_scratch[DCN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_lock;
void* g_address[kMaxDevices];  // device address of dcn_scratch, per device ordinal

// Device address of the scratch array on the current device, looked up on
// the first call for that device and remembered.
int scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return DCN_ERR_CUDA;
  if (dev >= kMaxDevices) return DCN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> hold(g_lock);
  if (g_address[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, dcn_scratch) != cudaSuccess || ptr == nullptr)
      return DCN_ERR_CUDA;
    g_address[dev] = ptr;
  }
  *out = g_address[dev];
  return DCN_OK;
}

}  // namespace

extern "C" int dcn_core_bwd_noalloc(const dcn_params_t* p, const void* grad_out,
                                    const void* input, const void* offset, const void* mask,
                                    void* grad_input, void* grad_offset, void* grad_mask,
                                    void* stream) {
  int H_out = 0, W_out = 0;
  const int rc = dcn_out_shape(p, &H_out, &W_out);  // every parameter check, host only
  if (rc != DCN_OK) return rc;
  const size_t need = dcn_core_bwd_workspace(p);
  if (need > DCN_NOALLOC_SCRATCH_BYTES) return DCN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (need > 0) {
    const int src = scratch_on_current_device(&scratch);
    if (src != DCN_OK) return src;
  }
  // dcn_core_bwd clears the accumulator (cudaMemsetAsync) before using it.
  return dcn_core_bwd(p, grad_out, input, offset, mask, grad_input, grad_offset, grad_mask,
                      scratch, need, stream);
}
