// moe_nvfp4_layer_static: the whole layer step for callers that cannot
// allocate device memory. Its workspace is a file-scope device array of
// MOE_NVFP4_STATIC_SCRATCH_BYTES; the step itself is moe_nvfp4_layer,
// unchanged, pointed at that array.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) unsigned char g_layer_scratch[MOE_NVFP4_STATIC_SCRATCH_BYTES];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxScratchDevices] = {nullptr};

// Device address of g_layer_scratch on the current device. On the host the
// array's name is only a stand-in, so the address is looked up once per
// device (with that device current) and cached.
void* scratch_address(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) {
    *status = MOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_layer_scratch) != cudaSuccess || !ptr) {
      *status = MOE_ERR_CUDA;
      return nullptr;
    }
    g_scratch_addr[dev] = ptr;
  }
  *status = MOE_OK;
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace moe

extern "C" int moe_nvfp4_layer_static(const uint16_t* x, int T, int H, int I, const int32_t* topk_ids,
                                      const float* topk_w, int k, const moe_nvfp4_weights_t* w, uint16_t* y,
                                      cudaStream_t stream) {
  // the same argument checks (and status codes) as moe_nvfp4_layer, before the size limit
  const int arg_status = moe::layer_arg_status(x, T, H, I, topk_ids, topk_w, k, w, y);
  if (arg_status != MOE_OK) return arg_status;
  if (T > 0 && k > 0 && moe_nvfp4_layer_workspace_size(T, k, w->E, H, I) > (size_t)MOE_NVFP4_STATIC_SCRATCH_BYTES)
    return MOE_ERR_WORKSPACE;
  int status = MOE_OK;
  void* scratch = moe::scratch_address(&status);
  if (status != MOE_OK) return status;
  return moe_nvfp4_layer(x, T, H, I, topk_ids, topk_w, k, w, scratch, MOE_NVFP4_STATIC_SCRATCH_BYTES, y, stream);
}
