// noalloc.cu -- moe_decode_noalloc: the decode step with its workspace in a
// fixed, statically sized device array of this library instead of a buffer
// the caller allocates.
//
// Who needs it: a host that has no device allocator to hand (a plain C
// runtime without a caching allocator), or one that must not allocate while
// it serves a step: cudaMalloc and cudaFree synchronise the device, which
// stalls every other stream of the process, and an allocator that has
// already handed all of HBM to its own pool has nothing left to give.  This
// entry point makes no allocation of any kind (no cudaMalloc / cudaFree, no
// allocating library routine).
#include <cstddef>
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace {

// Largest workspace this entry point serves: moe_workspace_bytes(layer, B)
// above it is rejected.  4 MiB holds, e.g., H=7168 E=512 top-16 F=Fs=2048
// up to B = 16.
constexpr size_t kScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};  // device address of g_scratch, per device, once set up

}  // namespace

namespace moe {
int report_error(int code, const char* msg);  // sets moe_last_error()
int layer_device(const moe_layer* L);         // -1 for an invalid handle
}  // namespace moe

extern "C" int moe_decode_noalloc(moe_layer* layer, const uint16_t* x, int32_t B, uint16_t* out_bf16,
                                  float* out_f32, int32_t* ids, float* weights, void* stream) {
  const int ldev = moe::layer_device(layer);
  if (ldev < 0) return moe::report_error(MOE_ERR_ARG, "moe_decode_noalloc: invalid layer handle");
  if (B == 0) return MOE_OK;
  const size_t need = moe_workspace_bytes(layer, B);
  if (need == 0) {
    char msg[160];
    std::snprintf(msg, sizeof msg, "moe_decode_noalloc: token count %d outside [0, max_tokens]", B);
    return moe::report_error(MOE_ERR_ARG, msg);
  }
  if (need > kScratchBytes) {
    char msg[256];
    std::snprintf(msg, sizeof msg,
                  "moe_decode_noalloc: B=%d needs %zu B of workspace, more than the %zu B static scratch; "
                  "use moe_decode with a caller-allocated workspace",
                  B, need, kScratchBytes);
    return moe::report_error(MOE_ERR_ARG, msg);
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return moe::report_error(MOE_ERR_CUDA, "moe_decode_noalloc: cudaGetDevice failed");
  if (dev != ldev)
    return moe::report_error(MOE_ERR_ARG, "moe_decode_noalloc: the layer's device must be the current device");
  if (dev >= kMaxDevices) return moe::report_error(MOE_ERR_ARG, "moe_decode_noalloc: device ordinal above 63");
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ws = g_addr[dev];
    if (!ws) {
      // First call on this device: look up the scratch's address (with this
      // device current) and zero it on the caller's stream, ordered before
      // the step below.
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_scratch)) != cudaSuccess)
        return moe::report_error(MOE_ERR_CUDA, "moe_decode_noalloc: cudaGetSymbolAddress of the scratch failed");
      if ((e = cudaMemsetAsync(p, 0, kScratchBytes, static_cast<cudaStream_t>(stream))) != cudaSuccess)
        return moe::report_error(MOE_ERR_CUDA, "moe_decode_noalloc: zeroing the scratch failed");
      g_addr[dev] = ws = p;
    }
  }
  return moe_decode(layer, x, B, out_bf16, out_f32, ids, weights, ws, kScratchBytes, stream);
}
