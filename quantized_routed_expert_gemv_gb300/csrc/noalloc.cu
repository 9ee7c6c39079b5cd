// noalloc.cu -- moe_decode_noalloc: the decode step with its workspace in a
// fixed, statically sized device array of this library instead of a buffer
// the caller allocates; moe_check_noalloc: its status and reset.
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
// above it is rejected (the header names the largest B of the large layer).
constexpr size_t kScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};  // device address of g_scratch, per device, once set up

}  // namespace

namespace moe {
int report_error(int code, const char* msg);  // sets moe_last_error()
int layer_device(const moe_layer* L);         // -1 for an invalid handle
int check_scratch(void* ws, cudaStream_t st, const char* name);
}  // namespace moe

// The current device, which must be the layer's; -1 (with the error set)
// otherwise.
static int current_layer_device(const moe_layer* layer, const char* name, int* rc) {
  char msg[192];
  const int ldev = moe::layer_device(layer);
  if (ldev < 0) {
    std::snprintf(msg, sizeof msg, "%s: invalid layer handle", name);
    *rc = moe::report_error(MOE_ERR_ARG, msg);
    return -1;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    std::snprintf(msg, sizeof msg, "%s: cudaGetDevice failed", name);
    *rc = moe::report_error(MOE_ERR_CUDA, msg);
    return -1;
  }
  if (dev != ldev || dev >= kMaxDevices) {
    std::snprintf(msg, sizeof msg, "%s: the layer's device must be the current device (ordinal below %d)",
                  name, kMaxDevices);
    *rc = moe::report_error(MOE_ERR_ARG, msg);
    return -1;
  }
  return dev;
}

extern "C" int moe_decode_noalloc(moe_layer* layer, const uint16_t* x, int32_t B, uint16_t* out_bf16,
                                  float* out_f32, int32_t* ids, float* weights, void* stream) {
  if (moe::layer_device(layer) < 0) return moe::report_error(MOE_ERR_ARG, "moe_decode_noalloc: invalid layer handle");
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
  int rc = MOE_OK;
  const int dev = current_layer_device(layer, "moe_decode_noalloc", &rc);
  if (dev < 0) return rc;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ws = g_addr[dev];
    if (!ws) {
      // First call on this device: look up the scratch's address (with this
      // device current) and zero it on the caller's stream, ordered before
      // the step below.
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess)
        return moe::report_error(MOE_ERR_CUDA, "moe_decode_noalloc: cudaGetSymbolAddress of the scratch failed");
      if (cudaMemsetAsync(p, 0, kScratchBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return moe::report_error(MOE_ERR_CUDA, "moe_decode_noalloc: zeroing the scratch failed");
      g_addr[dev] = ws = p;
    }
  }
  return moe_decode(layer, x, B, out_bf16, out_f32, ids, weights, ws, kScratchBytes, stream);
}

extern "C" int moe_check_noalloc(const moe_layer* layer, void* stream) {
  int rc = MOE_OK;
  const int dev = current_layer_device(layer, "moe_check_noalloc", &rc);
  if (dev < 0) return rc;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ws = g_addr[dev];
  }
  if (!ws) return MOE_OK;  // no no-alloc step has run on this device
  return moe::check_scratch(ws, static_cast<cudaStream_t>(stream), "moe_check_noalloc");
}
