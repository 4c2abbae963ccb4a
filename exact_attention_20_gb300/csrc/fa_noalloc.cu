// fa_fwd_noalloc: the attention forward with a static scratch in place of the
// per-stream workspace, for callers that must not allocate device memory
// during a call.  A server that reserves its whole device-memory budget when
// it starts (weights, a fixed pool for keys and values) has no room for the
// library to take more later, and a cudaMalloc or cudaFree in the middle of a
// step can block on work queued on other streams.  Such callers get the same
// kernels and the same results with no allocation at any call.
//
// The scratch is a file-scope __device__ array in its own translation unit,
// so its module (and the array's device memory) is loaded only when this
// entry point is first used; fa_fwd never touches it.
#include <cuda_runtime.h>

#include <mutex>

#include "fa_gb300.h"
#include "fa_internal.h"

namespace {

// Room for the split-item workspace of up to 160 CTAs at d <= 128:
// 2 parts per CTA x 256 rows x (128 O values + 1 logsumexp) fp32, then 2048
// arrival counters (8 per split item: query tile x warp quadrant; at most
// 256 split items).
constexpr size_t kScratchFloats = static_cast<size_t>(FA_NOALLOC_MAX_CTAS) * 2 * 256 * 129 + 2048;
static_assert(kScratchFloats * sizeof(float) == FA_NOALLOC_SCRATCH_BYTES,
              "the header states the scratch size");

static __device__ __align__(256) float g_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};

// The scratch's device address on the current device, looked up once per
// device (with that device current); nullptr if the set-up failed.  The
// set-up also clears the whole array, so that the arrival counters start at
// zero (every call leaves them at zero again).
float* scratch_address(int dev) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) return nullptr;
    if (cudaMemset(p, 0, kScratchFloats * sizeof(float)) != cudaSuccess) return nullptr;
    if (cudaDeviceSynchronize() != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int N, int d, int causal, float scale, void* stream) {
  const int rc = fa_internal::check_fwd_args(q, k, v, o, lse, B, H, N, d, causal, scale);
  if (rc != FA_OK) return rc;
  // the device first, as fa_fwd does: the module that holds the scratch is
  // built for sm_103a only and does not load on another device
  fa_internal::DeviceView view;
  if (!fa_internal::current_device(&view)) return FA_ERR_LAUNCH;
  if (!view.supported) return FA_ERR_DEVICE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_LAUNCH;
  float* ptr = scratch_address(dev);
  if (ptr == nullptr) return FA_ERR_LAUNCH;
  return fa_internal::fwd_with_scratch(q, k, v, o, lse, B, H, N, d, causal, scale, stream,
                                       fa_internal::Scratch{ptr, FA_NOALLOC_SCRATCH_BYTES});
}
