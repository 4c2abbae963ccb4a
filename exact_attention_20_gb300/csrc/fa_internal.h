// Internal interface between the library's translation units (not part of
// the C ABI).
#pragma once

#include <cstddef>

namespace fa_internal {

// Device memory a caller supplies for the parts of split work items in place
// of the per-stream workspace; ptr == nullptr selects the per-stream one.
struct Scratch {
  float* ptr = nullptr;
  size_t bytes = 0;
};

// fa_fwd's host-side argument checks (no CUDA call); FA_OK or an fa_status.
int check_fwd_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   int B, int H, int N, int d, int causal, float scale);

// fa_fwd with the given scratch for the parts of split items; FA_ERR_SCRATCH
// when the scratch is smaller than the workspace layout the launch needs.
int fwd_with_scratch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int N, int d, int causal, float scale, void* stream, const Scratch& scratch);

// The current device as the library sees it: its status word (written by a
// kernel whose bounded wait gave up), whether it is an sm_103 part, and its
// SM count.  False when a CUDA call failed.
struct DeviceView {
  int* status = nullptr;
  bool supported = false;
  int num_sms = 0;
};
bool current_device(DeviceView* out);

// Frees the backward's workspace of `stream` on device `dev`, if it has one
// (the caller has synchronised the stream).  False when cudaFree failed.
bool release_bwd_workspace(int dev, void* stream);

// Wait limit of every pipeline wait inside the kernels, in nanoseconds.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

}  // namespace fa_internal
