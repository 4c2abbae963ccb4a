// C ABI of the fused attention forward: argument checks, TMA tensor maps,
// persistent-grid launch, and the device status word of the bounded waits.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa_gb300.h"
#include "fa_fwd_kernel.cuh"
#include "tma_host.h"

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait
constexpr int kMaxDevices = 64;

__device__ int g_status;  // first failing wait site, 0 when healthy

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  int* status = nullptr;
  bool attr_set[2][2] = {{false, false}, {false, false}};
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// Host-only checks, done before any CUDA call.
int check_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
               int H, int N, int d, int causal, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  const long long elems = static_cast<long long>(B) * H * N * d;
  if (elems >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  auto mis16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (mis16(q) || mis16(k) || mis16(v) || mis16(o)) return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_ALIGN;
  const size_t tb = static_cast<size_t>(elems) * 2;
  const size_t lb = static_cast<size_t>(B) * H * N * 4;
  for (const void* in : {q, k, v}) {
    if (overlaps(o, tb, in, tb) || overlaps(lse, lb, in, tb)) return FA_ERR_ALIAS;
  }
  if (overlaps(o, tb, lse, lb)) return FA_ERR_ALIAS;
  return FA_OK;
}

DeviceInfo* device_info(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  *dev_out = dev;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return nullptr;
    di.supported = (prop.major == 10 && prop.minor == 3);
    di.num_sms = prop.multiProcessorCount;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    di.status = static_cast<int*>(p);
    di.ready = true;
  }
  return &di;
}

template <int D, bool CAUSAL>
int launch(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int N,
           float scale, cudaStream_t stream, DeviceInfo* di, unsigned long long wait_limit_ns,
           int starve_kv, int max_ctas) {
  using C = fa::Cfg<D>;
  CUtensorMap tq, tk, tv;
  if (!fa::encode_bf16_3d(&tq, q, D, N, BH, 64, fa::kBlockM) ||
      !fa::encode_bf16_3d(&tk, k, D, N, BH, 64, fa::kBlockN) ||
      !fa::encode_bf16_3d(&tv, v, D, N, BH, 64, fa::kBlockN))
    return FA_ERR_LAUNCH;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    bool& set = di->attr_set[D == 128][CAUSAL];
    if (!set) {
      if (cudaFuncSetAttribute(fa::fa_fwd_kernel<D, CAUSAL>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::kSmemBytes) != cudaSuccess)
        return FA_ERR_LAUNCH;
      set = true;
    }
  }
  fa::FwdParams p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.status = di->status;
  p.N = N;
  p.BH = BH;
  p.n_key_tiles = (N + fa::kBlockN - 1) / fa::kBlockN;
  p.n_row_blocks = (N + fa::kItemRows - 1) / fa::kItemRows;
  p.num_items = BH * p.n_row_blocks;
  p.qk_scale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.wait_limit_ns = wait_limit_ns;
  p.starve_kv = starve_kv;
  int grid = p.num_items < di->num_sms ? p.num_items : di->num_sms;
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  fa::fa_fwd_kernel<D, CAUSAL><<<grid, fa::kNumThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int dispatch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
             int d, int causal, float scale, cudaStream_t stream, unsigned long long wait_limit_ns,
             int starve_kv, int max_ctas) {
  int rc = check_args(q, k, v, o, lse, B, H, N, d, causal, scale);
  if (rc != FA_OK) return rc;
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (di == nullptr) return FA_ERR_LAUNCH;
  if (!di->supported) return FA_ERR_DEVICE;
  const int BH = B * H;
  if (d == 128)
    return causal ? launch<128, true>(q, k, v, o, lse, BH, N, scale, stream, di, wait_limit_ns, starve_kv, max_ctas)
                  : launch<128, false>(q, k, v, o, lse, BH, N, scale, stream, di, wait_limit_ns, starve_kv, max_ctas);
  return causal ? launch<64, true>(q, k, v, o, lse, BH, N, scale, stream, di, wait_limit_ns, starve_kv, max_ctas)
                : launch<64, false>(q, k, v, o, lse, BH, N, scale, stream, di, wait_limit_ns, starve_kv, max_ctas);
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, int causal, float scale, void* stream) {
  return dispatch(q, k, v, o, lse, B, H, N, d, causal, scale, static_cast<cudaStream_t>(stream),
                  kWaitLimitNs, 0, 0);
}

const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "FA_OK: success";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid size, head dimension, mask flag or scale";
    case FA_ERR_NULL: return "FA_ERR_NULL: a required pointer is NULL";
    case FA_ERR_ALIGN: return "FA_ERR_ALIGN: q, k, v, o must be 16-byte aligned and lse 4-byte aligned";
    case FA_ERR_ALIAS: return "FA_ERR_ALIAS: an output overlaps an input or the other output";
    case FA_ERR_DEVICE: return "FA_ERR_DEVICE: the current device is not sm_103 (GB300)";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: a CUDA call failed";
    case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT: a pipeline wait inside the kernel gave up";
    default: return "unknown fa status code";
  }
}

int fa_get_device_status(void* stream) {
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (di == nullptr) return FA_ERR_LAUNCH;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int h = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_LAUNCH;
  if (cudaMemcpy(&h, di->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_LAUNCH;
  if (h == 0) return FA_OK;
  const int zero = 0;
  if (cudaMemcpy(di->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return FA_ERR_DEVICE_TIMEOUT;
}

int fa_watchdog_selftest(const void* q, const void* k, const void* v, void* o, float* lse,
                         int limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 10000) return FA_ERR_INVALID_ARG;
  const unsigned long long lim = static_cast<unsigned long long>(limit_ms) * 1000000ull;
  int rc = dispatch(q, k, v, o, lse, 1, 1, 128, 64, 0, 0.125f, static_cast<cudaStream_t>(stream),
                    lim, /*starve_kv=*/1, /*max_ctas=*/1);
  if (rc != FA_OK) return rc;
  return fa_get_device_status(stream);
}

int fa_version(void) { return kVersion; }

}  // extern "C"
