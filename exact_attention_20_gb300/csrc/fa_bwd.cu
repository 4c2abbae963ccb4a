// C ABI of the exact attention backward: argument checks, the per-stream
// workspace (fp32 dQ accumulator, per-row L and D), TMA tensor maps, and the
// three launches (prep, the fused backward kernel, dQ conversion).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "fa_bwd_kernel.cuh"
#include "fa_gb300.h"
#include "fa_internal.h"
#include "tma_host.h"

namespace {

constexpr int kMaxDevices = 64;

struct Workspace {
  int dev;
  cudaStream_t stream;
  void* ptr;
  size_t bytes;
};

std::mutex g_mu;
std::vector<Workspace> g_ws;
bool g_attr[kMaxDevices][2][2];

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace layout: the fp32 dQ accumulator [BH][Nq][d], then L * log2(e)
// and D = rowsum(dO * O), each [BH][Nq_pad] fp32.
struct Layout {
  size_t lp, dsum, total;
};

Layout layout(long long BH, int Nq, int Nq_pad, int d) {
  Layout l;
  l.lp = align256(static_cast<size_t>(BH) * Nq * d * 4);
  l.dsum = l.lp + align256(static_cast<size_t>(BH) * Nq_pad * 4);
  l.total = l.dsum + align256(static_cast<size_t>(BH) * Nq_pad * 4);
  return l;
}

// This stream's workspace, grown when a call needs more.  A buffer being
// replaced may still be in use by earlier calls on the stream, which are
// waited for first.
void* stream_workspace(int dev, cudaStream_t s, size_t bytes) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto& w : g_ws) {
    if (w.dev != dev || w.stream != s) continue;
    if (w.bytes >= bytes) return w.ptr;
    if (cudaStreamSynchronize(s) != cudaSuccess) return nullptr;
    cudaFree(w.ptr);
    w.ptr = nullptr;
    w.bytes = 0;
    if (cudaMalloc(&w.ptr, bytes) != cudaSuccess) {
      w.ptr = nullptr;
      return nullptr;
    }
    w.bytes = bytes;
    return w.ptr;
  }
  void* p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) return nullptr;
  g_ws.push_back(Workspace{dev, s, p, bytes});
  return p;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// Host-only checks, done before any CUDA call.
int check_bwd_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dout, const void* dq, const void* dk, const void* dv, int B, int H,
                   int Nq, int Nk, int d, int causal, float scale) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const long long nq_pad = (static_cast<long long>(Nq) + 63) / 64 * 64;
  if (BH * nq_pad * d >= (1ll << 31) || BH * Nk * d >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (BH > 65535) return FA_ERR_INVALID_ARG;  // the grid's y dimension without the mask
  if (causal && (static_cast<long long>(Nk) + 127) / 128 > 65535) return FA_ERR_INVALID_ARG;  // ... with it
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_NULL;
  auto mis16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  for (const void* p : {q, k, v, o, dout, dq, dk, dv})
    if (mis16(p)) return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_ALIGN;
  const size_t qb = static_cast<size_t>(BH) * Nq * d * 2;
  const size_t kb = static_cast<size_t>(BH) * Nk * d * 2;
  const size_t lb = static_cast<size_t>(BH) * Nq * 4;
  const void* ins[6] = {q, k, v, o, dout, lse};
  const size_t in_bytes[6] = {qb, kb, kb, qb, qb, lb};
  const void* outs[3] = {dq, dk, dv};
  const size_t out_bytes[3] = {qb, kb, kb};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 6; ++j)
      if (overlaps(outs[i], out_bytes[i], ins[j], in_bytes[j])) return FA_ERR_ALIAS;
    for (int j = i + 1; j < 3; ++j)
      if (overlaps(outs[i], out_bytes[i], outs[j], out_bytes[j])) return FA_ERR_ALIAS;
  }
  return FA_OK;
}

template <int D, bool CAUSAL>
int launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
               const void* dout, void* dq, void* dk, void* dv, int BH, int Nq, int Nk, float scale,
               cudaStream_t stream, int dev, const fa_internal::DeviceView& view) {
  using C = fa::bwd::Cfg<D>;
  const int nq_pad = (Nq + fa::bwd::kBlockQ - 1) / fa::bwd::kBlockQ * fa::bwd::kBlockQ;
  const int n_kb = (Nk + fa::bwd::kBlockK - 1) / fa::bwd::kBlockK;
  const Layout lay = layout(BH, Nq, nq_pad, D);
  char* ws = static_cast<char*>(stream_workspace(dev, stream, lay.total));
  if (ws == nullptr) return FA_ERR_LAUNCH;
  float* acc = reinterpret_cast<float*>(ws);
  float* lp = reinterpret_cast<float*>(ws + lay.lp);
  float* dsum = reinterpret_cast<float*>(ws + lay.dsum);

  CUtensorMap tq, tk, tv, tdo;
  if (!fa::encode_bf16_3d(&tq, q, D, Nq, BH, 64, fa::bwd::kBlockQ) ||
      !fa::encode_bf16_3d(&tdo, dout, D, Nq, BH, 64, fa::bwd::kBlockQ) ||
      !fa::encode_bf16_3d(&tk, k, D, Nk, BH, 64, fa::bwd::kBlockK) ||
      !fa::encode_bf16_3d(&tv, v, D, Nk, BH, 64, fa::bwd::kBlockK))
    return FA_ERR_LAUNCH;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    bool& set = g_attr[dev][D == 128][CAUSAL];
    if (!set) {
      if (cudaFuncSetAttribute(fa::bwd::fa_bwd_kernel<D, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::kSmemBytes) != cudaSuccess)
        return FA_ERR_LAUNCH;
      set = true;
    }
  }

  const long long prep_rows = static_cast<long long>(BH) * nq_pad;
  const int prep_blocks =
      static_cast<int>(std::min<long long>((prep_rows + 7) / 8, static_cast<long long>(view.num_sms) * 16));
  fa::bwd::fa_bwd_prep_kernel<D><<<prep_blocks, 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, lp, dsum, acc, BH, Nq,
      nq_pad);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;

  fa::bwd::BwdParams p;
  p.dq_acc = acc;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.lp = lp;
  p.dsum = dsum;
  p.status = view.status;
  p.Nq = Nq;
  p.Nk = Nk;
  p.Nq_pad = nq_pad;
  p.n_qt = nq_pad / fa::bwd::kBlockQ;
  p.qk_scale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.scale = scale;
  p.wait_limit_ns = fa_internal::kWaitLimitNs;
  fa::bwd::fa_bwd_kernel<D, CAUSAL>
      <<<CAUSAL ? dim3(BH, n_kb) : dim3(n_kb, BH), fa::bwd::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;

  const long long n8 = static_cast<long long>(BH) * Nq * D / 8;
  const int cvt_blocks =
      static_cast<int>(std::min<long long>((n8 + 255) / 256, static_cast<long long>(view.num_sms) * 8));
  fa::bwd::fa_bwd_dq_kernel<<<cvt_blocks, 256, 0, stream>>>(acc, static_cast<__nv_bfloat16*>(dq), n8, scale);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  return FA_OK;
}

}  // namespace

namespace fa_internal {

bool release_bwd_workspace(int dev, void* stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (size_t i = 0; i < g_ws.size(); ++i) {
    if (g_ws[i].dev != dev || g_ws[i].stream != static_cast<cudaStream_t>(stream)) continue;
    const bool ok = cudaFree(g_ws[i].ptr) == cudaSuccess;
    g_ws.erase(g_ws.begin() + static_cast<long>(i));
    return ok;
  }
  return true;
}

}  // namespace fa_internal

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
           void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, int causal, float scale,
           void* stream) {
  const int rc = check_bwd_args(q, k, v, o, lse, dout, dq, dk, dv, B, H, Nq, Nk, d, causal, scale);
  if (rc != FA_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_LAUNCH;
  fa_internal::DeviceView view;
  if (!fa_internal::current_device(&view)) return FA_ERR_LAUNCH;
  if (!view.supported) return FA_ERR_DEVICE;
  const int BH = B * H;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 128)
    return causal ? launch_bwd<128, true>(q, k, v, o, lse, dout, dq, dk, dv, BH, Nq, Nk, scale, s, dev, view)
                  : launch_bwd<128, false>(q, k, v, o, lse, dout, dq, dk, dv, BH, Nq, Nk, scale, s, dev, view);
  return causal ? launch_bwd<64, true>(q, k, v, o, lse, dout, dq, dk, dv, BH, Nq, Nk, scale, s, dev, view)
                : launch_bwd<64, false>(q, k, v, o, lse, dout, dq, dk, dv, BH, Nq, Nk, scale, s, dev, view);
}

}  // extern "C"
