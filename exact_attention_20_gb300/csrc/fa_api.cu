// C ABI of the fused attention forward: argument checks, TMA tensor maps,
// persistent-grid launch, and the device status word of the bounded waits.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <utility>
#include <vector>

#include "fa_gb300.h"
#include "fa_decode.cuh"
#include "fa_fwd_kernel.cuh"
#include "fa_internal.h"
#include "tma_host.h"

namespace {

constexpr int kVersion = 100;  // 0.1.0
using fa_internal::kWaitLimitNs;  // 2 s per pipeline wait
constexpr int kMaxDevices = 64;

__device__ int g_status;  // first failing wait site, 0 when healthy

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  int* status = nullptr;
  bool attr_set[2][2][2][2] = {};  // [FP8 path][d == 128][causal][items pair heads]
  bool decode_attr_set[2][3] = {};  // decode kernels: [d == 128][rows 1, 2, 4]
  // Workspace for the parts of split items, one per stream so that calls on
  // different streams never share it.  Allocated on a stream's first call.
  std::vector<std::pair<cudaStream_t, float*>> workspaces;
  // Caller-supplied scratch areas used so far (their counters are cleared
  // with the per-stream ones after a kernel gave up).
  std::vector<float*> fixed_scratch;
};

std::mutex g_mu;
std::mutex g_plan_mu;    // guards the shared launch parameter block
DeviceInfo g_dev[kMaxDevices];

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

// Host-only checks, done before any CUDA call.  q and o hold Nq rows per
// (b, h), k and v hold Nk.
int check_args(const void* q, const void* k, const void* v, const void* o, const float* lse, int B,
               int H, int Nq, int Nk, int d, int causal, float scale) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  const long long elems_q = static_cast<long long>(B) * H * Nq * d;
  const long long elems_k = static_cast<long long>(B) * H * Nk * d;
  if (elems_q >= (1ll << 31) || elems_k >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  auto mis16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (mis16(q) || mis16(k) || mis16(v) || mis16(o)) return FA_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_ALIGN;
  const size_t qb = static_cast<size_t>(elems_q) * 2;  // q and o
  const size_t kb = static_cast<size_t>(elems_k) * 2;  // k and v
  const size_t lb = static_cast<size_t>(B) * H * Nq * 4;
  if (overlaps(o, qb, q, qb) || overlaps(lse, lb, q, qb)) return FA_ERR_ALIAS;
  for (const void* in : {k, v}) {
    if (overlaps(o, qb, in, kb) || overlaps(lse, lb, in, kb)) return FA_ERR_ALIAS;
  }
  if (overlaps(o, qb, lse, lb)) return FA_ERR_ALIAS;
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

// Host copy of the kernel's work accounting (decode_item, tiles_for, item_steps).
struct PlanShape {
  int Nq, BH, nkt, nrb;  // query rows, heads of the items, key tiles, row blocks
  bool causal;
  bool paired;           // each item pairs two heads' single query tiles
};

// Items pair two heads when every head has one query tile (Nq <= 128), the
// heads pair up evenly, and the pairs alone fill every CTA (with fewer, the
// keys of each item would be split, and merging parts of 256 rows costs more
// than the pairing gains); then B*H / 2 items of one row block.
bool pairs_heads(int BH, int Nq, int num_ctas) {
  return Nq <= fa::kBlockM && BH % 2 == 0 && BH / 2 >= num_ctas;
}
PlanShape plan_shape(int BH, int Nq, int Nk, bool causal, int num_ctas) {
  const bool paired = pairs_heads(BH, Nq, num_ctas);
  const int nkt = (Nk + fa::kBlockN - 1) / fa::kBlockN;
  const int nrb = paired ? 1 : (Nq + fa::kItemRows - 1) / fa::kItemRows;
  return PlanShape{Nq, paired ? BH / 2 : BH, nkt, nrb, causal, paired};
}

int host_tiles_for(const PlanShape& s, int rb, int t) {
  const int r0 = fa::tile_row0(rb, t, s.paired);
  if (r0 >= s.Nq) return 0;
  return s.causal ? std::min(r0 / fa::kBlockN + 1, s.nkt) : s.nkt;
}

int host_item_steps(const PlanShape& s, int item) {
  int rb, bh;
  fa::decode_item_shape(item, s.BH, s.nrb, rb, bh);
  return std::max(host_tiles_for(s, rb, 0), host_tiles_for(s, rb, 1));
}

// What a split item costs its CTAs beyond its steps, in steps: publishing
// the parts (fp32 O of 256 rows) and merging them.  Measured on short items
// (1024 tokens, d = 64: whole items faster by 10-20 %) against long ones
// (3001 and 4096 tokens: split faster by 5-25 %).
constexpr long long kMergeSteps = 4;

// The longest CTA's steps when each CTA takes a contiguous run of whole
// items (ceil(items / grid) of them), as plan_launch's fallback assigns them.
long long whole_item_makespan(const std::vector<long long>& start, int items, int grid) {
  const int per = (items + grid - 1) / grid;
  long long worst = 0;
  for (int a = 0; a < items; a += per) worst = std::max(worst, start[std::min(items, a + per)] - start[a]);
  return worst;
}

// Splits the concatenated steps of all items into `grid` equal contiguous
// ranges (one per CTA) and lists the items that end up in several parts.
// With more items than SMs, the ranges are used only when their length plus
// a merge's cost is below the longest run of whole items.  With no more
// items than SMs the keys are split only when every CTA keeps at least 16
// steps; otherwise each CTA takes one whole item.
// Returns false when whole items are the better plan or a split would need
// more parts per item than the merge takes; the caller then uses whole
// items.  num_split = split items.
bool make_plan(const PlanShape& s, int num_ctas, bool allow_split, fa::FwdParams& p, int& grid,
               int& num_split) {
  const int items = s.BH * s.nrb;
  num_split = 0;
  int nslots = 0;
  if (!allow_split) return false;
  std::vector<long long> start(items + 1, 0);
  for (int i = 0; i < items; ++i) start[i + 1] = start[i] + host_item_steps(s, i);
  const long long W = start[items];
  grid = num_ctas;
  if (items > num_ctas &&
      whole_item_makespan(start, items, num_ctas) <= (W + num_ctas - 1) / num_ctas + kMergeSteps)
    return false;
  if (items <= num_ctas) {
    // Few items (few query rows over many keys, the decode shape): their
    // keys are split over more CTAs while each CTA keeps enough steps to
    // amortise the merge, and no item goes into more parts than it takes.
    constexpr long long kMinStepsPerCta = 16;
    grid = static_cast<int>(std::min<long long>(
        {static_cast<long long>(num_ctas), W / kMinStepsPerCta,
         static_cast<long long>(items) * (fa::kMaxPartsPerItem - 1)}));
    if (grid <= items) return false;
  }
  auto locate = [&](long long g, int& item, int& step) {
    item = static_cast<int>(std::upper_bound(start.begin(), start.end(), g) - start.begin()) - 1;
    step = static_cast<int>(g - start[item]);
  };
  auto item_cost = [&](int item) { return host_item_steps(s, item); };
  auto add_part = [&](int item, int slot) {  // returns the split item's index
    const int k = num_split;
    if (k > 0 && p.merge_item[k - 1] == item) {
      p.merge_slots[p.merge_first[k - 1] + p.merge_count[k - 1]] = slot;
      ++p.merge_count[k - 1];
      return k - 1;
    }
    p.merge_item[k] = item;
    p.merge_first[k] = k == 0 ? 0 : p.merge_first[k - 1] + p.merge_count[k - 1];
    p.merge_count[k] = 1;
    p.merge_slots[p.merge_first[k]] = slot;
    ++num_split;
    return k;
  };
  for (int c = 0; c < grid; ++c) {
    const long long g0 = W * c / grid, g1 = W * (c + 1) / grid;
    fa::WorkRange& r = p.range[c];
    fa::SlotPair& sp = p.slots[c];
    sp = {-1, -1, 0, 0};
    if (g1 <= g0) {
      r = {0, 0, -1, 0};
      continue;
    }
    int ib, sb, il, sl;
    locate(g0, ib, sb);
    locate(g1 - 1, il, sl);
    r = {ib, sb, il, sl + 1};
    const int end0 = il == ib ? sl + 1 : item_cost(ib);
    if (sb > 0 || end0 < item_cost(ib)) {
      sp.first = nslots++;
      sp.k_first = add_part(ib, sp.first);
    }
    if (il != ib && sl + 1 < item_cost(il)) {
      sp.last = nslots++;
      sp.k_last = add_part(il, sp.last);
    }
  }
  for (int k = 0; k < num_split; ++k)
    if (p.merge_count[k] > fa::kMaxPartsPerItem) return false;
  return true;
}

// The launch plan: fills p.range / p.slots (and p's merge lists when items
// are split) and returns the attention kernel's grid.
int plan_launch(const PlanShape& shape, int num_ctas, bool allow_split, fa::FwdParams& p,
                int& num_split) {
  int grid = 0;
  if (make_plan(shape, num_ctas, allow_split, p, grid, num_split)) return grid;
  // whole items: each CTA a contiguous run of whole items
  num_split = 0;
  const int items = shape.BH * shape.nrb;
  grid = std::min(items, num_ctas);
  const int per = (items + grid - 1) / grid;
  for (int c = 0; c < grid; ++c) {
    const int a = c * per, b = std::min(items, (c + 1) * per) - 1;
    p.range[c] = a <= b ? fa::WorkRange{a, 0, b, host_item_steps(shape, b)} : fa::WorkRange{0, 0, -1, 0};
    p.slots[c] = {-1, -1, 0, 0};
  }
  return grid;
}

int num_ctas_for(const DeviceInfo* di, int max_ctas) {
  int n = std::min(di->num_sms, fa::kMaxCtas);
  return max_ctas > 0 ? std::min(n, max_ctas) : n;
}

// Workspace layout: part O [slots][256][128] fp32, part LSE [slots][256]
// fp32, then the arrival counters: one int per split item, query tile and
// warp quadrant (zero between launches).
size_t ws_slots(const DeviceInfo* di) { return 2 * static_cast<size_t>(std::min(di->num_sms, fa::kMaxCtas)); }
size_t ws_counter_offset(const DeviceInfo* di) { return ws_slots(di) * fa::kItemRows * (128 + 1); }
size_t ws_bytes(const DeviceInfo* di) { return (ws_counter_offset(di) + fa::kNumCounters) * sizeof(float); }

void remember_fixed_scratch(DeviceInfo* di, float* ws) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (float* f : di->fixed_scratch)
    if (f == ws) return;
  di->fixed_scratch.push_back(ws);
}

// This stream's workspace, allocated on its first splitting call.  Its
// arrival counters are zeroed on `stream` itself, so the kernel that follows
// on the same stream is ordered after the clear whatever kind of stream it
// is (a non-blocking stream is not ordered after the legacy default stream).
float* stream_workspace(DeviceInfo* di, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto& w : di->workspaces)
    if (w.first == stream) return w.second;
  float* ptr = nullptr;
  if (cudaMalloc(&ptr, ws_bytes(di)) != cudaSuccess) return nullptr;
  if (cudaMemsetAsync(ptr + ws_counter_offset(di), 0, fa::kNumCounters * sizeof(int), stream) != cudaSuccess) {
    cudaFree(ptr);
    return nullptr;
  }
  di->workspaces.emplace_back(stream, ptr);
  return ptr;
}

// The FP8 path's per-block scales (all null on the bf16 path).
struct Fp8Scales {
  const float* q = nullptr;
  const float* k = nullptr;
  const float* v = nullptr;
};

template <int D, bool CAUSAL, int E = 2>
int launch(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int Nq, int Nk,
           float scale, cudaStream_t stream, DeviceInfo* di, unsigned long long wait_limit_ns,
           int starve_kv, int max_ctas, const fa_internal::Scratch& fixed, const Fp8Scales& sc = {}) {
  using C = fa::Cfg<D, E>;
  CUtensorMap tq, tk, tv;
  if constexpr (E == 2) {
    if (!fa::encode_bf16_3d(&tq, q, D, Nq, BH, 64, fa::kBlockM) ||
        !fa::encode_bf16_3d(&tk, k, D, Nk, BH, 64, fa::kBlockN) ||
        !fa::encode_bf16_3d(&tv, v, D, Nk, BH, 64, fa::kBlockN))
      return FA_ERR_LAUNCH;
  } else {
    // e4m3 codes: Q [BH][Nq][D] and K [BH][Nk][D] in 128-row boxes of one
    // 128-byte row each; V transposed, [BH][D][Nk_pad], in boxes of D rows of
    // 128 keys
    const uint64_t nk_pad = (static_cast<uint64_t>(Nk) + fa::kBlockN - 1) / fa::kBlockN * fa::kBlockN;
    if (!fa::encode_u8_3d(&tq, q, D, Nq, BH, 128, fa::kBlockM) ||
        !fa::encode_u8_3d(&tk, k, D, Nk, BH, 128, fa::kBlockN) ||
        !fa::encode_u8_3d(&tv, v, nk_pad, D, BH, fa::kBlockN, D))
      return FA_ERR_LAUNCH;
  }
  const PlanShape shape = plan_shape(BH, Nq, Nk, CAUSAL, num_ctas_for(di, max_ctas));
  // the kernel instance: items of one head's two query tiles, or paired heads
  auto kernel = shape.paired ? fa::fa_fwd_kernel<D, CAUSAL, E, true> : fa::fa_fwd_kernel<D, CAUSAL, E, false>;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    bool& set = di->attr_set[E == 1][D == 128][CAUSAL][shape.paired];
    if (!set) {
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
        return FA_ERR_LAUNCH;
      set = true;
    }
  }
  // large (work plan, merge lists): kept off the stack; guarded by g_plan_mu
  static fa::FwdParams p;
  std::lock_guard<std::mutex> plan_lock(g_plan_mu);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.status = di->status;
  p.Nq = Nq;
  p.Nk = Nk;
  p.BH = shape.BH;
  p.n_key_tiles = shape.nkt;
  p.n_row_blocks = shape.nrb;
  p.num_items = shape.BH * shape.nrb;
  p.qk_scale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.wait_limit_ns = wait_limit_ns;
  p.starve_kv = starve_kv;
  p.q_scale = sc.q;
  p.k_scale = sc.k;
  p.v_scale = sc.v;
  p.part_o = nullptr;
  p.part_lse = nullptr;
  int num_split = 0;
  const int grid = plan_launch(shape, num_ctas_for(di, max_ctas), max_ctas == 0, p, num_split);
  p.counters = nullptr;
  if (num_split > 0) {
    // the caller's fixed scratch when given (checked to hold the workspace
    // layout; its counters start at zero), else this stream's own workspace
    float* ws = nullptr;
    if (fixed.ptr != nullptr) {
      if (fixed.bytes < ws_bytes(di)) return FA_ERR_SCRATCH;
      ws = fixed.ptr;
      remember_fixed_scratch(di, ws);
    } else {
      ws = stream_workspace(di, stream);
    }
    if (ws == nullptr) return FA_ERR_LAUNCH;
    p.part_o = ws;
    p.part_lse = ws + ws_slots(di) * fa::kItemRows * 128;
    p.counters = reinterpret_cast<int*>(ws + ws_counter_offset(di));
  }
  kernel<<<grid, fa::kNumThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  return FA_OK;
}

// Few query rows without the causal mask go to the decode kernels.
bool takes_decode(int BH, int Nq, int causal) {
  return causal == 0 && Nq <= fa::decode::kMaxRows && BH <= 65535;
}

// The decode kernels' key chunks: about eight CTAs per SM (two resident at a
// time, so four waves and a short tail), every chunk a whole number of
// rounds (64 keys) and at least four of them, and the chunks' partial
// results within the workspace's part area.
struct DecodePlan {
  int keys_per_chunk;
  int n_chunks;
};
DecodePlan decode_plan(const DeviceInfo* di, int BH, int Nq, int Nk, int d) {
  constexpr int R = fa::decode::kKeysPerRound;
  const int target = std::min(fa::decode::kMaxChunks, std::max(1, (8 * di->num_sms + BH - 1) / BH));
  int kpc = (Nk + target - 1) / target;
  kpc = std::max(4 * R, (kpc + R - 1) / R * R);
  int n = (Nk + kpc - 1) / kpc;
  const size_t cap = ws_counter_offset(di);  // floats before the arrival counters
  const size_t per_chunk = static_cast<size_t>(BH) * Nq * (d + 1);
  if (n > 1 && static_cast<size_t>(n) * per_chunk > cap) {
    const int n_max = static_cast<int>(cap / per_chunk);
    if (n_max < 2) {
      n = 1;
      kpc = (Nk + R - 1) / R * R;
    } else {
      kpc = ((Nk + n_max - 1) / n_max + R - 1) / R * R;
      n = (Nk + kpc - 1) / kpc;
    }
  }
  return DecodePlan{kpc, n};
}

template <int D>
int launch_decode(const void* q, const void* k, const void* v, void* o, float* lse, int BH, int Nq, int Nk,
                  float scale, cudaStream_t stream, DeviceInfo* di) {
  namespace dc = fa::decode;
  const DecodePlan plan = decode_plan(di, BH, Nq, Nk, D);
  dc::Params p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.Nq = Nq;
  p.Nk = Nk;
  p.keys_per_chunk = plan.keys_per_chunk;
  p.n_chunks = plan.n_chunks;
  p.qk_scale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  if (plan.n_chunks > 1) {
    float* ws = stream_workspace(di, stream);
    if (ws == nullptr) return FA_ERR_LAUNCH;
    p.part_o = ws;
    p.part_lse = ws + static_cast<size_t>(BH) * Nq * plan.n_chunks * D;
    // one arrival counter per (b, h) in the workspace's counters (zero
    // between launches): the chunks are then merged in the same launch
    if (BH <= fa::kNumCounters) p.counters = reinterpret_cast<int*>(ws + ws_counter_offset(di));
  }
  p.status = di->status;
  p.wait_limit_ns = kWaitLimitNs;
  const dim3 grid(plan.n_chunks, BH);
  constexpr int smem = dc::smem_bytes<D>();
  auto run = [&](auto kernel, int which) -> bool {
    {
      std::lock_guard<std::mutex> lock(g_mu);
      bool& set = di->decode_attr_set[D == 128][which];
      if (!set) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
          return false;
        set = true;
      }
    }
    kernel<<<grid, dc::kThreadsAll, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess;
  };
  const bool launched = Nq == 1 ? run(dc::partial_kernel<D, 1>, 0)
                        : Nq == 2 ? run(dc::partial_kernel<D, 2>, 1)
                                  : run(dc::partial_kernel<D, 4>, 2);
  if (!launched) return FA_ERR_LAUNCH;
  if (plan.n_chunks > 1 && p.counters == nullptr) {
    dc::merge_kernel<D><<<BH * Nq, D, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

int dispatch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
             int Nk, int d, int causal, float scale, cudaStream_t stream,
             unsigned long long wait_limit_ns, int starve_kv, int max_ctas,
             const fa_internal::Scratch& fixed) {
  int rc = check_args(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale);
  if (rc != FA_OK) return rc;
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (di == nullptr) return FA_ERR_LAUNCH;
  if (!di->supported) return FA_ERR_DEVICE;
  const int BH = B * H;
  // the decode kernels (not for the watchdog self-test, a CTA cap or a
  // caller's fixed scratch, which are the forward kernel's)
  if (takes_decode(BH, Nq, causal) && starve_kv == 0 && max_ctas == 0 && fixed.ptr == nullptr)
    return d == 128 ? launch_decode<128>(q, k, v, o, lse, BH, Nq, Nk, scale, stream, di)
                    : launch_decode<64>(q, k, v, o, lse, BH, Nq, Nk, scale, stream, di);
  if (d == 128)
    return causal ? launch<128, true>(q, k, v, o, lse, BH, Nq, Nk, scale, stream, di, wait_limit_ns, starve_kv, max_ctas, fixed)
                  : launch<128, false>(q, k, v, o, lse, BH, Nq, Nk, scale, stream, di, wait_limit_ns, starve_kv, max_ctas, fixed);
  return causal ? launch<64, true>(q, k, v, o, lse, BH, Nq, Nk, scale, stream, di, wait_limit_ns, starve_kv, max_ctas, fixed)
                : launch<64, false>(q, k, v, o, lse, BH, Nq, Nk, scale, stream, di, wait_limit_ns, starve_kv, max_ctas, fixed);
}

}  // namespace

namespace fa_internal {

int check_fwd_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   int B, int H, int N, int d, int causal, float scale) {
  return check_args(q, k, v, o, lse, B, H, N, N, d, causal, scale);
}

bool current_device(DeviceView* out) {
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (di == nullptr) return false;
  out->status = di->status;
  out->supported = di->supported;
  out->num_sms = di->num_sms;
  return true;
}

int fwd_with_scratch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int N, int d, int causal, float scale, void* stream, const Scratch& scratch) {
  return dispatch(q, k, v, o, lse, B, H, N, N, d, causal, scale, static_cast<cudaStream_t>(stream),
                  kWaitLimitNs, 0, 0, scratch);
}

}  // namespace fa_internal

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, int causal, float scale, void* stream) {
  return dispatch(q, k, v, o, lse, B, H, N, N, d, causal, scale, static_cast<cudaStream_t>(stream),
                  kWaitLimitNs, 0, 0, fa_internal::Scratch{});
}

int fa_fwd_rect(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int Nq, int Nk, int d, int causal, float scale, void* stream) {
  return dispatch(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, static_cast<cudaStream_t>(stream),
                  kWaitLimitNs, 0, 0, fa_internal::Scratch{});
}

int fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale, const float* k_scale,
               const float* v_scale, void* o, float* lse, int B, int H, int N, int d, int causal, float scale,
               void* stream) {
  if (B < 1 || H < 1 || N < 1 || d != 128 || (causal != 0 && causal != 1)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  const long long n_pad = (static_cast<long long>(N) + fa::kBlockN - 1) / fa::kBlockN * fa::kBlockN;
  if (BH * n_pad * d >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (!q8 || !k8 || !vt8 || !q_scale || !k_scale || !v_scale || !o || !lse) return FA_ERR_NULL;
  auto mis = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (mis(q8, 16) || mis(k8, 16) || mis(vt8, 16) || mis(o, 16)) return FA_ERR_ALIGN;
  if (mis(q_scale, 4) || mis(k_scale, 4) || mis(v_scale, 4) || mis(lse, 4)) return FA_ERR_ALIGN;
  const size_t nblk = static_cast<size_t>(n_pad / fa::kBlockN);
  const size_t ob = static_cast<size_t>(BH) * N * d * 2, lb = static_cast<size_t>(BH) * N * 4;
  const void* ins[6] = {q8, k8, vt8, q_scale, k_scale, v_scale};
  const size_t in_bytes[6] = {static_cast<size_t>(BH) * N * d, static_cast<size_t>(BH) * N * d,
                              static_cast<size_t>(BH) * d * n_pad, BH * nblk * 4, BH * nblk * 4,
                              static_cast<size_t>(BH) * 4};
  for (int i = 0; i < 6; ++i)
    if (overlaps(o, ob, ins[i], in_bytes[i]) || overlaps(lse, lb, ins[i], in_bytes[i])) return FA_ERR_ALIAS;
  if (overlaps(o, ob, lse, lb)) return FA_ERR_ALIAS;
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (di == nullptr) return FA_ERR_LAUNCH;
  if (!di->supported) return FA_ERR_DEVICE;
  Fp8Scales sc;
  sc.q = q_scale;
  sc.k = k_scale;
  sc.v = v_scale;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return causal ? launch<128, true, 1>(q8, k8, vt8, o, lse, static_cast<int>(BH), N, N, scale, s, di, kWaitLimitNs,
                                       0, 0, fa_internal::Scratch{}, sc)
                : launch<128, false, 1>(q8, k8, vt8, o, lse, static_cast<int>(BH), N, N, scale, s, di,
                                        kWaitLimitNs, 0, 0, fa_internal::Scratch{}, sc);
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
    case FA_ERR_SCRATCH:
      return "FA_ERR_SCRATCH: the work plan needs more scratch than fa_fwd_noalloc's static scratch holds";
    default: return "unknown fa status code";
  }
}

int fa_get_device_status(void* stream) {
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (di == nullptr) return FA_ERR_LAUNCH;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int h = 0;
  if (cudaMemcpyAsync(&h, di->status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FA_ERR_LAUNCH;
  if (h == 0) return FA_OK;
  // A kernel that gave up may have left the arrival counters of some
  // workspace or scratch non-zero, and the status word does not say which
  // stream's kernel it was.  Once every stream of the device is idle, clear
  // the status word and every area's counters, ordered on `stream`, and wait
  // for the clears before returning.
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_LAUNCH;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (cudaMemsetAsync(di->status, 0, sizeof(int), s) != cudaSuccess) return FA_ERR_LAUNCH;
    std::vector<float*> areas = di->fixed_scratch;
    for (auto& w : di->workspaces) areas.push_back(w.second);
    for (float* a : areas)
      if (cudaMemsetAsync(a + ws_counter_offset(di), 0, fa::kNumCounters * sizeof(int), s) != cudaSuccess)
        return FA_ERR_LAUNCH;
  }
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_LAUNCH;
  return FA_ERR_DEVICE_TIMEOUT;
}

int fa_release_stream(void* stream) {
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (di == nullptr) return FA_ERR_LAUNCH;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_LAUNCH;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (size_t i = 0; i < di->workspaces.size(); ++i) {
      if (di->workspaces[i].first != s) continue;
      if (cudaFree(di->workspaces[i].second) != cudaSuccess) return FA_ERR_LAUNCH;
      di->workspaces.erase(di->workspaces.begin() + static_cast<long>(i));
      break;
    }
  }
  return fa_internal::release_bwd_workspace(dev, s) ? FA_OK : FA_ERR_LAUNCH;
}

int fa_watchdog_selftest(const void* q, const void* k, const void* v, void* o, float* lse,
                         int limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 10000) return FA_ERR_INVALID_ARG;
  const unsigned long long lim = static_cast<unsigned long long>(limit_ms) * 1000000ull;
  int rc = dispatch(q, k, v, o, lse, 1, 1, 128, 128, 64, 0, 0.125f, static_cast<cudaStream_t>(stream),
                    lim, /*starve_kv=*/1, /*max_ctas=*/1, fa_internal::Scratch{});
  if (rc != FA_OK) return rc;
  return fa_get_device_status(stream);
}

int fa_fwd_plan(int B, int H, int Nq, int Nk, int d, int causal, int* num_ctas,
                int* num_split_items) {
  if (num_ctas == nullptr || num_split_items == nullptr) return FA_ERR_NULL;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || (d != 64 && d != 128) || (causal != 0 && causal != 1))
    return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * Nq * d >= (1ll << 31) ||
      static_cast<long long>(B) * H * Nk * d >= (1ll << 31))
    return FA_ERR_INVALID_ARG;
  int dev = 0;
  DeviceInfo* di = device_info(&dev);
  if (di == nullptr) return FA_ERR_LAUNCH;
  if (!di->supported) return FA_ERR_DEVICE;
  const int BH = B * H;
  if (takes_decode(BH, Nq, causal)) {
    // the decode kernels: one CTA per key chunk and (batch, head); the heads'
    // keys are split when there is more than one chunk
    const DecodePlan plan = decode_plan(di, BH, Nq, Nk, d);
    *num_ctas = plan.n_chunks * BH;
    *num_split_items = plan.n_chunks > 1 ? BH : 0;
    return FA_OK;
  }
  static fa::FwdParams p;
  int num_split = 0;
  std::lock_guard<std::mutex> plan_lock(g_plan_mu);
  const int ctas = num_ctas_for(di, 0);
  *num_ctas = plan_launch(plan_shape(BH, Nq, Nk, causal == 1, ctas), ctas, true, p, num_split);
  *num_split_items = num_split;
  return FA_OK;
}

int fa_version(void) { return kVersion; }

}  // extern "C"
