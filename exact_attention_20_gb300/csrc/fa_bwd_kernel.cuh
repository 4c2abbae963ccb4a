// Exact attention backward for sm_103a: dQ, dK and dV from Q, K, V, the
// forward's O and logsumexp L, and the upstream gradient dO.
//
// The method ("FlashAttention and kernels.", section "The backward pass:
// recompute instead of remember"; "FlashAttention 2 from PyTorch to Triton",
// section "What I am building"): the forward never stores P; every tile of it
// is rebuilt from the scores and L as P = exp(S - L), with no running
// maximum.  With D = rowsum(dO * O), one number per query row computed once,
//   dV += P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//   dQ += scale dS K,  dK += scale dS^T Q.
// Exponentials are taken in base 2: L is passed in log2 units and the scale
// is folded into one FMA (the forward's exp2 trick, "How to profile and
// optimise kernels", Round 4).
//
// GB300 mapping.  One CTA per (batch*head, block of 128 keys).  It keeps the
// block's K and V in shared memory and its dK and dV accumulators in tensor
// memory for the whole launch, and walks the query rows 64 at a time (a
// step).  Every product is taken transposed so that the 128 keys are the
// tensor-memory lanes and one thread owns one key row:
//   S^T  = K Q^T      M = 128 keys, N = 64 queries, K = d
//   dP^T = V dO^T     same shape
//   dV  += P^T dO     M = 128 keys, N = d, K = 64 queries (P^T read from TMEM)
//   dK  += dS^T Q     same shape (dS^T read from TMEM)
//   dQ^T = K^T dS^T   M = d (128 lanes), N = 64 queries, K = 128 keys (dS^T
//                     read from shared memory)
// Every key block adds to every query row's dQ, so each step's dQ^T is added
// into an fp32 accumulator in global memory: the drain warps write it to a
// shared-memory tile (64 query rows of d values, the accumulator's own row
// layout) and one bulk reduction adds the tile to the step's rows, the adds
// done in L2.  With d = 64 the dQ^T product
// still has M = 128: rows 64-127 of its A operand are V^T (the tile that
// follows K in shared memory) and those lanes are ignored.
//
// Warp roles (12 warps, 384 threads):
//   warp 0     TMA producer: K and V once; Q, dO and their rows' L and D per step
//   warp 1     MMA issuer B (one lane issues): dV, dK, dQ^T; owner of the
//              TMEM allocation
//   warp 2     MMA issuer A (one lane issues): S^T, dP^T
//   warp 3     idle
//   warps 4-7  P and dS, one key row per thread; then dV of the row
//   warps 8-11 dQ drain: one row of dQ^T (a column of d) per thread, reduced
//              into the fp32 accumulator; then scale * dK of a key row
// Tensor memory (32-bit columns): three 64-column buffers at 0, 64 and 128,
// one per step in turn: a step's S^T, then its P^T and dS^T (bf16, the
// first and the second 32 columns, written over S^T by the threads), then
// its dQ^T (written once dV and dK have read P^T and dS^T); dP^T at 192, dV
// at 256, dK at 384.  The dS^T tile in shared memory has two buffers.  A
// buffer takes S^T again once the drain has read its dQ^T, so S^T runs up to
// three steps ahead of the threads.
//
// At M = 128 the tensor core takes an N = 64 instruction every 48 cycles and
// accepts about one more than it is running, so an issuer that stops to wait
// for a barrier leaves it idle; a product's result reaches the threads about
// 220 cycles after its last instruction.  The products are therefore issued
// by two warps, each waiting only for its own operands: issuer A computes
// the threads' next operands (dP^T(it+1) as soon as the threads have read
// dP^T(it), S^T(it+2) as soon as the drain has read dQ^T(it-1) from its
// buffer), issuer B the products of the threads' last step (dV(it), dK(it),
// dQ^T(it)).  While one waits, the other's instructions keep the tensor core
// busy.
#pragma once

#include <cuda_bf16.h>

#include "sm103_ptx.cuh"

namespace fa {
namespace bwd {

constexpr int kBlockK = 128;   // keys per CTA
constexpr int kBlockQ = 64;    // query rows per step
constexpr int kThreads = 384;
constexpr int kLoadWarp = 0;
constexpr int kMmaWarp = 1;    // dV, dK, dQ^T; owns the tensor memory
constexpr int kMmaWarpA = 2;   // S^T, dP^T
constexpr int kDsWarp0 = 4;    // first warp of the P / dS warpgroup
constexpr int kDrainWarp0 = 8; // first warp of the dQ drain warpgroup
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;        // S^T buffers (and dS^T tiles in shared memory)
constexpr uint32_t kColS = 0;    // buffer of step it at kColS + 64 * (it % kSBufs): S^T, then P^T and
                                 // dS^T over it, then dQ^T
constexpr uint32_t kColDP = 192;
constexpr uint32_t kColDV = 256;
constexpr uint32_t kColDK = 384;

// Codes recorded in the device status word when a wait gives up.
constexpr int kSiteProducer = 11;
constexpr int kSiteMma = 12;
constexpr int kSiteDs = 13;
constexpr int kSiteDrain = 14;
constexpr int kSiteAlign = 15;  // dynamic shared memory not 1024-byte aligned
// Steps ahead of the one being loaded whose Q and dO tiles (and L, D) are
// prefetched into L2: the CTAs of a head walk the same steps at about the
// same time, and a tile's first request would otherwise wait on DRAM.
constexpr int kPrefetchSteps = 4;

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dimension 64 or 128");
  // Q / dO ring depth: a step's tiles are requested two steps ahead.
  static constexpr int kStages = 3;
  // A stage is loaded again once dQ^T of the step that last used it is done
  // (below): that barrier must not complete again before the load.
  static_assert(kStages <= kSBufs, "ring deeper than the S^T buffers");
  static constexpr int kKSlab = kBlockK * 128;  // 128 rows x 64 bf16 (one TMA box)
  static constexpr int kQSlab = kBlockQ * 128;  // 64 rows x 64 bf16
  static constexpr int kKTile = (D / 64) * kKSlab;
  static constexpr int kQTile = (D / 64) * kQSlab;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKTile;  // directly after K (see the d = 64 note above)
  static constexpr int kStageOff = kVOff + kKTile;
  static constexpr int kStageBytes = 2 * kQTile;  // Q, then dO
  static constexpr int kDsOff = kStageOff + kStages * kStageBytes;
  static constexpr int kDsBytes = kBlockK * kBlockQ * 2;  // dS^T, bf16 [128 keys][64 queries], two tiles
  static constexpr int kDqOff = kDsOff + 2 * kDsBytes;    // dQ of a step, fp32 [64 queries][D], for the reduction
  static constexpr int kDqBytes = kBlockQ * D * 4;
  static constexpr int kLdOff = kDqOff + kDqBytes;        // per stage: L[64] then D[64], fp32
  static constexpr int kLdBytes = 2 * kBlockQ * 4;
  static constexpr int kBarOff = kLdOff + kStages * kLdBytes;
  static constexpr int kNumBars = 11 + 4 * kSBufs + kStages;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem slot, abort flag
  // No alignment slack: the dynamic shared memory of a CTA starts on a
  // 1024-byte boundary (after the 1 KB the system reserves); the kernel checks
  // this and gives up (status word) if it ever does not.
  static constexpr int kSmemBytes = kMiscOff + 16;
  static_assert(kStageOff % 1024 == 0 && kDsOff % 1024 == 0 && kStageBytes % 1024 == 0 && kDsBytes % 1024 == 0,
                "operand tiles must sit on 1024-byte swizzle atoms");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};

struct BwdParams {
  float* dq_acc;          // workspace [BH][Nq][D] fp32, zero on entry; dQ / scale on exit
  __nv_bfloat16* dk;      // [BH][Nk][D]
  __nv_bfloat16* dv;      // [BH][Nk][D]
  const float* lp;        // workspace [BH][Nq_pad]: L * log2(e); +inf on padding rows
  const float* dsum;      // workspace [BH][Nq_pad]: rowsum(dO * O); 0 on padding rows
  int* status;            // device status word (0 = ok)
  int Nq, Nk, Nq_pad;     // query rows, keys, query rows rounded up to 64
  int n_qt;               // ceil(Nq / 64)
  float qk_scale;         // scale * log2(e)
  float scale;
  unsigned long long wait_limit_ns;
};

// Barrier addresses.  Barriers that come in sets (one per stage or buffer)
// are adjacent, so the one of buffer b is the first one's address + 8 b (no
// run-time array index, which would put the struct in local memory).
// Buffer barriers complete once every kSBufs steps:
//   s_full(b)   S^T of a step in buffer b
//   sm_done(b)  the threads' P^T, dS^T of a step in buffer b are in, and its
//               dS^T tile in shared memory
//   dq_full(b)  dQ^T of a step in buffer b: the drain reads it, the
//               step's dS^T tile (step % 2) may be written again, and so
//               may its Q / dO stage (every product that reads the stage
//               completed before it: S^T and dP^T before the threads' P and
//               dS, dV and dK before dQ^T in issue order)
//   dq_free(b)  the drain has read it: buffer b may take S^T again
// and once per step:
//   dp_full     dP^T of a step in tensor memory
//   dp_read     the threads have read it: the next step's dP^T may go there
// Every parity wait is safe by construction: the barrier's next completion
// after the awaited one needs an action that comes after the wait.
struct Sync {
  uint32_t kv_full, stage_full0, s_full0, dp_full, dp_read, sm_done0, dq_full0, dq_free0,
      acc_done, a_done;
  volatile int* abort_flag;
  __device__ __forceinline__ uint32_t stage_full(int b) const { return stage_full0 + 8 * b; }
  __device__ __forceinline__ uint32_t s_full(int b) const { return s_full0 + 8 * b; }
  __device__ __forceinline__ uint32_t sm_done(int b) const { return sm_done0 + 8 * b; }
  __device__ __forceinline__ uint32_t dq_full(int b) const { return dq_full0 + 8 * b; }
  __device__ __forceinline__ uint32_t dq_free(int b) const { return dq_free0 + 8 * b; }
};

// Step it's buffer and the parity of its buffer barriers' completion for it.
__device__ __forceinline__ int sbuf(int it) { return it % kSBufs; }
__device__ __forceinline__ uint32_t spar(int it) { return static_cast<uint32_t>(it / kSBufs) & 1u; }

// Bounded wait: true when the phase completed; false if this CTA is aborting
// or the wait ran past the limit (then the failure is recorded).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Sync& sy,
                                           const BwdParams& p, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t polls = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++polls & 31u) == 0u) {
      if (*sy.abort_flag) return false;
      if (global_timer_ns() - t0 > p.wait_limit_ns) {
        *sy.abort_flag = 1;
        atomicCAS(p.status, 0, site);
        return false;
      }
    }
  }
}

// dst += v in global memory, performed in L2 (no value returned).
__device__ __forceinline__ void red_add_f32(float* dst, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(dst), "f"(v) : "memory");
}

// ---------------------------------------------------------------------------
// TMA producer (one thread)
// ---------------------------------------------------------------------------
// K and V are read once per CTA (evict first); the Q and dO tiles of a head
// are read by all of its key blocks, so they are kept in L2 (evict last).
template <int D>
__device__ __forceinline__ void run_producer(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                             const CUtensorMap* tmV, const CUtensorMap* tmDO,
                                             uint32_t sbase, const Sync& sy, const BwdParams& p,
                                             int bh, int kb, int j0, int n) {
  using C = Cfg<D>;
  const uint64_t pol_kv = l2_policy_evict_first();
  const uint64_t pol_q = l2_policy_evict_last();
  mbar_arrive_expect_tx(sy.kv_full, 2 * C::kKTile);
#pragma unroll
  for (int s = 0; s < D / 64; ++s) {
    tma_load_3d_hint(sbase + C::kKOff + s * C::kKSlab, tmK, sy.kv_full, s * 64, kb * kBlockK, bh, pol_kv);
    tma_load_3d_hint(sbase + C::kVOff + s * C::kKSlab, tmV, sy.kv_full, s * 64, kb * kBlockK, bh, pol_kv);
  }
  auto prefetch_step = [&](int s) {
    const int q0 = (j0 + s) * kBlockQ;
#pragma unroll
    for (int x = 0; x < D / 64; ++x) {
      tma_prefetch_3d(tmQ, x * 64, q0, bh);
      tma_prefetch_3d(tmDO, x * 64, q0, bh);
    }
    const size_t row0 = static_cast<size_t>(bh) * p.Nq_pad + q0;
    prefetch_l2_bulk(p.lp + row0, kBlockQ * 4);
    prefetch_l2_bulk(p.dsum + row0, kBlockQ * 4);
  };
  for (int s = 0; s < kPrefetchSteps + C::kStages && s < n; ++s) prefetch_step(s);
  int it = 0;
  for (; it < n; ++it) {
    const int st = it % C::kStages;
    if (it + kPrefetchSteps + C::kStages < n) prefetch_step(it + kPrefetchSteps + C::kStages);
    // The stage was last read by step it - kStages: wait for its dQ^T.
    if (it >= C::kStages &&
        !wait_phase(sy.dq_full(sbuf(it - C::kStages)), spar(it - C::kStages), sy, p, kSiteProducer))
      break;
    const int q0 = (j0 + it) * kBlockQ;
    const uint32_t full = sy.stage_full(st);
    mbar_arrive_expect_tx(full, C::kStageBytes + C::kLdBytes);
    const uint32_t dst = sbase + C::kStageOff + st * C::kStageBytes;
#pragma unroll
    for (int s = 0; s < D / 64; ++s) {
      tma_load_3d_hint(dst + s * C::kQSlab, tmQ, full, s * 64, q0, bh, pol_q);
      tma_load_3d_hint(dst + C::kQTile + s * C::kQSlab, tmDO, full, s * 64, q0, bh, pol_q);
    }
    // L and D of the step's rows: 256 bytes each, 16-byte aligned because
    // the workspace rows are padded to a multiple of 64
    const size_t row0 = static_cast<size_t>(bh) * p.Nq_pad + q0;
    const uint32_t ld = sbase + C::kLdOff + st * C::kLdBytes;
    bulk_load(ld, p.lp + row0, kBlockQ * 4, full);
    bulk_load(ld + kBlockQ * 4, p.dsum + row0, kBlockQ * 4, full);
  }
  // Drain: every copy this thread started lands before the CTA exits.
  mbar_wait_bounded(sy.kv_full, 0, p.wait_limit_ns);
  for (int c = it > C::kStages ? it - C::kStages : 0; c < it; ++c)
    mbar_wait_bounded(sy.stage_full(c % C::kStages), (c / C::kStages) & 1, p.wait_limit_ns);
}

// ---------------------------------------------------------------------------
// MMA issuer (one warp; lane 0 issues)
// ---------------------------------------------------------------------------
// Operand descriptors.  K and V tiles: 64-column slabs of 128 rows (16 KB);
// Q and dO tiles: slabs of 64 rows (8 KB); dS^T: one slab of 128 rows.  All
// 128-byte swizzled; 8-row groups are 1024 bytes apart (the stride byte
// offset).  As a K-major operand a tile advances 32 bytes per 16 columns of
// d inside a slab; as an MN-major operand it advances 2048 bytes per 16 rows
// and its slabs (64 values of the N or M dimension each) are the leading
// byte offset apart.
// Stage and buffer b's descriptors are the first one's, moved by b times the
// stage (or buffer) size.
template <int D>
struct Desc {
  using C = Cfg<D>;
  uint64_t k_kmaj, v_kmaj, kt_mn, q_kmaj0, do_kmaj0, q_mn0, do_mn0, ds_mn0;
  __device__ __forceinline__ explicit Desc(uint32_t sbase) {
    k_kmaj = sdesc_sw128(sbase + C::kKOff, 16, 1024);
    v_kmaj = sdesc_sw128(sbase + C::kVOff, 16, 1024);
    kt_mn = sdesc_sw128(sbase + C::kKOff, C::kKSlab, 1024);
    const uint32_t st = sbase + C::kStageOff;
    q_kmaj0 = sdesc_sw128(st, 16, 1024);
    do_kmaj0 = sdesc_sw128(st + C::kQTile, 16, 1024);
    q_mn0 = sdesc_sw128(st, C::kQSlab, 1024);
    do_mn0 = sdesc_sw128(st + C::kQTile, C::kQSlab, 1024);
    const uint32_t ds = sbase + C::kDsOff;
    ds_mn0 = sdesc_sw128(ds, C::kDsBytes, 1024);  // N = 64: one slab, the leading offset is not used
  }
  __device__ __forceinline__ uint64_t ds_mn(int b) const { return sdesc_advance(ds_mn0, b * C::kDsBytes); }
  __device__ __forceinline__ uint64_t q_kmaj(int b) const { return sdesc_advance(q_kmaj0, b * C::kStageBytes); }
  __device__ __forceinline__ uint64_t do_kmaj(int b) const { return sdesc_advance(do_kmaj0, b * C::kStageBytes); }
  __device__ __forceinline__ uint64_t q_mn(int b) const { return sdesc_advance(q_mn0, b * C::kStageBytes); }
  __device__ __forceinline__ uint64_t do_mn(int b) const { return sdesc_advance(do_mn0, b * C::kStageBytes); }
};

// S^T = K Q^T and dP^T = V dO^T: A = the K or V tile (128 keys), B = the Q
// or dO tile (64 rows), both K-major over d in shared memory.
template <int D>
__device__ __forceinline__ void issue_kmaj(uint32_t d_tmem, uint64_t a, uint64_t b) {
  using C = Cfg<D>;
  constexpr uint32_t idesc = idesc_bf16_f32_ab(kBlockK, kBlockQ, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    umma_ss(d_tmem, sdesc_advance(a, (kk / 4) * C::kKSlab + (kk % 4) * 32),
            sdesc_advance(b, (kk / 4) * C::kQSlab + (kk % 4) * 32), idesc, kk > 0 ? 1u : 0u);
}

// Issuer A: S^T and dP^T, the threads' operands.  Order:
//   before the loop:  S^T(0)  dP^T(0)  S^T(1)  S^T(2)
//   step it:          [the threads have read dP^T(it)]          dP^T(it+1)
//                     [the drain has read dQ^T(it-1), buffer]   S^T(it+2) into it
template <int D>
__device__ __forceinline__ void run_mma_a(uint32_t sbase, uint32_t tmem, const Sync& sy, const BwdParams& p, int n) {
  using C = Cfg<D>;
  const bool leader = (threadIdx.x & 31) == 0;
  bool ok = true;
  auto wait_voted = [&](uint32_t bar, uint32_t par) {
    ok = __all_sync(0xffffffffu, ok && wait_phase(bar, par, sy, p, kSiteMma));
  };
  const Desc<D> ds(sbase);
  wait_voted(sy.kv_full, 0);
  auto issue_s_step = [&](int step) {  // S^T(step) into its buffer, once its stage is in
    wait_voted(sy.stage_full(step % C::kStages), (step / C::kStages) & 1);
    if (!ok) return;
    tc_fence_after_sync();
    if (leader) {
      issue_kmaj<D>(tmem + kColS + sbuf(step) * 64, ds.k_kmaj, ds.q_kmaj(step % C::kStages));
      umma_commit(sy.s_full(sbuf(step)));
    }
    __syncwarp();
  };
  auto issue_dp_step = [&](int step) {  // dP^T(step) (its stage is in: S^T(step) read it)
    tc_fence_after_sync();
    if (leader) {
      issue_kmaj<D>(tmem + kColDP, ds.v_kmaj, ds.do_kmaj(step % C::kStages));
      umma_commit(sy.dp_full);
    }
    __syncwarp();
  };
  if (n > 0) {
    issue_s_step(0);
    if (ok) issue_dp_step(0);
    for (int step = 1; step < kSBufs && step < n && ok; ++step) issue_s_step(step);
  }
  for (int it = 0; it < n && ok; ++it) {
    if (it + 1 < n) {
      wait_voted(sy.dp_read, it & 1);  // the threads have read dP^T(it)
      if (!ok) break;
      issue_dp_step(it + 1);
    }
    const int next = it + kSBufs - 1;  // the S^T that goes into step it-1's buffer
    if (it >= 1 && next < n) {
      wait_voted(sy.dq_free(sbuf(it - 1)), spar(it - 1));  // the drain has read dQ^T(it-1)
      if (!ok) break;
      issue_s_step(next);
    }
  }
  if (leader) umma_commit(sy.a_done);
  __syncwarp();
  mbar_wait_bounded(sy.a_done, 0, p.wait_limit_ns);
}

// Issuer B: the products of the threads' step it, once its P^T and dS^T are
// in: dV(it), dK(it), then dQ^T(it) into the same buffer (in issue order, so
// after dV and dK have read P^T and dS^T there).
template <int D, bool CAUSAL>
__device__ __forceinline__ void run_mma(uint32_t sbase, uint32_t tmem, const Sync& sy,
                                        const BwdParams& p, int n) {
  using C = Cfg<D>;
  const bool leader = (threadIdx.x & 31) == 0;
  bool ok = true;
  auto wait_voted = [&](uint32_t bar, uint32_t par) {
    ok = __all_sync(0xffffffffu, ok && wait_phase(bar, par, sy, p, kSiteMma));
  };
  const Desc<D> ds(sbase);
  const uint32_t tm_dv = tmem + kColDV, tm_dk = tmem + kColDK;
  constexpr uint32_t id_acc = idesc_bf16_f32_ab(kBlockK, D, false, true);      // dV, dK
  constexpr uint32_t id_dq = idesc_bf16_f32_ab(128, kBlockQ, true, true);      // dQ^T
  wait_voted(sy.kv_full, 0);
  for (int it = 0; it < n && ok; ++it) {
    const int st = it % C::kStages;
    const int b = sbuf(it);
    const uint32_t tm_s = tmem + kColS + b * 64;
    wait_voted(sy.sm_done(b), spar(it));  // P^T, dS^T of step it in
    if (!ok) break;
    tc_fence_after_sync();
    const uint32_t acc = it > 0 ? 1u : 0u;
    if (leader) {
#pragma unroll
      for (int kk = 0; kk < kBlockQ / 16; ++kk)  // dV += P^T dO
        umma_ts(tm_dv, tm_s + kk * 8, sdesc_advance(ds.do_mn(st), kk * 2048), id_acc, kk > 0 ? 1u : acc);
#pragma unroll
      for (int kk = 0; kk < kBlockQ / 16; ++kk)  // dK += dS^T Q
        umma_ts(tm_dk, tm_s + 32 + kk * 8, sdesc_advance(ds.q_mn(st), kk * 2048), id_acc, kk > 0 ? 1u : acc);
#pragma unroll
      for (int kk = 0; kk < kBlockK / 16; ++kk)  // dQ^T = K^T dS^T, over P^T and dS^T
        umma_ss(tm_s, sdesc_advance(ds.kt_mn, kk * 2048), sdesc_advance(ds.ds_mn(it & 1), kk * 2048), id_dq,
                kk > 0 ? 1u : 0u);
      umma_commit(sy.dq_full(b));
    }
    __syncwarp();
  }
  // Completes when every product issued above has: the epilogue's signal,
  // and the condition for releasing tensor memory.
  if (leader) umma_commit(sy.acc_done);
  __syncwarp();
  mbar_wait_bounded(sy.acc_done, 0, p.wait_limit_ns);
}

// mul * (an accumulator row of d fp32 values in tensor memory, from column
// address t) to key row `key` of dst [BH][Nk][D] in bf16, if key < Nk.  A
// block with no visible query row (causal, keys past the last query: n = 0)
// writes zeros.
template <int D>
__device__ __forceinline__ void store_acc_row(uint32_t t, __nv_bfloat16* dst, float mul, int bh, int key, int Nk,
                                              int n) {
  const bool store = key < Nk;
  uint4* out = reinterpret_cast<uint4*>(dst + (static_cast<size_t>(bh) * Nk + key) * D);
#pragma unroll
  for (int c0 = 0; c0 < D; c0 += 32) {
    uint32_t a[32];
    if (n > 0) {
      tmem_ld32_wait(t + c0, a);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = 0u;
    }
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      pk[i] = pack_bf16x2(__uint_as_float(a[2 * i]) * mul, __uint_as_float(a[2 * i + 1]) * mul);
    if (store) {
#pragma unroll
      for (int i = 0; i < 4; ++i) out[c0 / 8 + i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    }
  }
}

// ---------------------------------------------------------------------------
// P and dS (warps 4-7, one key row per thread), then the dV epilogue
// ---------------------------------------------------------------------------
template <int D, bool CAUSAL>
__device__ __forceinline__ void run_ds(uint8_t* smem, uint32_t tmem, const Sync& sy,
                                       const BwdParams& p, int bh, int kb, int j0, int n) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int quad = warp & 3;                 // TMEM lanes 32*quad .. 32*quad+31
  const int r = quad * 32 + lane;            // key row within the block
  const int key = kb * kBlockK + r;
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint64_t qk2 = f2_pack(p.qk_scale, p.qk_scale);
  bool ok = true;
  for (int it = 0; it < n && ok; ++it) {
    const int b = sbuf(it);
    const int st = it % C::kStages;
    const int q0 = (j0 + it) * kBlockQ;
    // The step's waits, those that have usually completed first: dQ^T(it-2)
    // (it last read the dS^T tile this step writes; the next completion of
    // its barrier, step it+1's, needs this step's dS), the stage (L and D of
    // the step), then S^T.  Testing a completed barrier right after a wait
    // that had to sleep took about 100 cycles more than testing it first
    // (timestamped runs); in this order the step took 2.5 % less time.
    bool w = it < 2 || wait_phase(sy.dq_full(sbuf(it - 2)), spar(it - 2), sy, p, kSiteDs);
    w = w && wait_phase(sy.stage_full(st), (it / C::kStages) & 1, sy, p, kSiteDs);
    w = w && wait_phase(sy.s_full(b), spar(it), sy, p, kSiteDs);
    ok = __all_sync(0xffffffffu, w);
    if (!ok) break;
    tc_fence_after_sync();
    const float* Lrow = reinterpret_cast<const float*>(smem + C::kLdOff + st * C::kLdBytes);
    const float* Drow = Lrow + kBlockQ;
    const uint32_t tS = tmem + lane_off + kColS + b * 64;

    // P^T row: p_c = exp2(s_c * scale * log2 e - L_c * log2 e) for query q0 + c.
    // Query rows past the end have L = +inf (p = 0).  Key `key` is visible to
    // query q0 + c iff key < Nk and (not causal or key <= q0 + c).
    float pf[kBlockQ];
    {
      uint32_t s[kBlockQ];
      tmem_ld64_wait(tS, s);
#pragma unroll
      for (int c = 0; c < kBlockQ; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(Lrow + c);
        const uint64_t x01 = f2_fma(f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), qk2,
                                    f2_pack(-l4.x, -l4.y));
        const uint64_t x23 = f2_fma(f2_pack(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])), qk2,
                                    f2_pack(-l4.z, -l4.w));
        float a0, a1, a2, a3;
        f2_unpack(x01, a0, a1);
        f2_unpack(x23, a2, a3);
        pf[c] = ex2_approx(a0);
        pf[c + 1] = ex2_approx(a1);
        pf[c + 2] = ex2_approx(a2);
        pf[c + 3] = ex2_approx(a3);
      }
    }
    const int cmin = key >= p.Nk ? kBlockQ : (CAUSAL ? key - q0 : 0);  // first visible column
    if (cmin > 0) {
#pragma unroll
      for (int c = 0; c < kBlockQ; ++c) pf[c] = c < cmin ? 0.f : pf[c];
    }
    {
      // P^T over the first 32 columns of S^T (all of which are in registers)
      uint32_t pk[kBlockQ / 2];
#pragma unroll
      for (int i = 0; i < kBlockQ / 2; ++i) pk[i] = pack_bf16x2(pf[2 * i], pf[2 * i + 1]);
      tmem_st32(tS, pk);
    }

    // dS^T row: ds_c = p_c * (dP_c - D_c), rounded to bf16, stored to tensor
    // memory after P^T (the A operand of dK) and to the 128-byte-swizzled dS^T
    // tile it % 2 in shared memory (the B operand of dQ^T; 16-byte chunk ch of
    // row r at chunk ch ^ (r % 8)).
    w = wait_phase(sy.dp_full, it & 1, sy, p, kSiteDs);
    ok = __all_sync(0xffffffffu, w);
    if (!ok) break;
    tc_fence_after_sync();
    uint32_t dpt[kBlockQ];
    tmem_ld64_wait(tmem + lane_off + kColDP, dpt);
    // dP^T is in registers: the next step's dP^T may take its columns
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(sy.dp_read);
    uint8_t* ds_row = smem + C::kDsOff + (it & 1) * C::kDsBytes + r * 128;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t wds[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c = h * 32 + 2 * i;
        const float2 dd = *reinterpret_cast<const float2*>(Drow + c);
        const float g0 = pf[c] * (__uint_as_float(dpt[c]) - dd.x);
        const float g1 = pf[c + 1] * (__uint_as_float(dpt[c + 1]) - dd.y);
        wds[i] = pack_bf16x2(g0, g1);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int ch = h * 4 + q;
        *reinterpret_cast<uint4*>(ds_row + ((ch ^ (r & 7)) * 16)) =
            make_uint4(wds[4 * q], wds[4 * q + 1], wds[4 * q + 2], wds[4 * q + 3]);
      }
      tmem_st16(tS + 32 + h * 16, wds);
    }
    tmem_st_wait();            // P^T and dS^T are in tensor memory
    fence_proxy_async_smem();  // dS^T is visible to the tensor core
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(sy.sm_done(b));
  }

  // Epilogue: dV of this thread's key row (the drain warps write dK).
  bool w = wait_phase(sy.acc_done, 0, sy, p, kSiteDs);
  ok = __all_sync(0xffffffffu, ok && w);
  if (!ok || *sy.abort_flag) return;
  tc_fence_after_sync();
  store_acc_row<D>(tmem + lane_off + kColDV, p.dv, 1.f, bh, key, p.Nk, n);
}

// ---------------------------------------------------------------------------
// dQ drain (warps 8-11): thread = one row of dQ^T (one column of d)
// ---------------------------------------------------------------------------
// Per step each thread writes its 64 values of dQ^T (one column of d, 64
// query rows) into the shared-memory tile in the accumulator's row layout (a
// warp's store covers 32 consecutive floats of one row), and one thread adds
// the tile's rows below Nq to the accumulator with one bulk reduction.  The
// tile is written again once that reduction has read it.  With d = 64 only
// warps 8 and 9 hold dQ^T rows.
constexpr uint32_t kDrainBar = 1;  // named barrier of the four drain warps

template <int D>
__device__ __forceinline__ void run_drain(uint8_t* smem, uint32_t tmem, const Sync& sy, const BwdParams& p, int bh,
                                          int kb, int j0, int n) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const bool has_rows = quad * 32 < D;
  const bool issuer = warp == kDrainWarp0 && lane == 0;
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  float* tile = reinterpret_cast<float*>(smem + C::kDqOff) + quad * 32 + lane;
  // Every drain warp runs all n steps and takes both named barriers of each,
  // whatever its waits returned, so the barriers never wait for a warp that
  // has left; after a failed wait (the CTA is aborting) a warp only skips the
  // work, and the reduction is not issued.
  bool ok = true;
  for (int it = 0; it < n; ++it) {
    const int b = sbuf(it);
    const bool w = __all_sync(0xffffffffu, ok && wait_phase(sy.dq_full(b), spar(it), sy, p, kSiteDrain));
    ok = w;
    uint32_t x[kBlockQ];
    if (w) {
      tc_fence_after_sync();
      tmem_ld64_wait(tmem + lane_off + kColS + b * 64, x);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(sy.dq_free(b));
    }
    if (issuer && it > 0) tma_store_wait_read0();  // the last reduction has read the tile
    named_bar_sync(kDrainBar, 128);
    if (w && has_rows) {
#pragma unroll
      for (int c = 0; c < kBlockQ; ++c) tile[c * D] = __uint_as_float(x[c]);
    }
    fence_proxy_async_smem();  // the tile is visible to the bulk reduction
    named_bar_sync(kDrainBar, 128);
    if (issuer && w && !*sy.abort_flag) {
      const int q0 = (j0 + it) * kBlockQ;
      const int rows = min(kBlockQ, p.Nq - q0);
      bulk_reduce_add_f32(p.dq_acc + (static_cast<size_t>(bh) * p.Nq + q0) * D, smem_u32(smem + C::kDqOff),
                          static_cast<uint32_t>(rows * D * 4));
      tma_store_commit();
    }
  }

  // Epilogue: scale * dK of key row quad * 32 + lane, while the last
  // reductions run.
  const bool w = wait_phase(sy.acc_done, 0, sy, p, kSiteDrain);
  if (__all_sync(0xffffffffu, ok && w) && !*sy.abort_flag) {
    tc_fence_after_sync();
    store_acc_row<D>(tmem + lane_off + kColDK, p.dk, p.scale, bh, kb * kBlockK + quad * 32 + lane, p.Nk, n);
  }
  // The tile must stay in place until every reduction has read it; the
  // adds themselves are complete when the kernel is.
  if (issuer) tma_store_wait_read0();
}

// ---------------------------------------------------------------------------
// Kernel: grid (key blocks, B*H) without the mask: the CTAs of one head are
// adjacent in launch order, so the ones running together share their heads'
// Q and dO tiles in L2.  Under the causal mask a key block's work falls with
// its index (block kb walks the query rows from kb * 128 on), so the grid is
// (B*H, key blocks): every head's first key block, the longest, is launched
// first and the shortest last, and the last wave holds short blocks only.
// ---------------------------------------------------------------------------
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const BwdParams p) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  if ((sbase & 1023u) != 0) {  // the whole CTA leaves before any barrier
    if (threadIdx.x == 0) atomicCAS(p.status, 0, kSiteAlign);
    return;
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kb = CAUSAL ? blockIdx.y : blockIdx.x;
  const int bh = CAUSAL ? blockIdx.x : blockIdx.y;
  // Query steps of this key block: under the top-left causal mask key j is
  // seen by queries i >= j, so the first step is the one holding query kb*128.
  const int j0 = CAUSAL ? (kb * kBlockK) / kBlockQ : 0;
  const int n = p.n_qt > j0 ? p.n_qt - j0 : 0;

  Sync sy;
  {
    uint32_t b = sbase + C::kBarOff;
    auto next = [&]() { const uint32_t r = b; b += 8; return r; };
    sy.kv_full = next();
    sy.stage_full0 = next();
    for (int i = 1; i < C::kStages; ++i) next();
    sy.s_full0 = next();
    for (int i = 1; i < kSBufs; ++i) next();
    sy.sm_done0 = next();
    for (int i = 1; i < kSBufs; ++i) next();
    sy.dq_full0 = next();
    for (int i = 1; i < kSBufs; ++i) next();
    sy.dq_free0 = next();
    for (int i = 1; i < kSBufs; ++i) next();
    sy.dp_full = next();
    sy.dp_read = next();
    sy.acc_done = next();
    sy.a_done = next();
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  sy.abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  if (threadIdx.x == 0) {
    mbar_init(sy.kv_full, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(sy.stage_full(i), 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(sy.s_full(i), 1);
      mbar_init(sy.sm_done(i), 4);  // one arrival per P / dS warp
      mbar_init(sy.dq_full(i), 1);
      mbar_init(sy.dq_free(i), 4);  // one arrival per drain warp
    }
    mbar_init(sy.dp_full, 1);
    mbar_init(sy.dp_read, 4);  // one arrival per P / dS warp
    mbar_init(sy.acc_done, 1);
    mbar_init(sy.a_done, 1);
    *sy.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kLoadWarp) {
    if (lane == 0) run_producer<D>(&tmQ, &tmK, &tmV, &tmDO, sbase, sy, p, bh, kb, j0, n);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    run_mma<D, CAUSAL>(sbase, tmem, sy, p, n);
  } else if (warp == kMmaWarpA) {
    run_mma_a<D>(sbase, tmem, sy, p, n);
  } else if (warp >= kDsWarp0 && warp < kDsWarp0 + 4) {
    run_ds<D, CAUSAL>(smem, tmem, sy, p, bh, kb, j0, n);
  } else if (warp >= kDrainWarp0) {
    run_drain<D>(smem, tmem, sy, p, bh, kb, j0, n);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Before: D = rowsum(dO * O) and L in log2 units per query row (padded to a
// multiple of 64 rows per head: L = +inf, D = 0), and the dQ accumulator
// zeroed.  One warp per row; the products of two bf16 values are exact in
// fp32 and summed in fp32.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256)
fa_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                   const float* __restrict__ lse, float* __restrict__ lp, float* __restrict__ dsum,
                   float* __restrict__ dq_acc, int BH, int Nq, int Nq_pad) {
  constexpr int kPer = D / 32;  // elements per lane
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long rows = static_cast<long long>(BH) * Nq_pad;
  for (long long row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += warps) {
    const int bh = static_cast<int>(row / Nq_pad);
    const int i = static_cast<int>(row % Nq_pad);
    float dot = 0.f;
    if (i < Nq) {
      const size_t base = (static_cast<size_t>(bh) * Nq + i) * D + lane * kPer;
      __nv_bfloat162 ov[kPer / 2], gv[kPer / 2];
      if constexpr (kPer == 4) {
        const uint2 a = *reinterpret_cast<const uint2*>(o + base);
        const uint2 g = *reinterpret_cast<const uint2*>(dout + base);
        ov[0] = *reinterpret_cast<const __nv_bfloat162*>(&a.x);
        ov[1] = *reinterpret_cast<const __nv_bfloat162*>(&a.y);
        gv[0] = *reinterpret_cast<const __nv_bfloat162*>(&g.x);
        gv[1] = *reinterpret_cast<const __nv_bfloat162*>(&g.y);
      } else {
        ov[0] = *reinterpret_cast<const __nv_bfloat162*>(o + base);
        gv[0] = *reinterpret_cast<const __nv_bfloat162*>(dout + base);
      }
#pragma unroll
      for (int e = 0; e < kPer / 2; ++e) {
        const float2 a = __bfloat1622float2(ov[e]);
        const float2 g = __bfloat1622float2(gv[e]);
        dot = fmaf(a.x, g.x, dot);
        dot = fmaf(a.y, g.y, dot);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      float* acc = dq_acc + (static_cast<size_t>(bh) * Nq + i) * D + lane * kPer;
      if constexpr (kPer == 4) {
        *reinterpret_cast<float4*>(acc) = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        *reinterpret_cast<float2*>(acc) = make_float2(0.f, 0.f);
      }
    }
    if (lane == 0) {
      lp[row] = i < Nq ? lse[static_cast<size_t>(bh) * Nq + i] * 1.4426950408889634f : INFINITY;
      dsum[row] = i < Nq ? dot : 0.f;
    }
  }
}

// After: dQ = bf16(scale * accumulator), eight values per thread.
__global__ void __launch_bounds__(256)
fa_bwd_dq_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq, long long n8,
                 float scale) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    reinterpret_cast<uint4*>(dq)[i] =
        make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                   pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
  }
}

}  // namespace bwd
}  // namespace fa
