// Fused exact attention forward for sm_103a: one persistent CTA per SM, each
// work item = two adjacent 128-row query tiles of one (batch, head), or, when
// every head has one tile, the tiles of two heads.
//
// The method is the FlashAttention-2 forward ("FlashAttention and kernels.",
// sections "From a sum to an output row" and "FlashAttention's forward pass";
// "Kernels and FlashAttention: When the Same Math Runs 7.6x Faster",
// section 2.8): query tiles outer, key/value tiles inner, running row maximum
// m, running row sum l and an unnormalised fp32 accumulator rescaled by
// alpha = exp(m_old - m_new), divided by l once at the end, plus the per-row
// logsumexp.  Exponentials are taken in base 2 with the softmax scale folded
// into one FMA, m kept in log2 units and L converted back with ln 2 ("How to
// profile and optimise kernels", Round 4, "exp2").  Key tiles above the
// diagonal are never visited; only the diagonal tile and a ragged last tile
// are masked (same article, Round 4, "Causal tile-skipping").
//
// GB300 mapping (warp specialisation, FlashAttention-3's idea of separate
// load and math warps carried over to tcgen05):
//   warps 0-3  softmax warpgroup for query tile 0 (one row per thread)
//   warps 4-7  softmax warpgroup for query tile 1
//   warp  8    TMA producer: Q tiles once per item, then K_j, V_j into a ring
//   warps 9-10 MMA issuers, one thread each, one per query tile, taking
//              turns: S_t = Q_t K_j^T and O_t += P_t V_j on the tensor core,
//              accumulators in tensor memory; warp 9 owns the TMEM allocation
//   warp  11   idle (it completes the third warpgroup, which setmaxnreg needs)
// Tensor memory (512 columns x 128 lanes, fp32): S_0 at column 0, S_1 at 128,
// O_0 at 256, O_1 at 384.  P_t (bf16, two per column) overwrites the first
// 64 columns of S_t and is the A operand of the P.V product.  While one
// warpgroup exponentiates, the tensor core works on the other query tile.
#pragma once

#include <cuda_bf16.h>

#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBlockM = 128;                 // query rows per tile
constexpr int kBlockN = 128;                 // keys per K/V tile
constexpr int kQTiles = 2;                   // query tiles per work item
constexpr int kItemRows = kBlockM * kQTiles; // query rows per work item
constexpr int kSlabBytes = 128 * 64 * 2;     // one 128-row x 64-column bf16 TMA box
constexpr int kNumThreads = 384;             // three warpgroups
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
// Register split: the launch gives every thread 168 (65536 / 384, rounded
// down to 8); the load/MMA warpgroup drops to 104 and the two softmax
// warpgroups rise to 192: 128*104 + 256*192 = 62464 <= 384*168.
constexpr uint32_t kRegsAux = 104;
constexpr uint32_t kRegsSoftmax = 192;
static_assert(128 * kRegsAux + 256 * kRegsSoftmax <= 384 * 168, "register split exceeds the launch");
constexpr uint32_t kTmemCols = 512;
// The reference maximum moves only when a tile's maximum exceeds it by more
// than this many log2 units, so exponentials stay <= 2^threshold.  With FP8
// operands P is rounded to e4m3 (largest finite value 448): 8, P <= 256.
// With bf16, P and the fp32 sums keep their relative precision at any
// magnitude, and 32 keeps them far from overflow (P <= 2^32; the row sum of
// at most 2^24 keys <= 2^56): a move, which costs the warp a second pass
// over the tile and a rescale of O, then needs a jump of the row maximum by
// a factor of 2^32 rather than 2^8.
template <int E>
constexpr float kRescaleThreshold = E == 1 ? 8.0f : 32.0f;

// Codes recorded in the device status word when a wait gives up.
constexpr int kSiteProducer = 1;
constexpr int kSiteMma = 2;
constexpr int kSiteSoftmax = 3;

// E is the operand size in bytes: 2 for bf16, 1 for the FP8 (e4m3) path.
// A slab is 128 rows of 128 bytes (64 bf16 or 128 e4m3 values), one TMA box.
template <int D, int E = 2>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dimension 64 or 128");
  static_assert(E == 2 || (E == 1 && D == 128), "the FP8 path takes d = 128");
  static constexpr int kSlabs = D * E / 128;                       // slabs per 128 x D tile
  static constexpr int kTileBytes = kSlabs * kSlabBytes;           // one 128 x D tile
  static constexpr int kStages = kTileBytes == 2 * kSlabBytes ? 5 : 9;  // K/V ring depth (tiles)
  static constexpr int kQkInstr = D * E / 32;                      // S = Q K^T: 32 bytes of K each
  static constexpr int kPvInstr = kBlockN * E / 32;                // O += P V: likewise
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQTiles * kTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
  // barriers: q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] p_ready[2]
  //           o_done[2] o_free[2] drain[1] turn[2]
  static constexpr int kNumBars = 2 * 2 + 2 * kStages + 2 * 4 + 1 + 2;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;           // tmem slot, abort flag
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;           // + alignment slack
};

// Work distribution.  The forward's work is a list of items (256 query rows
// of one batch*head), each made of steps (one 128-key tile visited by both
// query tiles).  Every CTA gets a contiguous range of the concatenated steps
// of equal length, so all SMs finish together.  A range boundary may fall
// inside an item: each side then covers part of the item's keys and writes a
// normalised partial result (O over its keys, and that part's logsumexp) to a
// workspace slot.  The CTA whose arrival completes an item's parts merges
// them through their logsumexps once its own work is done (the merge of
// partial states over key ranges that Flash-Decoding uses, "FlashAttention
// and kernels."); no CTA ever waits for another.
constexpr int kMaxCtas = 256;

struct WorkRange {
  int item_begin;  // first item touched
  int step_begin;  // first step within it
  int item_last;   // last item touched (item_last < item_begin: empty range)
  int step_end;    // one past the last step within item_last
};

struct SlotPair {
  int first;    // workspace slot of the first chunk when it is a part of an item, else -1
  int last;     // the same for the last chunk (when it differs from the first)
  int k_first;  // the split item (index into the merge lists) of the first chunk
  int k_last;   // ... and of the last chunk
};

struct FwdParams {
  __nv_bfloat16* o;        // [BH][N][D]
  float* lse;              // [BH][N]
  int* status;             // device status word (0 = ok)
  float* part_o;           // workspace: [slot][256][D] fp32, O of a part, normalised within it
  float* part_lse;         // workspace: [slot][256] fp32, the part's natural-log logsumexp
  int Nq;                  // query rows (of O and LSE)
  int Nk;                  // keys (of K and V)
  int BH;                  // heads the items run over: B*H, or B*H / 2 when the items pair heads
  int n_key_tiles;         // ceil(N / 128)
  int n_row_blocks;        // ceil(N / 256)
  int num_items;           // BH * n_row_blocks
  float qk_scale;          // scale * log2(e)
  unsigned long long wait_limit_ns;
  int starve_kv;           // watchdog self-test: the producer never delivers K/V
  const float* q_scale;    // FP8 path: [BH][ceil(Nq / 128)], one per 128 query rows
  const float* k_scale;    // FP8 path: [BH][ceil(Nk / 128)], one per 128 keys
  const float* v_scale;    // FP8 path: [BH], one per head
  int* counters;           // workspace: per (split item, query tile, warp quadrant) part arrivals (0 between launches)
  WorkRange range[kMaxCtas];
  SlotPair slots[kMaxCtas];
  int merge_item[kMaxCtas];       // per split item: the item
  int merge_first[kMaxCtas];      // ... its first entry in merge_slots
  int merge_count[kMaxCtas];      // ... its number of parts
  int merge_slots[2 * kMaxCtas];  // the parts' workspace slots, item after item
};

// Work item -> (row block, batch*head).  Row blocks are taken in pairs (the
// last and the first, then the second-last and the second, ...) and the two
// blocks of a pair alternate item by item, heads varying slowest within the
// pair.  Under the causal mask a late row block visits many key tiles and an
// early one few, so any contiguous run of items mixes long and short ones and
// every CTA's range holds about the same number of items.  (The pages order
// the longest tiles first, "How to profile and optimise kernels", Round 5;
// with ranges of equal work the mix matters more than the order.)
__host__ __device__ __forceinline__ void decode_item_shape(int item, int BH, int nrb, int& rb,
                                                           int& bh) {
  const int npairs = nrb / 2;
  const int paired = 2 * BH * npairs;
  if (item < paired) {
    const int pair = item / (2 * BH);
    const int r = item % (2 * BH);
    bh = r / 2;
    rb = (r & 1) ? pair : nrb - 1 - pair;
  } else {  // the middle row block of an odd count
    rb = npairs;
    bh = item - paired;
  }
}

__device__ __forceinline__ void decode_item(int item, const FwdParams& p, int& rb, int& bh) {
  decode_item_shape(item, p.BH, p.n_row_blocks, rb, bh);
}

// The head and first query row of query tile t of item (rb, bh).  An item
// is normally two adjacent 128-row tiles of one head; with at most 128 query
// rows (one tile per head) it pairs two heads instead, so that both query
// tiles, and both softmax warpgroups, have work: each tile then streams its
// own head's K and V.
__host__ __device__ __forceinline__ int tile_head(int bh, int t, int paired) { return paired ? 2 * bh + t : bh; }
__host__ __device__ __forceinline__ int tile_row0(int rb, int t, int paired) {
  return paired ? 0 : rb * kItemRows + t * kBlockM;
}

// Number of key tiles query tile t of row block rb visits (0 if the tile
// lies beyond the last query row).  Causal is the top-left mask: key j for
// query i iff j <= i, so rows past the last key see every key tile.
template <bool CAUSAL, bool PAIRED>
__device__ __forceinline__ int tiles_for(int rb, int t, const FwdParams& p) {
  const int r0 = tile_row0(rb, t, PAIRED);
  if (r0 >= p.Nq) return 0;
  if (CAUSAL) return min(r0 / kBlockN + 1, p.n_key_tiles);
  return p.n_key_tiles;
}

// Steps of an item: the key tiles its longer query tile visits.
template <bool CAUSAL, bool PAIRED>
__device__ __forceinline__ int item_steps(int rb, const FwdParams& p) {
  return max(tiles_for<CAUSAL, PAIRED>(rb, 0, p), tiles_for<CAUSAL, PAIRED>(rb, 1, p));
}

// One chunk of this CTA's range: key tiles [kb, ke) of one item.
struct Chunk {
  int rb, bh;
  int kb, ke;
  int slot;   // workspace slot when the chunk is only a part of its item, else -1
  int k;      // its split item, when slot >= 0
  int todo;   // 0 for the CTA's first chunk, 1 otherwise
  bool last;  // the CTA's last chunk
};

__device__ __forceinline__ int num_chunks(const WorkRange& wr) {
  return wr.item_last >= wr.item_begin ? wr.item_last - wr.item_begin + 1 : 0;
}

__device__ __forceinline__ int chunk_item(int q, const WorkRange& wr) { return wr.item_begin + q; }

__device__ __forceinline__ Chunk chunk_of(int item, int nkv, const WorkRange& wr,
                                          const SlotPair& sp, const FwdParams& p) {
  Chunk c;
  decode_item(item, p, c.rb, c.bh);
  c.kb = item == wr.item_begin ? wr.step_begin : 0;
  c.ke = item == wr.item_last ? wr.step_end : nkv;
  const bool part = c.kb > 0 || c.ke < nkv;
  c.slot = !part ? -1 : (item == wr.item_begin ? sp.first : sp.last);
  c.k = item == wr.item_begin ? sp.k_first : sp.k_last;
  c.todo = item == wr.item_begin ? 0 : 1;
  c.last = item == wr.item_last;
  return c;
}

struct Sync {
  uint32_t q_full[2], q_empty[2], s_full[2], p_ready[2], o_done[2], o_free[2], drain;
  uint32_t turn[2];              // hand-over between the two MMA issuers
  uint32_t kv_full0, kv_empty0;  // arrays of kStages barriers, 8 bytes apart
  volatile int* abort_flag;
};

// Bounded wait: true when the phase completed; false if this CTA is aborting
// or the wait ran past the limit (then the failure is recorded).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Sync& sy,
                                           const FwdParams& p, int site) {
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

// ---------------------------------------------------------------------------
// TMA producer (one thread)
// ---------------------------------------------------------------------------
template <int D, bool CAUSAL, int E = 2, bool PAIRED = false>
__device__ __forceinline__ void run_producer(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                             uint32_t sbase, const Sync& sy, const FwdParams& p) {
  using C = Cfg<D, E>;
  uint32_t q_loads[2] = {0, 0};
  uint32_t kv_count = 0;
  const uint64_t pol_q = l2_policy_evict_first();
  const uint64_t pol_kv = l2_policy_evict_last();
  bool ok = true;
  const WorkRange wr = p.range[blockIdx.x];
  const SlotPair sp = p.slots[blockIdx.x];
  for (int q = 0, nq = num_chunks(wr); q < nq && ok; ++q) {
    const int item = chunk_item(q, wr);
    int rb, bh;
    decode_item(item, p, rb, bh);
    const int nkv = item_steps<CAUSAL, PAIRED>(rb, p);
    const Chunk ch = chunk_of(item, nkv, wr, sp, p);
    if (ch.slot >= 0 && ch.last) {
      // The CTA's last chunk is a part of a split item: its warps will most
      // likely merge the item when the chunk ends, and the other parts were
      // published long ago, when their CTAs started.  Bring them back into
      // L2 while the chunk runs.
      const int first = p.merge_first[ch.k], count = p.merge_count[ch.k];
      for (int i = 0; i < count; ++i) {
        const int slot = p.merge_slots[first + i];
        if (slot == ch.slot) continue;
        prefetch_l2_bulk(p.part_o + static_cast<size_t>(slot) * kItemRows * D, kItemRows * D * 4);
        prefetch_l2_bulk(p.part_lse + static_cast<size_t>(slot) * kItemRows, kItemRows * 4);
      }
    }
    for (int t = 0; t < kQTiles && ok; ++t) {
      if (min(ch.ke, tiles_for<CAUSAL, PAIRED>(rb, t, p)) <= ch.kb) continue;  // no tile of its own here
      ok = wait_phase(sy.q_empty[t], (q_loads[t] & 1u) ^ 1u, sy, p, kSiteProducer);
      if (!ok) break;
      ++q_loads[t];
      mbar_arrive_expect_tx(sy.q_full[t], C::kTileBytes);
      const uint32_t dst = sbase + C::kQOff + t * C::kTileBytes;
      const int row = tile_row0(rb, t, PAIRED);
      const int head = tile_head(bh, t, PAIRED);
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s)
        tma_load_3d_hint(dst + s * kSlabBytes, tmQ, sy.q_full[t], s * (128 / E), row, head, pol_q);
    }
    if (p.starve_kv) continue;  // self-test: never deliver K/V
    // per step: K then V (normal), or K of both heads then V of both (paired)
    const int heads = PAIRED ? 2 : 1;
    for (int j = ch.kb; j < ch.ke && ok; ++j) {
#pragma unroll
      for (int n = 0; n < 2 * heads; ++n) {
        if (!ok) break;
        const int which = n / heads;
        const int head = PAIRED ? 2 * bh + n % heads : bh;
        const uint32_t slot = kv_count % C::kStages;
        const uint32_t par = ((kv_count / C::kStages) & 1u) ^ 1u;
        ok = wait_phase(sy.kv_empty0 + 8 * slot, par, sy, p, kSiteProducer);
        if (!ok) break;
        const uint32_t full = sy.kv_full0 + 8 * slot;
        mbar_arrive_expect_tx(full, C::kTileBytes);
        const uint32_t dst = sbase + C::kKVOff + slot * C::kTileBytes;
        const CUtensorMap* map = which == 0 ? tmK : tmV;
        if (E == 1 && which == 1) {
          // the FP8 path's V is stored transposed, [BH][D][keys]: the tile is
          // D rows of 128 keys
          tma_load_3d_hint(dst, map, full, j * kBlockN, 0, head, pol_kv);
        } else {
#pragma unroll
          for (int s = 0; s < C::kSlabs; ++s)
            tma_load_3d_hint(dst + s * kSlabBytes, map, full, s * (128 / E), j * kBlockN, head, pol_kv);
        }
        ++kv_count;
      }
    }
  }
  // Drain: wait until every copy this thread started has landed, so none is
  // still writing shared memory when the CTA exits (also after an abort).
  // These waits ignore the abort flag: copies in flight land whatever happened.
  const uint32_t first = kv_count > (uint32_t)C::kStages ? kv_count - C::kStages : 0;
  for (uint32_t c = first; c < kv_count; ++c)
    mbar_wait_bounded(sy.kv_full0 + 8 * (c % C::kStages), (c / C::kStages) & 1u, p.wait_limit_ns);
  for (int t = 0; t < kQTiles; ++t)
    if (q_loads[t] > 0) mbar_wait_bounded(sy.q_full[t], (q_loads[t] - 1) & 1u, p.wait_limit_ns);
}

// ---------------------------------------------------------------------------
// MMA issuer (one thread)
// ---------------------------------------------------------------------------
// S = Q K^T: 16 columns of d per instruction, 4 instructions per 64-column
// swizzled slab.  q_desc and k_desc describe the first slab of each tile;
// every other operand address is a constant offset from them.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tmem_s, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBlockM, kBlockN, /*b_mn_major=*/false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk / 4) * kSlabBytes + (kk % 4) * 32;
    umma_ss(tmem_s, sdesc_advance(q_desc, off), sdesc_advance(k_desc, off), idesc, kk > 0 ? 1u : 0u);
  }
}

// O += P V: V is [keys][d] with d contiguous, an MN-major B operand.  16 keys
// per instruction = two 8-row swizzle groups (2048 bytes); the 64-column
// slabs of d are 16 KB apart (the descriptor's leading byte offset).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t v_desc,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBlockM, D, /*b_mn_major=*/true);
  umma_ts(tmem_o, tmem_p, v_desc, idesc, accumulate ? 1u : 0u);
#pragma unroll
  for (int kk = 1; kk < kBlockN / 16; ++kk)
    umma_ts(tmem_o, tmem_p + kk * 8, sdesc_advance(v_desc, kk * 2048), idesc, 1u);
}

// MMA issue is split between two threads, one per query tile, that take
// strict turns.  A tcgen05.mma returns to its issuer roughly when the tensor
// core accepts the next instruction, so a single issuer would leave the tensor
// core idle while it checks barriers between groups.  Here the thread whose
// turn it is feeds its group (O_t += P_t V_{j-1}, then S_t = Q_t K_j^T) while
// the other thread has already done its waits and only needs the hand-over.
// The tensor core therefore sees the same order as one issuer would produce:
// tile 0's group, tile 1's group, tile 0's next group, ...  Each tile's
// instructions stay in one thread, in issue order, so P_t(j-1) is read before
// S_t(j) overwrites the same tensor-memory columns.
template <int D, bool CAUSAL, int E = 2, bool PAIRED = false>
__device__ __forceinline__ void run_mma(int t, uint32_t sbase, uint32_t tmem, const Sync& sy,
                                        const FwdParams& p) {
  using C = Cfg<D, E>;
  const uint32_t bar_q_full = t ? sy.q_full[1] : sy.q_full[0];
  const uint32_t bar_q_empty = t ? sy.q_empty[1] : sy.q_empty[0];
  const uint32_t bar_s_full = t ? sy.s_full[1] : sy.s_full[0];
  const uint32_t bar_p_ready = t ? sy.p_ready[1] : sy.p_ready[0];
  const uint32_t bar_o_done = t ? sy.o_done[1] : sy.o_done[0];
  const uint32_t bar_o_free = t ? sy.o_free[1] : sy.o_free[0];
  const uint32_t my_turn = t ? sy.turn[1] : sy.turn[0];
  const uint32_t next_turn = t ? sy.turn[0] : sy.turn[1];
  // Descriptors are built once; per tile and per instruction they only move by
  // constant offsets (the tensor core consumes one N=128 instruction every 64
  // cycles, faster than a descriptor can be assembled from scratch).
  const uint64_t q_desc = sdesc_advance(sdesc_sw128(sbase + C::kQOff, 16, 1024), t * C::kTileBytes);
  const uint64_t k_desc0 = sdesc_sw128(sbase + C::kKVOff, 16, 1024);
  // bf16: V [keys][d], an MN-major operand, slabs of d 16 KB apart; FP8:
  // V^T [d][keys], a K-major operand like K
  const uint64_t v_desc0 =
      E == 2 ? sdesc_sw128(sbase + C::kKVOff, kSlabBytes, 1024) : sdesc_sw128(sbase + C::kKVOff, 16, 1024);
  const uint32_t tm_s = tmem + t * 128;
  const uint32_t tm_o = tmem + 256 + t * 128;
  uint32_t q_uses = 0, kv_count = 0, pr_par = 0, of_par = 1, turn_par = 0;
  bool ok = true;
  auto full = [&](uint32_t c) { return sy.kv_full0 + 8 * (c % C::kStages); };
  auto empty = [&](uint32_t c) { return sy.kv_empty0 + 8 * (c % C::kStages); };
  // The whole warp runs this loop, so that everything but the MMA
  // instructions themselves is warp-uniform (descriptors live in uniform
  // registers); every wait is voted so the warp stays converged, and one
  // lane issues the MMAs, commits and arrivals.
  const bool leader = (threadIdx.x & 31) == 0;
  auto wait_voted = [&](uint32_t bar, uint32_t par) {
    ok = __all_sync(0xffffffffu, ok && wait_phase(bar, par, sy, p, kSiteMma));
  };
  auto wait_full = [&](uint32_t c) { wait_voted(full(c), (c / C::kStages) & 1u); };
  // A K/V slot is released twice: once per query tile normally, and both
  // times by its one user when the item pairs two heads.
  const int rel = PAIRED ? 2 : 1;
  auto release_unused = [&](uint32_t c) {  // a K/V tile this query tile skips
    wait_full(c);                          // its previous phase is then complete
    if (ok && leader)
      for (int i = 0; i < rel; ++i) mbar_arrive(empty(c));
  };
  if (t == 1 && leader) mbar_arrive(sy.turn[0]);  // tile 0 takes the first turn

  const WorkRange wr = p.range[blockIdx.x];
  const SlotPair sp = p.slots[blockIdx.x];
  for (int q = 0, nq = num_chunks(wr); q < nq && ok; ++q) {
    const int item = chunk_item(q, wr);
    int rb0, bh0;
    decode_item(item, p, rb0, bh0);
    const int nkv_item = item_steps<CAUSAL, PAIRED>(rb0, p);
    const Chunk ch = chunk_of(item, nkv_item, wr, sp, p);
    // this query tile's key tiles inside the chunk: [kb, ne)
    const int kb = ch.kb;
    const int ne = min(ch.ke, tiles_for<CAUSAL, PAIRED>(ch.rb, t, p));
    const int n_steps = ch.ke - kb;  // both issuers walk the same steps
    const uint32_t kvps = PAIRED ? 4u : 2u;   // K/V slots per step
    const uint32_t koff = PAIRED ? t : 0u;    // this tile's K among them
    const uint32_t voff = PAIRED ? 2u + t : 1u;  // and its V
    if (ne > kb) {
      wait_voted(bar_q_full, q_uses & 1u);
      ++q_uses;
    }
    // step s issues O_t += P_t(s-1) V_{s-1} (if kb <= s-1 < ne) and S_t(s) (if s < ne)
    for (int s = kb; s <= ch.ke && ok; ++s) {
      const bool do_pv = s - 1 >= kb && s - 1 < ne;
      const bool do_s = s < ne;
      // slots per step: K, V (normal) or K of both heads, V of both (paired)
      const uint32_t cv = kv_count + kvps * (s - 1 - kb) + voff;  // V_{s-1}
      const uint32_t ck = kv_count + kvps * (s - kb) + koff;      // K_s
      // K/V (landed long before, as a rule) first, then the descriptors, and
      // the softmax's P last: once P is in, only the turn stands between it
      // and the products.  A full barrier's wait is by parity: it tells fill
      // n of a slot from fill n-1 only, so the waiter must know that fill n-1
      // is complete.  Without pairing both issuers wait for every position of
      // the ring, in order, which guarantees it.  With pairing a slot's
      // consecutive fills go to different tiles' K and V, and the fill before
      // this issuer's was waited for by the other issuer in its previous
      // group: this issuer waits for its K/V only once it has the turn, that
      // is once that group is issued (before, it could take the earlier fill,
      // still being loaded, for its own).
      if (!PAIRED && do_pv) wait_full(cv);
      if (!PAIRED && do_s) wait_full(ck);
      uint64_t dv[C::kPvInstr], dq[C::kQkInstr], dk[C::kQkInstr];
      {
        const uint64_t v0 = sdesc_advance(v_desc0, (cv % C::kStages) * C::kTileBytes);
        const uint64_t k0 = sdesc_advance(k_desc0, (ck % C::kStages) * C::kTileBytes);
        // P.V: bf16 takes 16 keys (two 8-row groups, 2048 bytes) of the
        // MN-major V per instruction, FP8 32 keys (32 bytes) of the K-major V^T
#pragma unroll
        for (int kk = 0; kk < C::kPvInstr; ++kk) dv[kk] = sdesc_advance(v0, E == 2 ? kk * 2048 : kk * 32);
#pragma unroll
        for (int kk = 0; kk < C::kQkInstr; ++kk) {
          const uint32_t off = (kk / 4) * kSlabBytes + (kk % 4) * 32;
          dq[kk] = sdesc_advance(q_desc, off);
          dk[kk] = sdesc_advance(k0, off);
        }
      }
      const uint32_t acc0 = s > kb + 1 ? 1u : 0u;
      if (do_pv) {
        if (s == kb + 1) {
          wait_voted(bar_o_free, of_par);
          of_par ^= 1u;
        }
        wait_voted(bar_p_ready, pr_par);
        pr_par ^= 1u;
      }
      // Every operand of the group is computed before the turn is taken, so
      // that the turn holds only the MMA instructions themselves.
      wait_voted(my_turn, turn_par);
      turn_par ^= 1u;
      if (PAIRED && do_pv) wait_full(cv);
      if (PAIRED && do_s) wait_full(ck);
      if (!ok) break;
      tc_fence_after_sync();
      if (leader) {
      // A = P from tensor memory: 8 columns per instruction either way (16
      // bf16 or 32 e4m3 values of each row)
      if (do_pv) {
        if constexpr (E == 2) {
          constexpr uint32_t idesc_pv = idesc_bf16_f32(kBlockM, D, /*b_mn_major=*/true);
#pragma unroll
          for (int kk = 0; kk < C::kPvInstr; ++kk) umma_ts(tm_o, tm_s + kk * 8, dv[kk], idesc_pv, kk > 0 ? 1u : acc0);
        } else {
          constexpr uint32_t idesc_pv = idesc_e4m3_f32(kBlockM, D, /*b_mn_major=*/false);
#pragma unroll
          for (int kk = 0; kk < C::kPvInstr; ++kk)
            umma_ts_f8(tm_o, tm_s + kk * 8, dv[kk], idesc_pv, kk > 0 ? 1u : acc0);
        }
      }
      if (do_s) {
        if constexpr (E == 2) {
          constexpr uint32_t idesc_qk = idesc_bf16_f32(kBlockM, kBlockN, /*b_mn_major=*/false);
#pragma unroll
          for (int kk = 0; kk < C::kQkInstr; ++kk) umma_ss(tm_s, dq[kk], dk[kk], idesc_qk, kk > 0 ? 1u : 0u);
        } else {
          constexpr uint32_t idesc_qk = idesc_e4m3_f32(kBlockM, kBlockN, /*b_mn_major=*/false);
#pragma unroll
          for (int kk = 0; kk < C::kQkInstr; ++kk) umma_ss_f8(tm_s, dq[kk], dk[kk], idesc_qk, kk > 0 ? 1u : 0u);
        }
      }
      // The turn goes to the other issuer as soon as the last product is
      // issued: the tensor core holds about one instruction beyond the one it
      // runs, so the other issuer's wake-up has to overlap the end of this
      // group (handing over after the commits measured 2 % slower).  The
      // commits come after both products so that the two run back to back.
      // A group has as few as it can: S_t's completion also tells the softmax
      // that the P.V of the same group is done (what a rescale of O needs),
      // and o_done is committed only by the chunk's last group, the P.V
      // alone, for the epilogue.
      mbar_arrive(next_turn);
      if (do_s) umma_commit(bar_s_full);
      if (do_pv && !do_s) umma_commit(bar_o_done);
      if (do_s && s == ne - 1) umma_commit(bar_q_empty);
      for (int i = 0; i < rel; ++i) {
        if (do_pv) umma_commit(empty(cv));
        if (do_s) umma_commit(empty(ck));
      }
      }
      __syncwarp();
      if (!do_pv && s - 1 >= kb) release_unused(cv);
      if (!do_s && s < ch.ke) release_unused(ck);
    }
    kv_count += kvps * n_steps;
  }
  // Every MMA this thread issued must finish before tensor memory is released.
  if (leader) umma_commit(sy.drain);
  __syncwarp();
  mbar_wait_bounded(sy.drain, 0, p.wait_limit_ns);
}

constexpr int kMaxPartsPerItem = 8;  // the plan splits no item into more parts

// Workspace slot layout: a slot holds one part of an item, 256 rows of D
// fp32 values, stored as D / 8 groups of eight columns, each group with its
// 256 rows one after the other (32 bytes a row).  A thread owns a row (as in
// tensor memory), so a warp's 32-byte access to one group covers 1 KB of
// consecutive memory instead of 32 rows' separate sectors.
template <int D>
__device__ __forceinline__ size_t part_index(int slot, int row_in_item, int group) {
  return (static_cast<size_t>(slot) * kItemRows * D) + (static_cast<size_t>(group) * kItemRows + row_in_item) * 8;
}

// A warp publishes its 32 rows of one part of a split item: O normalised over
// the part's keys (the accumulator scaled by inv_l) in fp32, and the part's
// natural-log logsumexp.  An empty part (no key of the chunk lies at or below
// the tile's rows) publishes L = -inf only; the merge gives it weight 0 and
// never reads its O.
template <int D>
__device__ __forceinline__ void publish_part(const Chunk& ch, int t, int row_in_tile, uint32_t tO,
                                             float inv_l, float lse_part, bool empty,
                                             const FwdParams& p) {
  const size_t prow = static_cast<size_t>(ch.slot) * kItemRows + t * kBlockM + row_in_tile;
  const int r = t * kBlockM + row_in_tile;
  if (!empty) {
    const uint64_t il2 = f2_pack(inv_l, inv_l);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32_wait(tO + c * 32, o);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float a, b;
        f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il2), a, b);
        o[2 * i] = __float_as_uint(a);
        o[2 * i + 1] = __float_as_uint(b);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) st_global_v8(p.part_o + part_index<D>(ch.slot, r, c * 4 + i), o + i * 8);
    }
  }
  p.part_lse[prow] = lse_part;
}

constexpr int kCountersPerItem = 2 * 4;                // per query tile and warp quadrant
constexpr int kNumCounters = kMaxCtas * kCountersPerItem;  // workspace counters (split items <= CTAs)

// The parts of a split item meet through one counter per (item, query tile,
// warp quadrant): the warps holding the same 32 rows in each part count
// their arrivals there.  The warp whose arrival completes the parts merges
// those 32 rows when its CTA's own work is done, reading its own part from
// tensor memory when it is still there (the CTA's last chunk: nothing later
// overwrites that O), and the other parts from the workspace.  In the last
// chunk every lane of a warp first reads the counter: if every other part is
// already in, the warp is the last and publishes nothing.  A part in the
// CTA's first chunk (its range starts inside an item) is published with
// plain stores and its arrival is deferred: the warp makes it (a fence, then
// the increment) at the start of its next chunk, while that chunk's first
// scores are on their way, and looks at the increment's old value, which
// says whether it merges, only after the last chunk.  No warp ever waits for
// another CTA; the merging warp resets the counter for the next launch.
struct PartSlots {
  int n;                       // parts of the item
  int slot[kMaxPartsPerItem];  // their workspace slots
};

constexpr int kInTmem = 1;    // this warp's part is still in tensor memory
constexpr int kOwnEmpty = 2;  // this warp's part has no key for these rows (L = -inf, no O)
constexpr int kAcquired = 4;  // every lane has read the counter with acquire and seen all other parts in

struct PendingMerge {
  int k;          // split item, or -1 for none
  int own_slot;   // this warp's part's workspace slot (read from there unless in TMEM)
  int flags;      // kInTmem | kOwnEmpty | kAcquired
  float inv_l;    // 1 / lq of the own part (the accumulator -> normalised O)
  float lse_own;  // natural-log logsumexp of the own part
  int rb, bh;
};

// The warp's arrival on a part counter, once its part's rows are stored:
// returns the counter's old value in lane 0 (0 in the other lanes).
__device__ __forceinline__ int part_arrive(int* ctr, int lane) {
  __threadfence();
  __syncwarp();
  int old = 0;
  if (lane == 0) old = atomicAdd(ctr, 1);
  return old;
}

// End of a chunk that is a part of its item.  Sets `arrival` to -1 when the
// part is stored and its arrival is left to the caller (the CTA's first chunk).
template <int D>
__device__ __forceinline__ PendingMerge part_done(const Chunk& ch, int t, int quad, int lane,
                                                  int row_in_tile, uint32_t tO, float inv_l,
                                                  float lse_part, bool empty, int& arrival, const FwdParams& p) {
  int* ctr = p.counters + ch.k * kCountersPerItem + t * 4 + quad;
  const int count = p.merge_count[ch.k];
  PendingMerge pm{-1, ch.slot, (ch.last ? kInTmem : 0) | (empty ? kOwnEmpty : 0), inv_l, lse_part, ch.rb, ch.bh};
  if (ch.last) {
    // every lane acquires: the other parts' rows were stored and fenced before
    // their arrivals were counted
    if (__all_sync(0xffffffffu, ld_acquire_gpu(ctr) == count - 1)) {  // merge, publish nothing
      pm.k = ch.k;
      pm.flags |= kAcquired;
      return pm;
    }
  }
  publish_part<D>(ch, t, row_in_tile, tO, inv_l, lse_part, empty, p);
  if (!ch.last) {  // the arrival is left to the caller
    pm.k = ch.k;
    arrival = -1;
    return pm;
  }
  if (__shfl_sync(0xffffffffu, part_arrive(ctr, lane), 0) == count - 1) pm.k = ch.k;  // arrived last after all
  return pm;
}

// Merges one warp's 32 rows (thread = row, as in tensor memory) of a split
// item: L = ln sum_r exp(L_r), O = sum_r exp(L_r - L) O_r, the largest L_r
// subtracted first; parts with L_r = -inf weigh 0 and their O is not used.
// The own part comes from tensor memory or its slot, the others from their
// slots.  With two parts (the usual case) the other part's logsumexp and its
// first 32 columns are loaded together, and each next 32 columns while the
// current ones are combined; with more parts each part's 32 columns are
// loaded in turn.  Writes the final bf16 O and L of rows < Nq.
template <int D>
__device__ __forceinline__ void merge_rows(const PendingMerge pm, const PartSlots ps, int t, int quad,
                                        uint32_t tO, int* ctr, __nv_bfloat16* __restrict__ o,
                                        float* __restrict__ lse, const float* __restrict__ part_o,
                                        const float* __restrict__ part_lse, int Nq, int paired) {
  const int lane = threadIdx.x & 31;
  const int r = t * kBlockM + quad * 32 + lane;  // row within the item (and its slot)
  const int row = tile_row0(pm.rb, t, paired) + quad * 32 + lane;
  const int head = tile_head(pm.bh, t, paired);
  // Every lane acquires the counter itself (unless it already did), then it
  // is reset for the next launch: every arrival for these rows has happened.
  if (!(pm.flags & kAcquired)) (void)ld_acquire_gpu(ctr);
  __syncwarp();
  if (lane == 0) *ctr = 0;
  const bool in_tmem = pm.flags & kInTmem;
  const bool own_empty = pm.flags & kOwnEmpty;
  constexpr float kLog2e = 1.4426950408889634f;
  const bool store = row < Nq;
  __nv_bfloat16* orow = o + (static_cast<size_t>(head) * Nq + (store ? row : 0)) * D;
  const bool wide = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
  // the own part's 32 columns c0.., times f
  auto own_cols = [&](int c0, float f, float* acc) {
    if (own_empty) {
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    } else if (in_tmem) {
      uint32_t x[32];
      tmem_ld32_wait(tO + c0, x);
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(x[i]) * f;
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) ld_global_cg_v8(part_o + part_index<D>(pm.own_slot, r, c0 / 8 + i), acc + i * 8);
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] *= f;
    }
  };
  auto store_cols = [&](int c0, const float* acc) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
    if (store) {
      __nv_bfloat16* dst = orow + c0;
      if (wide) {
        st_global_v8(dst, pk);
        st_global_v8(dst + 16, pk + 8);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          reinterpret_cast<uint4*>(dst)[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
  };
  float lse_out;
  if (ps.n == 2) {
    const int s1 = ps.slot[0] == pm.own_slot ? ps.slot[1] : ps.slot[0];  // the other part
    // 32 columns of the other part at a time, the next ones in flight while
    // the current ones are combined (an empty part's rows were never
    // written: loaded, then given weight 0)
    float xa[32], xb[32];
    const float l1 = __ldcg(part_lse + static_cast<size_t>(s1) * kItemRows + r);
#pragma unroll
    for (int i = 0; i < 4; ++i) ld_global_cg_v8(part_o + part_index<D>(s1, r, i), xa + i * 8);
    const float m = fmaxf(pm.lse_own, l1);
    const float w_own = own_empty ? 0.f : exp2f((pm.lse_own - m) * kLog2e);
    const float w1 = l1 == -INFINITY ? 0.f : exp2f((l1 - m) * kLog2e);
    const float wsum = w_own + w1;
    const float inv_w = 1.f / wsum;
    const float f_own = (in_tmem ? w_own * pm.inv_l : w_own) * inv_w;
    const float f1 = w1 * inv_w;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float* cur = (c & 1) ? xb : xa;
      float* nxt = (c & 1) ? xa : xb;
      if (c + 1 < D / 32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) ld_global_cg_v8(part_o + part_index<D>(s1, r, (c + 1) * 4 + i), nxt + i * 8);
      }
      float acc[32];
      own_cols(c * 32, f_own, acc);
      if (w1 != 0.f) {
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] += f1 * cur[i];
      }
      store_cols(c * 32, acc);
    }
    lse_out = m + logf(wsum);
  } else {
    // three parts or more: the largest logsumexp, the weights' sum, then 32
    // columns at a time with each other part's columns loaded in turn
    float m = pm.lse_own;
#pragma unroll 1
    for (int q = 0; q < ps.n; ++q) {
      const int sq = ps.slot[q];
      if (sq != pm.own_slot) m = fmaxf(m, __ldcg(part_lse + static_cast<size_t>(sq) * kItemRows + r));
    }
    const float w_own = own_empty ? 0.f : exp2f((pm.lse_own - m) * kLog2e);
    float wsum = w_own;
#pragma unroll 1
    for (int q = 0; q < ps.n; ++q) {
      const int sq = ps.slot[q];
      if (sq == pm.own_slot) continue;
      const float lq = __ldcg(part_lse + static_cast<size_t>(sq) * kItemRows + r);
      wsum += lq == -INFINITY ? 0.f : exp2f((lq - m) * kLog2e);
    }
    const float inv_w = 1.f / wsum;
    const float f_own = (in_tmem ? w_own * pm.inv_l : w_own) * inv_w;
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 32) {
      float acc[32];
      own_cols(c0, f_own, acc);
#pragma unroll 1
      for (int q = 0; q < ps.n; ++q) {
        const int sq = ps.slot[q];
        if (sq == pm.own_slot) continue;
        const float lq = __ldcg(part_lse + static_cast<size_t>(sq) * kItemRows + r);
        if (lq == -INFINITY) continue;  // never written, never read
        const float wq = exp2f((lq - m) * kLog2e) * inv_w;
        float x[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) ld_global_cg_v8(part_o + part_index<D>(sq, r, c0 / 8 + i), x + i * 8);
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] += wq * x[i];
      }
      store_cols(c0, acc);
    }
    lse_out = m + logf(wsum);
  }
  if (store) lse[static_cast<size_t>(head) * Nq + row] = lse_out;
}

// ---------------------------------------------------------------------------
// Softmax / correction / epilogue warpgroup (128 threads, one row each)
// ---------------------------------------------------------------------------
template <int D, bool CAUSAL, int E = 2, bool PAIRED = false>
__device__ __forceinline__ void run_softmax(int t, uint32_t tmem, const Sync& sy, const FwdParams& p) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int quad = warp & 3;                       // TMEM lanes 32*quad .. 32*quad+31
  const int row_in_tile = quad * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t tS = tmem + lane_off + t * 128;
  const uint32_t tO = tmem + lane_off + 256 + t * 128;
  const float qk_base = p.qk_scale;
  const bool ragged = (p.Nk % kBlockN) != 0;
  // this warpgroup's barriers, selected once (no run-time array indexing)
  const uint32_t bar_s_full = t ? sy.s_full[1] : sy.s_full[0];
  const uint32_t bar_p_ready = t ? sy.p_ready[1] : sy.p_ready[0];
  const uint32_t bar_o_done = t ? sy.o_done[1] : sy.o_done[0];
  const uint32_t bar_o_free = t ? sy.o_free[1] : sy.o_free[0];
  uint32_t s_par = 0;
  uint32_t od_par = 0;  // o_done completes once per chunk in which this tile has keys
  // split items this warp's rows complete, merged after the last chunk
  PendingMerge pend0{-1, 0, 0, 0.f, 0.f, 0, 0}, pend1 = pend0;
  int arrival = -2;  // the first chunk's part: -2 none, -1 stored (arrival due), >= 0 arrived (lane 0: old value)
  bool ok = true;

  const WorkRange wr = p.range[blockIdx.x];
  const SlotPair sp = p.slots[blockIdx.x];
  for (int q = 0, nq = num_chunks(wr); q < nq && ok; ++q) {
    const int item = chunk_item(q, wr);
    int rb0, bh0;
    decode_item(item, p, rb0, bh0);
    const Chunk ch = chunk_of(item, item_steps<CAUSAL, PAIRED>(rb0, p), wr, sp, p);
    const int rb = ch.rb, bh = tile_head(ch.bh, t, PAIRED);  // this query tile's head
    const int n = tiles_for<CAUSAL, PAIRED>(rb, t, p);       // key tiles of this query tile in the item
    const int ne = min(ch.ke, n);                    // ... and its part in this chunk: [kb, ne)
    const int row = tile_row0(rb, t, PAIRED) + row_in_tile;
    // the first chunk's part: its arrival is made while this chunk's first
    // scores are on their way
    if (arrival == -1) arrival = part_arrive(p.counters + sp.k_first * kCountersPerItem + t * 4 + quad, lane);
    // FP8 path: this query tile's scale (one per 128 query rows)
    const float sq = E == 1 ? p.q_scale[static_cast<size_t>(bh) * ((p.Nq + kBlockM - 1) / kBlockM) +
                                        tile_row0(rb, t, PAIRED) / kBlockM]
                            : 1.f;
    if (ne <= ch.kb) {
      // No key tile of this query tile lies in the chunk (past its diagonal).
      // A part still reports its rows, as an empty part: LSE = -inf.
      if (ch.slot >= 0) {
        const PendingMerge pm = part_done<D>(ch, t, quad, lane, row_in_tile, tO, 0.f, -INFINITY, true, arrival, p);
        if (ch.todo) pend1 = pm; else pend0 = pm;
      }
      continue;
    }
    // m_ref: the reference maximum the exponentials are taken against (log2
    // units, already times qk_scale).  It is moved only when a tile's maximum
    // exceeds it by more than kRescaleThreshold, so P = exp2(s*qk - m_ref) may
    // reach 2^kRescaleThreshold (2^32 for bf16, 2^8 for e4m3).  l, lq and O
    // all use the same m_ref, so the shift cancels in O = acc / lq and in
    // L = m_ref + log2 l exactly as in the every-tile update ("Softmax, the
    // safe way": a common shift factors out).
    float m_ref = -INFINITY;
    float l = 0.f;        // running sum of exp2(s*qk - m_ref), for the logsumexp
    float lq = 0.f;       // the same terms rounded to bf16 (what P.V multiplies), for O

    for (int j = ch.kb; j < ne; ++j) {
      // the factor from the tensor core's sums to log2-units scores: the
      // softmax scale times log2 e, and on the FP8 path the Q and K tiles' scales
      const float qk = E == 1 ? qk_base * sq * p.k_scale[static_cast<size_t>(bh) * p.n_key_tiles + j] : qk_base;
      ok = wait_phase(bar_s_full, s_par, sy, p, kSiteSoftmax);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      s_par ^= 1u;
      tc_fence_after_sync();

      uint32_t s[128];
      tmem_ld128_wait(tS, s);

      // Mask the diagonal tile (causal) and the ragged last tile: a key is
      // kept iff key <= min(row, Nk-1) (causal) or key <= Nk-1.
      const bool need_mask = (CAUSAL && j == n - 1) || (ragged && j == p.n_key_tiles - 1);
      if (need_mask) {
        const int lim = (CAUSAL ? min(row, p.Nk - 1) : p.Nk - 1) - j * kBlockN;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) s[c] = __float_as_uint(-INFINITY);
      }

      const uint64_t qk2 = f2_pack(qk, qk);
      float alpha = 1.f;
      float sa, sb, lq_tile;
      // One pass over the tile: exponentials against m_use, P stored to
      // tensor memory over S, the fp32 and bf16 row sums, and (if asked) the
      // tile's row maximum from the same values.
      auto exp_pass = [&](float m_use, bool with_max) -> float {
        const uint64_t negm2 = f2_pack(-m_use, -m_use);
        uint64_t sum2 = f2_pack(0.f, 0.f);
        float lqs[4] = {0.f, 0.f, 0.f, 0.f};  // four short chains for the bf16 sum
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          if constexpr (E == 2) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int c = c4 * 32 + 2 * i;
              const uint64_t x = f2_fma(f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), qk2, negm2);
              float xa, xb;
              f2_unpack(x, xa, xb);
              const float a = ex2_approx(xa);
              const float b = ex2_approx(xb);
              pk[i] = pack_bf16x2(a, b);
              sum2 = f2_add(sum2, f2_pack(a, b));
              // also sum the bf16 values the P.V product multiplies, so that
              // O / lq is an exact weighted average of the value rows
              add_bf16x2_halves(lqs[(i & 1) * 2], lqs[(i & 1) * 2 + 1], pk[i]);
              if (with_max) mx[c4] = fmax3(mx[c4], __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
            }
            tmem_st16(tS + c4 * 16, pk);
          } else {
            // FP8 path: P rounded to e4m3, four per 32-bit column
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int c = c4 * 32 + 4 * i;
              const uint64_t x01 = f2_fma(f2_pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), qk2, negm2);
              const uint64_t x23 =
                  f2_fma(f2_pack(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])), qk2, negm2);
              float x0, x1, x2, x3;
              f2_unpack(x01, x0, x1);
              f2_unpack(x23, x2, x3);
              const float a = ex2_approx(x0), b = ex2_approx(x1), cc = ex2_approx(x2), dd = ex2_approx(x3);
              pk[i] = pack_e4m3x4(a, b, cc, dd);
              sum2 = f2_add(sum2, f2_add(f2_pack(a, b), f2_pack(cc, dd)));
              // the e4m3 values the P.V product multiplies, summed for lq
              add_e4m3x2_halves(lqs[0], lqs[1], static_cast<uint16_t>(pk[i] & 0xffffu));
              add_e4m3x2_halves(lqs[2], lqs[3], static_cast<uint16_t>(pk[i] >> 16));
              if (with_max) {
                mx[c4] = fmax3(mx[c4], __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
                mx[c4] = fmax3(mx[c4], __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
              }
            }
            tmem_st8(tS + c4 * 8, pk);
          }
        }
        f2_unpack(sum2, sa, sb);
        lq_tile = (lqs[0] + lqs[1]) + (lqs[2] + lqs[3]);
        return fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]) * qk;  // qk > 0: max commutes with the scale
      };
      // The row maximum over the tile, alone: four chains of 32 columns.
      auto row_max = [&]() -> float {
        float mx[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint32_t* sc = s + 32 * q4;
          mx[q4] = fmax3(__uint_as_float(sc[0]), __uint_as_float(sc[1]), __uint_as_float(sc[2]));
        }
#pragma unroll
        for (int i = 3; i < 31; i += 2) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            mx[q4] = fmax3(mx[q4], __uint_as_float(s[32 * q4 + i]), __uint_as_float(s[32 * q4 + i + 1]));
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) mx[q4] = fmaxf(mx[q4], __uint_as_float(s[32 * q4 + 31]));
        return fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]) * qk;
      };
      if constexpr (CAUSAL) {
        // The maximum first, then one pass (under the causal mask, whose short
        // items have many first tiles, this measured faster).
        const float m_tile = row_max();
        if (m_tile > m_ref + kRescaleThreshold<E>) {  // always taken on the first tile (m_ref = -inf)
          alpha = ex2_approx(m_ref - m_tile);      // 0 when m_ref = -inf
          m_ref = m_tile;
        }
        exp_pass(m_ref == -INFINITY ? 0.f : m_ref, false);  // 0: a fully masked row, P = 0
      } else {
        // The exponentials are taken against the current reference m_ref
        // while the tile's own maximum is found in the same pass.  Only if
        // some row's tile maximum exceeds m_ref by more than
        // kRescaleThreshold does the warp move that row's reference and take
        // the pass again, discarding the first one's P and sums (P may then
        // have overflowed; nothing of it is kept).  A chunk's first tile
        // (m_ref = -inf) takes its maximum first, so one pass is enough there.
        if (m_ref == -INFINITY) {
          m_ref = row_max();
          alpha = 0.f;  // nothing accumulated before this tile
        }
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
          const float m_tile = exp_pass(m_ref == -INFINITY ? 0.f : m_ref, true);
          const bool move = m_tile > m_ref + kRescaleThreshold<E>;
          if (!__any_sync(0xffffffffu, move)) break;
          if (move) {  // rare: move this row's reference, then the warp takes the pass again
            alpha = ex2_approx(m_ref - m_tile);
            m_ref = m_tile;
          }
          tmem_st_wait();  // the repeated pass stores P over this one's
        }
      }
      l = l * alpha + (sa + sb);
      lq = lq * alpha + lq_tile;

      if (j > ch.kb && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O_t holds the sum up to tile j-1 (that P.V went out in the same
        // group as S_t(j), whose completion was just waited for); bring it
        // to the new reference maximum where a row moved it (alpha = 1
        // elsewhere, exact).
        {
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t o[64];
            tmem_ld64_wait(tO + c * 64, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float lo, hi;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), a2), lo, hi);
              o[2 * i] = __float_as_uint(lo);
              o[2 * i + 1] = __float_as_uint(hi);
            }
            tmem_st32(tO + c * 64, o);
            tmem_st32(tO + c * 64 + 32, o + 32);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p_ready);  // one arrival per warp
    }
    if (!ok) break;

    // Epilogue: wait for the last P.V, then O = O_acc / l in bf16 and the
    // natural-log logsumexp L = (m + log2 l) * ln 2.
    ok = wait_phase(bar_o_done, od_par, sy, p, kSiteSoftmax);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    od_par ^= 1u;
    tc_fence_after_sync();
    // FP8 path: V's per-head scale comes in here (it is common to every key)
    const float inv_l = (E == 1 ? p.v_scale[bh] : 1.f) / lq;
    const uint64_t il2 = f2_pack(inv_l, inv_l);
    const float lse_row = (m_ref + log2f(l)) * 0.69314718055994531f;
    if (ch.slot < 0) {
      // the chunk is the whole item: final O in bf16 and LSE, rows < N only
      const bool store = row < p.Nq;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.Nq + (store ? row : 0)) * D;
      // rows are D * 2 bytes (a multiple of 32), so every row is 32-byte
      // aligned when O is; the API promises only 16
      const bool wide = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32_wait(tO + c * 32, o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float lo, hi;
          f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), il2), lo, hi);
          w[i] = pack_bf16x2(lo, hi);
        }
        if (store) {
          if (wide) {  // 32-byte stores: half the store instructions, whole sectors
            st_global_v8(orow + c * 32, w);
            st_global_v8(orow + c * 32 + 16, w + 8);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
      }
      if (store) p.lse[static_cast<size_t>(bh) * p.Nq + row] = lse_row;
    } else {
      // a part of the item: merged once every part is in (merge_item)
      const PendingMerge pm = part_done<D>(ch, t, quad, lane, row_in_tile, tO, inv_l, lse_row, false, arrival, p);
      if (ch.todo) pend1 = pm; else pend0 = pm;
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_o_free);  // one arrival per warp
  }
  // The merges of the split items these rows completed.  The last chunk's O
  // is still in tensor memory: no product of this tile follows it.
  if (!ok || *sy.abort_flag) return;
  // the first chunk's part, when no later chunk of this tile made its arrival
  if (arrival == -1) arrival = part_arrive(p.counters + sp.k_first * kCountersPerItem + t * 4 + quad, lane);
  if (arrival >= 0 && __shfl_sync(0xffffffffu, arrival, 0) != p.merge_count[sp.k_first] - 1) pend0.k = -1;
#pragma unroll 1
  for (int i = 0; i < 2; ++i) {
    const PendingMerge pm = i ? pend1 : pend0;
    if (pm.k < 0) continue;
    PartSlots ps;
    ps.n = p.merge_count[pm.k];
    const int first = p.merge_first[pm.k];
#pragma unroll
    for (int q = 0; q < kMaxPartsPerItem; ++q) ps.slot[q] = q < ps.n ? p.merge_slots[first + q] : -1;
    tc_fence_after_sync();
    merge_rows<D>(pm, ps, t, quad, tO, p.counters + pm.k * kCountersPerItem + t * 4 + quad, p.o, p.lse, p.part_o,
                  p.part_lse, p.Nq, PAIRED);
  }
}

// ---------------------------------------------------------------------------
// Kernel
// ---------------------------------------------------------------------------
template <int D, bool CAUSAL, int E = 2, bool PAIRED = false>
__global__ void __launch_bounds__(kNumThreads, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using C = Cfg<D, E>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  Sync sy;
  {
    uint32_t b = sbase + C::kBarOff;
    for (int t = 0; t < 2; ++t) sy.q_full[t] = b + 8 * t;
    b += 16;
    for (int t = 0; t < 2; ++t) sy.q_empty[t] = b + 8 * t;
    b += 16;
    sy.kv_full0 = b;
    b += 8 * C::kStages;
    sy.kv_empty0 = b;
    b += 8 * C::kStages;
    for (int t = 0; t < 2; ++t) sy.s_full[t] = b + 8 * t;
    b += 16;
    for (int t = 0; t < 2; ++t) sy.p_ready[t] = b + 8 * t;
    b += 16;
    for (int t = 0; t < 2; ++t) sy.o_done[t] = b + 8 * t;
    b += 16;
    for (int t = 0; t < 2; ++t) sy.o_free[t] = b + 8 * t;
    b += 16;
    sy.drain = b;
    b += 8;
    for (int t = 0; t < 2; ++t) sy.turn[t] = b + 8 * t;
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  sy.abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(sy.q_full[t], 1);
      mbar_init(sy.q_empty[t], 1);
      mbar_init(sy.s_full[t], 1);
      mbar_init(sy.p_ready[t], kBlockM / 32);  // one arrival per softmax warp
      mbar_init(sy.o_done[t], 1);
      mbar_init(sy.o_free[t], kBlockM / 32);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(sy.kv_full0 + 8 * s, 1);
      mbar_init(sy.kv_empty0 + 8 * s, 2);  // released by both MMA issuers
    }
    mbar_init(sy.drain, 2);  // one commit from each MMA issuer
    mbar_init(sy.turn[0], 1);
    mbar_init(sy.turn[1], 1);
    *sy.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    setmaxnreg_dec<kRegsAux>();
    if (warp == kLoadWarp) {
      if (lane == 0) run_producer<D, CAUSAL, E, PAIRED>(&tmQ, &tmK, &tmV, sbase, sy, p);
      __syncwarp();
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
      run_mma<D, CAUSAL, E, PAIRED>(warp - kMmaWarp, sbase, tmem, sy, p);
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    run_softmax<D, CAUSAL, E, PAIRED>(warp >> 2, tmem, sy, p);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
