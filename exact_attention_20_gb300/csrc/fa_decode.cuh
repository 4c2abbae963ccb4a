// Exact attention for a few query rows over many keys (decoding), on the CUDA
// cores: split keys, then a merge of the partial results.
//
// The work is bound by reading K and V once (about half a FLOP per byte), so
// no tensor core is used: a 128-row tile would be almost all padding rows.
// Keys are cut into equal chunks, one CTA per (chunk, batch*head), about
// eight CTAs per SM in all; each CTA streams its chunk through a
// shared-memory ring filled by bulk copies, and each of its consumer warps
// keeps an online softmax (running maximum m, running sum l, rescaled fp32
// accumulator: "FlashAttention and kernels.", section "From a sum to an
// output row").  The eight warps' states are combined through shared memory,
// and the chunks' normalised partial outputs are merged through their
// logsumexps ("FlashAttention and kernels.", the merge of partial states over
// key ranges that Flash-Decoding uses), by the last CTA of each (batch, head)
// in the same launch or, without arrival counters, by merge_kernel.  P stays
// in fp32: nothing is rounded before P.V.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace fa {
namespace decode {

constexpr int kWarps = 8;                     // consumer warps
constexpr int kThreadsAll = (kWarps + 1) * 32;  // and one producer warp
constexpr int kStages = 3;                    // shared-memory ring depth (rounds)
constexpr int kGroup = 8;                     // keys a warp loads together
constexpr int kKeysPerRound = kWarps * kGroup;  // consecutive keys the CTA reads per round
constexpr int kMaxRows = 4;                   // query rows this path takes
constexpr int kMaxChunks = 1024;              // key chunks per (batch, head), at most

struct Params {
  const __nv_bfloat16* q;  // [BH][Nq][D]
  const __nv_bfloat16* k;  // [BH][Nk][D]
  const __nv_bfloat16* v;  // [BH][Nk][D]
  __nv_bfloat16* o;        // [BH][Nq][D]
  float* lse;              // [BH][Nq], natural log
  float* part_o;           // split: [BH][Nq][n_chunks][D], O of each chunk normalised within it
  float* part_lse;         // split: [BH][Nq][n_chunks], each chunk's logsumexp in log2 units
  int Nq, Nk;
  int keys_per_chunk;      // a multiple of kKeysPerRound
  int n_chunks;
  float qk_scale;          // softmax scale * log2(e)
  int* status;             // device status word (0 = ok)
  unsigned long long wait_limit_ns;
  int* counters;           // split, merged in the same launch: [BH] chunk arrivals (0 between launches);
                           // nullptr: merge_kernel merges afterwards
};

constexpr int kSiteDecode = 5;  // status code: a decode wait gave up

// Dynamic shared memory of one CTA: the ring, then its barriers.
template <int D>
constexpr int smem_bytes() {
  return kStages * 2 * kKeysPerRound * D * 2 + 2 * kStages * 8;
}

// The lane's share of a row (EPL consecutive bf16 values), as loaded: one
// 8-byte (EPL = 4) or 4-byte (EPL = 2) word pair / word.  `row` already
// points at the lane's first element.
template <int EPL>
struct Packed {
  uint32_t w[EPL / 2];
};

template <int EPL>
__device__ __forceinline__ Packed<EPL> load_packed(const __nv_bfloat16* row) {
  Packed<EPL> r;
  if constexpr (EPL == 4) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(row));
    r.w[0] = u.x;
    r.w[1] = u.y;
  } else {
    r.w[0] = __ldg(reinterpret_cast<const uint32_t*>(row));
  }
  return r;
}

template <int EPL>
__device__ __forceinline__ Packed<EPL> load_packed_shared(const __nv_bfloat16* row) {
  Packed<EPL> r;
  if constexpr (EPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(row);
    r.w[0] = u.x;
    r.w[1] = u.y;
  } else {
    r.w[0] = *reinterpret_cast<const uint32_t*>(row);
  }
  return r;
}

// A bf16 pair (low half first) as an fp32 pair: each bf16 value is the upper
// half of the fp32 one, so the conversion is exact.
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// This lane's part of q . k (its EPL elements), from fp32 pairs of q and the
// packed bf16 of k.
template <int EPL>
__device__ __forceinline__ float dot_share(const uint64_t* q2, const Packed<EPL>& k) {
  uint64_t s2 = f2_mul(q2[0], bf16x2_to_f2(k.w[0]));
#pragma unroll
  for (int e = 1; e < EPL / 2; ++e) s2 = f2_fma(q2[e], bf16x2_to_f2(k.w[e]), s2);
  float lo, hi;
  f2_unpack(s2, lo, hi);
  return lo + hi;
}

// One CTA: key chunk blockIdx.x of batch*head blockIdx.y, rows 0 .. Nq-1
// (NQ >= Nq; rows past Nq are computed on zeros and never written).
//
// A producer warp streams the chunk through a ring of kStages shared-memory
// stages, one round (64 keys: K rows, then V rows, each block contiguous in
// global memory) per stage, with one bulk copy per block; the bytes in flight
// are then set by the ring, not by registers.  The eight consumer warps
// read a round from shared memory (each lane its D/32 elements of a row, so
// a warp reads whole rows) and release the stage.  Every wait is bounded: a
// wait that gives up records kSiteDecode in the status word and ends the
// CTA's loop.
template <int D, int NQ>
__global__ void __launch_bounds__(kThreadsAll, NQ == 4 ? 1 : 2) partial_kernel(const Params p) {
  constexpr int EPL = D / 32;                              // d-elements per lane
  constexpr uint32_t kBlockBytes = kKeysPerRound * D * 2;  // K (or V) rows of one round
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kStages * 2 * kBlockBytes;  // full[kStages], then empty[kStages]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x, bh = blockIdx.y;
  const int k_begin = chunk * p.keys_per_chunk;
  const int k_end = min(p.Nk, k_begin + p.keys_per_chunk);
  const int n_rounds = (k_end - k_begin + kKeysPerRound - 1) / kKeysPerRound;
  auto full = [&](int st) { return bar0 + 8 * st; };
  auto empty = [&](int st) { return bar0 + 8 * (kStages + st); };
  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(full(st), 1);
      mbar_init(empty(st), kWarps * 32);  // every consumer thread, once its reads are done
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // producer: one thread issues the copies of every round
    if (lane == 0) {
      const __nv_bfloat16* kg = p.k + (static_cast<size_t>(bh) * p.Nk + k_begin) * D;
      const __nv_bfloat16* vg = p.v + (static_cast<size_t>(bh) * p.Nk + k_begin) * D;
      int issued = 0;
      for (int r = 0; r < n_rounds; ++r) {
        const int st = r % kStages;
        if (r >= kStages && !mbar_wait_bounded(empty(st), ((r / kStages) - 1) & 1, p.wait_limit_ns)) {
          atomicCAS(p.status, 0, kSiteDecode);
          break;
        }
        const int keys = min(kKeysPerRound, k_end - k_begin - r * kKeysPerRound);
        const uint32_t bytes = static_cast<uint32_t>(keys) * D * 2;  // a multiple of 128
        mbar_arrive_expect_tx(full(st), 2 * bytes);
        const size_t off = static_cast<size_t>(r) * kKeysPerRound * D;
        bulk_load(sbase + st * 2 * kBlockBytes, kg + off, bytes, full(st));
        bulk_load(sbase + st * 2 * kBlockBytes + kBlockBytes, vg + off, bytes, full(st));
        issued = r + 1;
      }
      // Drain: every copy issued has landed before the CTA can exit, also
      // after a wait gave up (at most one round per stage can be in flight).
      for (int r = max(0, issued - kStages); r < issued; ++r)
        mbar_wait_bounded(full(r % kStages), (r / kStages) & 1, p.wait_limit_ns);
    }
    __syncwarp();
  }

  float m[NQ], l[NQ];
  uint64_t acc2[NQ][EPL / 2];  // the lane's share of each row's accumulator, as fp32 pairs
#pragma unroll
  for (int r = 0; r < NQ; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL / 2; ++e) acc2[r][e] = f2_pack(0.f, 0.f);
  }
  if (warp < kWarps) {
    // this lane's share of each query row, in log2 units (scale * log2 e
    // folded in), as fp32 pairs
    uint64_t q2[NQ][EPL / 2];
    const uint64_t qs2 = f2_pack(p.qk_scale, p.qk_scale);
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      const Packed<EPL> qp = r < p.Nq ? load_packed<EPL>(p.q + (static_cast<size_t>(bh) * p.Nq + r) * D + lane * EPL)
                                      : Packed<EPL>{};
#pragma unroll
      for (int e = 0; e < EPL / 2; ++e) q2[r][e] = f2_mul(bf16x2_to_f2(r < p.Nq ? qp.w[e] : 0u), qs2);
    }
    const bool b2 = (lane >> 2) & 1, b3 = (lane >> 3) & 1, b4 = (lane >> 4) & 1;
    const int kl = (lane >> 2) & 7;  // the key whose score this lane ends up holding
    // Round by round, warp w takes keys 8w .. 8w+7 of the round.
#pragma unroll 1
    for (int rd = 0; rd < n_rounds; ++rd) {
      const int st = rd % kStages;
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(full(st), (rd / kStages) & 1, p.wait_limit_ns));
      if (!ok) {
        if (lane == 0) atomicCAS(p.status, 0, kSiteDecode);
        break;
      }
      const int nk = min(kGroup, k_end - (k_begin + rd * kKeysPerRound + warp * kGroup));  // may be <= 0
      if (nk > 0) {
        const __nv_bfloat16* ks = reinterpret_cast<const __nv_bfloat16*>(smem + st * 2 * kBlockBytes) +
                                  warp * kGroup * D + lane * EPL;
        const __nv_bfloat16* vs = ks + kBlockBytes / 2;
        Packed<EPL> kp[kGroup], vp[kGroup];
#pragma unroll
        for (int i = 0; i < kGroup; ++i) {
          const int row = min(i, nk - 1);  // a key past the chunk re-reads the last one (masked below)
          kp[i] = load_packed_shared<EPL>(ks + row * D);
          vp[i] = load_packed_shared<EPL>(vs + row * D);
        }
        mbar_arrive(empty(st));  // this thread's rows are in registers
#pragma unroll
        for (int r = 0; r < NQ; ++r) {
          // Dot products of the eight keys, summed over the 32 lanes by a
          // reduce-scatter: afterwards lane l holds the score of key
          // kl = (l >> 2) & 7, each lane having shuffled 9 values, not 40.
          float v8[kGroup];
#pragma unroll
          for (int i = 0; i < kGroup; ++i) v8[i] = dot_share<EPL>(q2[r], kp[i]);
          float w4[4], x2[2];
#pragma unroll
          for (int i = 0; i < 4; ++i) {  // lanes 0-15 keep keys 0-3, lanes 16-31 keys 4-7
            const float send = b4 ? v8[i] : v8[i + 4];
            w4[i] = (b4 ? v8[i + 4] : v8[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
          }
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float send = b3 ? w4[i] : w4[i + 2];
            x2[i] = (b3 ? w4[i + 2] : w4[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
          }
          float sc = (b2 ? x2[1] : x2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? x2[0] : x2[1], 4);
          sc += __shfl_xor_sync(0xffffffffu, sc, 2);
          sc += __shfl_xor_sync(0xffffffffu, sc, 1);
          if (kl >= nk) sc = -INFINITY;  // a key past the chunk
          float mx = fmaxf(sc, __shfl_xor_sync(0xffffffffu, sc, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          // the group holds at least one key, so mx and m_new are finite
          const float m_new = fmaxf(m[r], mx);
          const float alpha = ex2_approx(m[r] - m_new);  // 0 on the first group (m = -inf)
          const float pl = ex2_approx(sc - m_new);       // this lane's key; 0 for a masked key
          float psum = pl + __shfl_xor_sync(0xffffffffu, pl, 4);
          psum += __shfl_xor_sync(0xffffffffu, psum, 8);
          psum += __shfl_xor_sync(0xffffffffu, psum, 16);
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
          for (int e = 0; e < EPL / 2; ++e) acc2[r][e] = f2_mul(acc2[r][e], a2);
#pragma unroll
          for (int i = 0; i < kGroup; ++i) {
            const float pi = __shfl_sync(0xffffffffu, pl, 4 * i);  // key i's P, from a lane holding it
            const uint64_t p2 = f2_pack(pi, pi);
#pragma unroll
            for (int e = 0; e < EPL / 2; ++e) acc2[r][e] = f2_fma(p2, bf16x2_to_f2(vp[i].w[e]), acc2[r][e]);
          }
          l[r] = l[r] * alpha + psum;
          m[r] = m_new;
        }
      } else {
        mbar_arrive(empty(st));
      }
    }
  }

  // The eight warps' states, combined: M = max m_w, L = sum l_w 2^(m_w - M),
  // O = sum acc_w 2^(m_w - M) / L.
  __shared__ float s_m[kWarps][NQ], s_l[kWarps][NQ];
  __shared__ float s_acc[kWarps][NQ][D];
  if (warp < kWarps) {
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      if (lane == 0) {
        s_m[warp][r] = m[r];
        s_l[warp][r] = l[r];
      }
#pragma unroll
      for (int e = 0; e < EPL / 2; ++e) {
        float lo, hi;
        f2_unpack(acc2[r][e], lo, hi);
        s_acc[warp][r][lane * EPL + 2 * e] = lo;
        s_acc[warp][r][lane * EPL + 2 * e + 1] = hi;
      }
    }
  }
  __syncthreads();
  const bool split = p.n_chunks > 1;
  for (int idx = threadIdx.x; idx < NQ * D; idx += kThreadsAll) {
    const int r = idx / D, e = idx % D;
    if (r >= p.Nq) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][r]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = s_m[w][r] == -INFINITY ? 0.f : exp2f(s_m[w][r] - M);  // a warp with no key weighs 0
      L += s_l[w][r] * f;
      O += s_acc[w][r][e] * f;
    }
    O /= L;
    const float lse2 = M + log2f(L);
    const size_t row = static_cast<size_t>(bh) * p.Nq + r;
    if (split) {
      p.part_o[(row * p.n_chunks + chunk) * D + e] = O;
      if (e == 0) p.part_lse[row * p.n_chunks + chunk] = lse2;
    } else {
      p.o[row * D + e] = __float2bfloat16_rn(O);
      if (e == 0) p.lse[row] = lse2 * 0.69314718055994531f;
    }
  }
  if (!split || p.counters == nullptr) return;
  // The CTA whose arrival completes this head's chunks merges them, while
  // the parts are still in L2: L = log2 sum_c 2^(L_c), O = sum_c 2^(L_c - L)
  // O_c, the largest L_c first.  Every CTA's rows are written (and fenced)
  // before its arrival is counted; the merging CTA resets the counter.
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(p.counters + bh, 1);
    s_last = old == p.n_chunks - 1;
    __threadfence();
  }
  __syncthreads();
  if (!s_last) return;
  for (int idx = threadIdx.x; idx < NQ * D; idx += kThreadsAll) {
    const int r = idx / D, e = idx % D;
    if (r >= p.Nq) continue;
    const size_t row = static_cast<size_t>(bh) * p.Nq + r;
    const float* lc = p.part_lse + row * p.n_chunks;
    const float* oc = p.part_o + row * p.n_chunks * D + e;
    float M = -INFINITY;
    for (int c = 0; c < p.n_chunks; ++c) M = fmaxf(M, __ldcg(lc + c));
    float W = 0.f, O = 0.f;
    int c = 0;
    for (; c + 8 <= p.n_chunks; c += 8) {  // eight chunks' loads in flight together
      float lv[8], ov[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        lv[i] = __ldcg(lc + c + i);
        ov[i] = __ldcg(oc + static_cast<size_t>(c + i) * D);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float w = exp2f(lv[i] - M);
        W += w;
        O = fmaf(w, ov[i], O);
      }
    }
    for (; c < p.n_chunks; ++c) {
      const float w = exp2f(__ldcg(lc + c) - M);
      W += w;
      O = fmaf(w, __ldcg(oc + static_cast<size_t>(c) * D), O);
    }
    p.o[row * D + e] = __float2bfloat16_rn(O / W);
    if (e == 0) p.lse[row] = (M + log2f(W)) * 0.69314718055994531f;
  }
  if (threadIdx.x == 0) p.counters[bh] = 0;
}

// One CTA per (batch*head, row): L = log2 sum_c 2^(L_c), O = sum_c 2^(L_c - L) O_c,
// the largest L_c subtracted first.  The chunks' logsumexps are read once,
// in parallel, into shared memory; then each thread (one output element)
// reads its chunks' values eight at a time, so the loads overlap.
template <int D>
__global__ void __launch_bounds__(D) merge_kernel(const Params p) {
  __shared__ float s_w[kMaxChunks];
  __shared__ float s_red[D / 32];
  const size_t row = blockIdx.x;
  const int e = threadIdx.x;
  const int n = p.n_chunks;  // <= kMaxChunks (the plan's bound)
  const float* lc = p.part_lse + row * p.n_chunks;
  float mx = -INFINITY;
  for (int c = e; c < n; c += D) {
    s_w[c] = lc[c];
    mx = fmaxf(mx, s_w[c]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if ((e & 31) == 0) s_red[e >> 5] = mx;
  __syncthreads();
  float M = s_red[0];
#pragma unroll
  for (int w = 1; w < D / 32; ++w) M = fmaxf(M, s_red[w]);
  for (int c = e; c < n; c += D) s_w[c] = exp2f(s_w[c] - M);
  __syncthreads();
  float W = 0.f, O = 0.f;
  const float* oc = p.part_o + row * p.n_chunks * D + e;
  int c = 0;
  for (; c + 8 <= n; c += 8) {
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = oc[static_cast<size_t>(c + i) * D];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      W += s_w[c + i];
      O = fmaf(s_w[c + i], x[i], O);
    }
  }
  for (; c < n; ++c) {
    W += s_w[c];
    O = fmaf(s_w[c], oc[static_cast<size_t>(c) * D], O);
  }
  p.o[row * D + e] = __float2bfloat16_rn(O / W);
  if (e == 0) p.lse[row] = (M + log2f(W)) * 0.69314718055994531f;
}

}  // namespace decode
}  // namespace fa
