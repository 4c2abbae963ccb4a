// FP8 (e4m3) quantisation with per-block scales, for the FP8 forward.
//
// A block of rows shares one scale s = amax / 448 (s = 1 for an all-zero
// block), 448 being e4m3's largest finite value; each element becomes
// e4m3(x / s), rounded to nearest even and saturating at +-448, the
// division in fp32 ("FlashAttention and kernels.", section "FlashAttention-2,
// -3, and what came after": FP8 with per-block scaling).  Q and K get one
// scale per 128 rows (the forward's tiles); V one per (batch, head), because
// its scale has to factor out of the sum over key tiles, and V is written
// transposed ([d][keys], keys padded to a multiple of 128 with zeros) so that
// it is a K-major operand of the P.V product.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace fa {
namespace fp8 {

constexpr int kRows = 128;        // rows per quantisation block (Q, K) and per tile
constexpr float kE4m3Max = 448.f;

// two fp32 values to e4m3 (round to nearest even, saturating): lo in bits
// 0-7, hi in bits 8-15
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// amax of one 128-row block of x [BH][N][d] (rows past N ignored): stored in
// amax[bh * nblk + blk], or, per_head, folded into amax[bh] with an integer
// max on the fp32 bits (valid for non-negative values; amax[] starts at 0).
template <int D>
__global__ void __launch_bounds__(256)
amax_kernel(const __nv_bfloat16* __restrict__ x, float* __restrict__ amax, int N, int per_head) {
  const int blk = blockIdx.x, bh = blockIdx.y, nblk = gridDim.x;
  const int r0 = blk * kRows;
  const int rows = min(kRows, N - r0);
  const uint4* src = reinterpret_cast<const uint4*>(x + (static_cast<size_t>(bh) * N + r0) * D);
  const int n8 = rows * D / 8;
  float m = 0.f;
  for (int i = threadIdx.x; i < n8; i += blockDim.x) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  __shared__ float wm[8];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i) m = fmaxf(m, wm[i]);
    if (per_head)
      atomicMax(reinterpret_cast<unsigned int*>(amax) + bh, __float_as_uint(m));
    else
      amax[static_cast<size_t>(bh) * nblk + blk] = m;
  }
}

__device__ __forceinline__ float scale_of(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f;
}

// x8 = e4m3(x / s) for one 128-row block.  transpose = 0: x8 [BH][N][D];
// transpose = 1: x8 [BH][D][N_pad], padding keys zero (the block goes through
// shared memory so that both the reads and the writes are whole rows).
template <int D>
__global__ void __launch_bounds__(256)
quantize_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ amax, uint8_t* __restrict__ x8,
                int N, int N_pad, int per_head, int transpose) {
  const int blk = blockIdx.x, bh = blockIdx.y, nblk = gridDim.x;
  const int r0 = blk * kRows;
  const int rows = min(kRows, N - r0);
  const float s = scale_of(per_head ? amax[bh] : amax[static_cast<size_t>(bh) * nblk + blk]);
  const uint4* src = reinterpret_cast<const uint4*>(x + (static_cast<size_t>(bh) * N + r0) * D);
  __shared__ __align__(16) uint8_t tile[D][kRows + 16];  // [column][row], padded rows
  for (int i = threadIdx.x; i < kRows * D / 8; i += blockDim.x) {
    const int r = i / (D / 8), c = (i % (D / 8)) * 8;
    uint32_t b[4] = {0u, 0u, 0u, 0u};
    if (r < rows) {
      const uint4 v = src[i];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
        b[k] = e4m3x2(__fdiv_rn(f.x, s), __fdiv_rn(f.y, s));
      }
    }
    if (!transpose) {
      if (r < rows)
        *reinterpret_cast<uint2*>(x8 + (static_cast<size_t>(bh) * N + r0 + r) * D + c) =
            make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        tile[c + 2 * k][r] = static_cast<uint8_t>(b[k] & 0xffu);
        tile[c + 2 * k + 1][r] = static_cast<uint8_t>(b[k] >> 8);
      }
    }
  }
  if (!transpose) return;
  __syncthreads();
  // D rows of 128 bytes: keys r0 .. r0 + 127 of each column (zeros past N)
  for (int i = threadIdx.x; i < D * kRows / 16; i += blockDim.x) {
    const int c = i / (kRows / 16), k16 = (i % (kRows / 16)) * 16;
    *reinterpret_cast<uint4*>(x8 + (static_cast<size_t>(bh) * D + c) * N_pad + r0 + k16) =
        *reinterpret_cast<const uint4*>(&tile[c][k16]);
  }
}

// scales[i] = amax[i] / 448 (1 for an all-zero block), in place
__global__ void __launch_bounds__(256) finalize_scales_kernel(float* __restrict__ amax, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) amax[i] = scale_of(amax[i]);
}

}  // namespace fp8
}  // namespace fa
