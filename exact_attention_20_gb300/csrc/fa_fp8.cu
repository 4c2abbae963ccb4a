// C ABI of the FP8 quantiser: bf16 Q, K (per 128-row block) and V (per head,
// transposed) to e4m3 codes and fp32 scales, in the layouts fa_fwd_fp8 reads.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_fp8_quant.cuh"
#include "fa_gb300.h"
#include "fa_internal.h"

namespace {

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

template <int D>
int quantize(const void* x, void* x8, float* scales, int BH, int N, int mode, cudaStream_t s) {
  namespace q8 = fa::fp8;
  const int nblk = (N + q8::kRows - 1) / q8::kRows;
  const int n_pad = nblk * q8::kRows;
  const int per_head = mode;
  const int n_scales = per_head ? BH : BH * nblk;
  if (cudaMemsetAsync(scales, 0, static_cast<size_t>(n_scales) * sizeof(float), s) != cudaSuccess)
    return FA_ERR_LAUNCH;
  const dim3 grid(nblk, BH);
  q8::amax_kernel<D><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), scales, N, per_head);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  q8::quantize_kernel<D><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), scales,
                                              static_cast<uint8_t*>(x8), N, n_pad, per_head, mode);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  q8::finalize_scales_kernel<<<(n_scales + 255) / 256, 256, 0, s>>>(scales, n_scales);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_quantize_fp8(const void* x, void* x8, float* scales, int B, int H, int N, int d, int mode, void* stream) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128) || (mode != 0 && mode != 1)) return FA_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 65535) return FA_ERR_INVALID_ARG;  // the grid's y dimension
  const long long nblk = (static_cast<long long>(N) + 127) / 128;
  if (BH * nblk * 128 * d >= (1ll << 31)) return FA_ERR_INVALID_ARG;
  if (!x || !x8 || !scales) return FA_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(x8) & 15u) ||
      (reinterpret_cast<uintptr_t>(scales) & 3u))
    return FA_ERR_ALIGN;
  const size_t xb = static_cast<size_t>(BH) * N * d * 2;
  const size_t x8b = mode ? static_cast<size_t>(BH) * d * nblk * 128 : static_cast<size_t>(BH) * N * d;
  const size_t sb = (mode ? static_cast<size_t>(BH) : static_cast<size_t>(BH * nblk)) * 4;
  if (overlaps(x8, x8b, x, xb) || overlaps(scales, sb, x, xb) || overlaps(scales, sb, x8, x8b))
    return FA_ERR_ALIAS;
  fa_internal::DeviceView view;
  if (!fa_internal::current_device(&view)) return FA_ERR_LAUNCH;
  if (!view.supported) return FA_ERR_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return d == 128 ? quantize<128>(x, x8, scales, static_cast<int>(BH), N, mode, s)
                  : quantize<64>(x, x8, scales, static_cast<int>(BH), N, mode, s);
}

}  // extern "C"
