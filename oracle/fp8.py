"""FP8 (e4m3) quantisation with per-block scales, and attention on the
dequantised values: the fp64 oracle for the FP8 forward.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs use it, and it
shares no code with the CUDA path.

What is computed, and where it comes from
-----------------------------------------
The pages name the method only in outline: FlashAttention-3's FP8 path
quantises with per-block scaling ("FlashAttention and kernels.", section
"FlashAttention-2, -3, and what came after"; "4 Triton and Custom Kernels",
section 4.8, which calls the FP8 path hardware- and kernel-specific).  The
readings taken here (listed in the design notes):

* ``e4m3_round`` — round to the nearest value of the e4m3 format (1 sign
  bit, 4 exponent bits with bias 7, 3 mantissa bits, subnormals, no
  infinities), ties to even, and values beyond the largest finite one
  (448 = 1.75 * 2^8) clamped to it (saturation, as the format has no
  infinity).  Written from that definition: for |x| >= 2^-6 the spacing is
  2^(floor(log2 |x|) - 3); below, the subnormal spacing 2^-9.
* ``quantize_blocks`` — a block of rows shares one scale: s = amax / 448
  (computed in fp32; s = 1 for an all-zero block), and each element becomes
  e4m3_round(x / s) with the division in fp32, so that the codes are the
  ones a kernel dividing in fp32 produces.
* ``attention_fp8`` — the plain attention definition (``attention``) on
  the dequantised inputs q8 * sQ, k8 * sK, v8 * sV, in fp64.  What the FP8
  kernel computes beyond that (P itself rounded to e4m3 before P V) is an
  approximation whose error the tests bound.

Parity status: pinned by tests/test_oracle_fp8_pins.py (torch's own e4m3
conversion for every finite e4m3 value and for random values inside the
range, the format's constants, ties, saturation, scale and block
bookkeeping, and the attention of exactly representable inputs).
"""
from __future__ import annotations

import math

import numpy as np

from .attention import attention

__all__ = ["E4M3_MAX", "e4m3_round", "quantize_blocks", "dequantize_blocks", "attention_fp8"]

E4M3_MAX = 448.0
_MIN_NORMAL = 2.0 ** -6
_SUB_STEP = 2.0 ** -9


def e4m3_round(x) -> np.ndarray:
    """Nearest e4m3 value of each element (ties to even), saturating at +-448; float64 out."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    normal = a >= _MIN_NORMAL
    # spacing of the grid at each magnitude: 2^(e - 3) for 2^e <= |x| < 2^(e+1)
    e = np.floor(np.log2(np.where(normal, a, 1.0)))
    # log2 may land a hair below an exact power of two; correct the exponent
    e = np.where(normal & (2.0 ** (e + 1) <= a), e + 1, e)
    e = np.where(normal & (2.0 ** e > a), e - 1, e)
    step = np.where(normal, 2.0 ** (e - 3), _SUB_STEP)
    q = a / step                                   # exact: step is a power of two
    r = np.floor(q)
    frac = q - r
    up = (frac > 0.5) | ((frac == 0.5) & (np.mod(r, 2.0) == 1.0))
    r = r + up
    mag = np.minimum(r * step, E4M3_MAX)           # the next grid value above 448 would be 480: clamp
    return np.copysign(mag, x)


def quantize_blocks(x, rows_per_scale: int):
    """Per-block e4m3 quantisation of x [..., N, d] along N.

    Returns (codes as float64 e4m3 values [..., N, d], scales float32
    [..., ceil(N / rows_per_scale)]).  Block b covers rows
    [b * rows_per_scale, min(N, (b + 1) * rows_per_scale)).
    """
    x32 = np.asarray(x, dtype=np.float32)
    n = x32.shape[-2]
    nb = -(-n // rows_per_scale)
    lead = x32.shape[:-2]
    codes = np.empty(x32.shape, dtype=np.float64)
    scales = np.empty(lead + (nb,), dtype=np.float32)
    for b in range(nb):
        r0, r1 = b * rows_per_scale, min(n, (b + 1) * rows_per_scale)
        blk = x32[..., r0:r1, :]
        amax = np.max(np.abs(blk), axis=(-2, -1)).astype(np.float32)
        s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
        scales[..., b] = s
        codes[..., r0:r1, :] = e4m3_round((blk / s[..., None, None]).astype(np.float32))
    return codes, scales


def dequantize_blocks(codes, scales, rows_per_scale: int) -> np.ndarray:
    """codes * scale of each row's block, in float64."""
    codes = np.asarray(codes, dtype=np.float64)
    s = np.repeat(np.asarray(scales, dtype=np.float64), rows_per_scale, axis=-1)[..., : codes.shape[-2]]
    return codes * s[..., None]


def attention_fp8(q8, sq, k8, sk, v8, sv, scale: float, causal: bool, q_rows: int = 128,
                  k_rows: int = 128, v_rows: int | None = None):
    """Attention (O, LSE in fp64) of the dequantised q8 * sQ, k8 * sK, v8 * sV.

    Q and K carry one scale per ``q_rows`` / ``k_rows`` rows; V one per
    ``v_rows`` rows (default: one per head, the whole sequence).
    """
    n_k = np.asarray(k8).shape[-2]
    v_rows = v_rows or n_k
    q = dequantize_blocks(q8, sq, q_rows)
    k = dequantize_blocks(k8, sk, k_rows)
    v = dequantize_blocks(v8, sv, v_rows)
    return attention(q, k, v, scale, causal)


def e4m3_grid() -> np.ndarray:
    """Every non-negative finite e4m3 value, ascending (from the bit layout)."""
    vals = []
    for ebits in range(16):
        for mbits in range(8):
            if ebits == 15 and mbits == 7:
                continue                               # the NaN encoding
            if ebits == 0:
                vals.append(mbits * _SUB_STEP)
            else:
                vals.append((1.0 + mbits / 8.0) * math.ldexp(1.0, ebits - 7))
    return np.array(vals)
