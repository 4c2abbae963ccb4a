"""Pins for the FP8 oracle (oracle/fp8.py).

The e4m3 rounding is checked against torch's own float8_e4m3fn conversion
(an independent implementation of the same format) on every finite e4m3
value and on random values inside the range, against the format's constants
and tie cases, and for the saturation the oracle reads into it.  The block
quantiser is checked on its bookkeeping (one scale per block, amax mapped to
448, ragged last block, zero blocks), and attention on the dequantised
values against attention on inputs that need no rounding at all.
"""
import numpy as np
import pytest
import torch

from oracle import fp8
from oracle.attention import attention


def torch_e4m3(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_grid_has_every_finite_value_once():
    g = fp8.e4m3_grid()
    assert g.size == 127 and g[0] == 0.0 and g[-1] == 448.0
    assert np.all(np.diff(g) > 0)
    assert g[1] == 2.0 ** -9 and 2.0 ** -6 in g            # smallest subnormal, smallest normal
    assert np.array_equal(fp8.e4m3_round(g), g) and np.array_equal(fp8.e4m3_round(-g), -g)
    assert np.array_equal(torch_e4m3(g), g)                 # the same grid as torch's type


def test_rounding_matches_torch_inside_the_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0)
    ] + [rng.uniform(-448, 448, 20000)]).astype(np.float32)
    assert np.array_equal(fp8.e4m3_round(x), torch_e4m3(x))
    # every midpoint between neighbours (ties): torch and the oracle agree, to even
    g = fp8.e4m3_grid()
    mid = ((g[1:] + g[:-1]) / 2).astype(np.float32)
    assert np.array_equal(fp8.e4m3_round(mid), torch_e4m3(mid))


def test_ties_go_to_even_and_large_values_saturate():
    assert fp8.e4m3_round(1.0625) == 1.0          # between 1.0 (m=000) and 1.125 (m=001)
    assert fp8.e4m3_round(1.1875) == 1.25         # between 1.125 (m=001) and 1.25 (m=010)
    assert fp8.e4m3_round(2.0 ** -10) == 0.0      # half the smallest subnormal: tie to 0
    assert fp8.e4m3_round(3 * 2.0 ** -10) == 2.0 ** -8
    assert fp8.e4m3_round(460.0) == 448.0 and fp8.e4m3_round(1e6) == 448.0
    assert fp8.e4m3_round(-500.0) == -448.0


@pytest.mark.parametrize("n,rows", [(256, 128), (300, 128), (5, 2), (7, 7)])
def test_block_quantiser_bookkeeping(n, rows):
    rng = np.random.default_rng(n)
    x = (rng.standard_normal((2, 3, n, 16)) * rng.uniform(0.1, 5, (2, 3, 1, 1))).astype(np.float32)
    x[1, 2, :min(rows, n)] = 0.0                   # an all-zero block gets scale 1 and zero codes
    codes, scales = fp8.quantize_blocks(x, rows)
    nb = -(-n // rows)
    assert scales.shape == (2, 3, nb) and scales.dtype == np.float32
    assert scales[1, 2, 0] == 1.0 and not codes[1, 2, :min(rows, n)].any()
    for b in range(nb):
        blk = x[..., b * rows:(b + 1) * rows, :]
        amax = np.abs(blk).max(axis=(-2, -1))
        want = np.where(amax > 0, (amax / np.float32(448)).astype(np.float32), 1.0)
        assert np.array_equal(scales[..., b], want)
        c = codes[..., b * rows:(b + 1) * rows, :]
        top = np.abs(c).max(axis=(-2, -1))
        assert np.all((top == 448.0) | (amax == 0))   # each block's largest element maps to 448
    assert np.array_equal(fp8.e4m3_round(codes), codes)
    # dequantised values are within half a step of e4m3 at each block's scale
    deq = fp8.dequantize_blocks(codes, scales, rows)
    rel = np.abs(deq - x) / np.maximum(np.abs(x), 2.0 ** -6 * np.repeat(scales, rows, -1)[..., :n, None])
    assert rel.max() <= 2.0 ** -4 + 1e-6


@pytest.mark.parametrize("causal", [False, True])
def test_attention_of_representable_inputs_is_plain_attention(causal):
    rng = np.random.default_rng(3)
    g = fp8.e4m3_grid()
    pick = lambda shape: rng.choice(np.concatenate([g[:90], -g[1:90]]), size=shape)  # noqa: E731
    q8, k8, v8 = pick((2, 200, 32)), pick((2, 200, 32)), pick((2, 200, 32))
    sq = np.full((2, 2), 0.5, np.float32)
    sk = np.full((2, 2), 0.25, np.float32)
    sv = np.full((2, 1), 2.0, np.float32)
    o, lse = fp8.attention_fp8(q8, sq, k8, sk, v8, sv, 0.1, causal)
    o2, lse2 = attention(q8 * 0.5, k8 * 0.25, v8 * 2.0, 0.1, causal)
    assert np.max(np.abs(o - o2)) <= 1e-12 and np.max(np.abs(lse - lse2)) <= 1e-12
