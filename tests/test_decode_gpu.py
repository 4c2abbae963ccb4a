"""GPU parity of the decode kernels: up to four query rows over many keys, no mask.

fa_fwd_rect (and fa_fwd, for N <= 4) hands these shapes to the split-key
decode kernels.  Every element of O and LSE is compared with the fp64 oracle
on the same bf16 inputs, with the tolerances of the other GPU tests.  The
shapes cover one to four rows (the three kernel instances), key counts that
end inside a 64-key round, inside an eight-key group and on a chunk edge, a
single key, keys that fit one chunk (no merge) and keys cut into many chunks
(merged in the same launch by the CTA that completes a head), both head
sizes, and the bench's decode shape in full.
"""
import numpy as np
import pytest
import torch

from exact_attention_20_gb300 import build as fa_build
from exact_attention_20_gb300.inputs import make_qkv
from tests.parity import assert_close, compare, to_f64

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def fa():
    fa_build.build()
    from exact_attention_20_gb300 import fa as mod
    mod.lib()
    return mod


def _inputs(B, H, Nq, Nk, d, seed, values="normal"):
    q, _, _ = make_qkv(B, H, Nq, d, seed=seed, values=values, device=DEV)
    _, k, v = make_qkv(B, H, Nk, d, seed=seed + 1, values=values, device=DEV)
    return q, k, v


def _check(fa, q, k, v, label):
    d = q.shape[-1]
    scale = d ** -0.5
    o, lse = fa.attention_rect(q, k, v, causal=False, scale=scale)
    torch.cuda.synchronize()
    ref = oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale, False)
    assert_close(compare(o, lse, *ref), label)


@pytest.mark.parametrize("Nq", [1, 2, 3, 4])
@pytest.mark.parametrize("Nk", [1, 7, 64, 65, 1000, 4097])
@pytest.mark.parametrize("d", [64, 128])
def test_decode_every_element(fa, Nq, Nk, d):
    q, k, v = _inputs(2, 3, Nq, Nk, d, seed=70)
    _check(fa, q, k, v, f"decode Nq={Nq} Nk={Nk} d={d}")


@pytest.mark.parametrize("Nq", [1, 4])
def test_decode_bench_shape_every_element(fa, Nq):
    # the decode bench's shape: 32 heads over 32768 keys, split into chunks
    q, k, v = _inputs(1, 32, Nq, 32768, 128, seed=71)
    grid, nsplit = fa.plan(1, 32, Nq, 128, False, n_keys=32768)
    assert nsplit == 32 and grid % 32 == 0 and grid // 32 > 1
    _check(fa, q, k, v, f"decode B1-H32-Nq{Nq}-Nk32768")


def test_decode_outliers(fa):
    # heavy-tailed scores: the running maximum moves often inside a chunk
    q, k, v = _inputs(2, 4, 3, 20000, 128, seed=72, values="outliers")
    _check(fa, q, k, v, "decode outliers")


def test_decode_one_chunk_vs_split(fa):
    # few keys: one chunk, written directly; many keys: chunks and a merge.
    # Both agree with the oracle (checked above); here the plan's choice.
    assert fa.plan(1, 32, 1, 128, False, n_keys=256)[1] == 0
    assert fa.plan(1, 32, 1, 128, False, n_keys=1 << 16)[1] == 32


def test_fa_fwd_few_rows_takes_decode(fa):
    # fa_fwd with N <= 4 and no mask is a decode shape too
    q, k, v = make_qkv(3, 5, 4, 64, seed=73, device=DEV)
    scale = 64 ** -0.5
    o, lse = fa.attention(q, k, v, causal=False, scale=scale)
    torch.cuda.synchronize()
    assert_close(compare(o, lse, *oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale, False)), "fa_fwd N=4")


def test_decode_repeatable(fa):
    # no atomics: the same inputs give the same bits
    q, k, v = _inputs(1, 8, 2, 9000, 128, seed=74)
    o1, l1 = fa.attention_rect(q, k, v, causal=False)
    o2, l2 = fa.attention_rect(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
