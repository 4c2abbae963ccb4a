"""GPU parity of fa_fwd_rect: Nq query rows over Nk keys, top-left causal mask.

Every element of O and LSE is compared with the fp64 oracle on the same
bf16 inputs, with the tolerances of the other GPU tests.  The shapes cover
few query rows over many keys (the decode shape, whose keys the plan splits
over several CTAs), more query rows than keys (rows past the last key see
every key), a single key, ragged key and row tiles, and both head sizes.
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


def _inputs(B, H, Nq, Nk, d, seed):
    q, _, _ = make_qkv(B, H, Nq, d, seed=seed, device=DEV)
    _, k, v = make_qkv(B, H, Nk, d, seed=seed + 1, device=DEV)
    return q, k, v


def _oracle(q, k, v, scale, causal):
    return oracle.attention(to_f64(q), to_f64(k), to_f64(v), scale, causal)


SHAPES = [
    (1, 3, 1, 4096, 128),      # one query row over 4096 keys
    (2, 4, 17, 3001, 64),      # few rows, ragged keys
    (1, 8, 128, 16384, 128),   # decode-like: 8 items over 128 key tiles each, keys split
    (1, 2, 300, 129, 128),     # more rows than keys
    (2, 3, 700, 1000, 64),     # mixed, ragged rows and keys
    (1, 2, 1000, 1, 64),       # a single key
]


@pytest.mark.parametrize("B,H,Nq,Nk,d", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_rect_every_element(fa, B, H, Nq, Nk, d, causal):
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=40)
    scale = d ** -0.5
    o, lse = fa.attention_rect(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert_close(compare(o, lse, *_oracle(q, k, v, scale, causal)), f"rect {Nq}x{Nk}")


def test_decode_shape_splits_keys(fa):
    # 8 heads of 128 rows: 8 items (too few to pair heads), each split
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid, nsplit = fa.plan(1, 8, 128, 128, False, n_keys=16384)
    assert nsplit == 8 and 8 < grid <= min(sms, 8 * 7)
    # too little work to share: whole items
    assert fa.plan(1, 2, 64, 128, False, n_keys=512) == (2, 0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_rect_paired_heads(fa, d, causal):
    # enough heads of <= 128 rows that each item pairs two heads' query tiles
    # (two K/V streams per item) with every CTA busy: every element, every head
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = 2 * sms + 16
    q, k, v = _inputs(1, H, 100, 1000, d, seed=42)
    scale = d ** -0.5
    grid, _ = fa.plan(1, H, 100, d, causal, n_keys=1000)
    assert grid == sms  # every CTA busy (stream-K may still cut items in two)
    o, lse = fa.attention_rect(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert_close(compare(o, lse, *_oracle(q, k, v, scale, causal)), f"paired heads d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_rect_paired_heads_repeated(fa, d, causal):
    # The K/V ring's slots take the two paired heads' tiles in turn, so an
    # issuer that waited for its tile before the other one had seen the
    # slot's previous fill could read that previous tile (one head's output
    # wrong in some launches, depending on load timing).  100 launches of the
    # paired shape on the same inputs: the first against the oracle, every
    # other one against the first (merge order may move the last bits).
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H = 2 * sms + 16
    q, k, v = _inputs(1, H, 100, 1000, d, seed=43)
    scale = d ** -0.5
    o0, lse0 = fa.attention_rect(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert_close(compare(o0, lse0, *_oracle(q, k, v, scale, causal)), f"paired heads d={d} causal={causal}")
    worst_o, worst_l = 0.0, 0.0
    for _ in range(100):
        o, lse = fa.attention_rect(q, k, v, causal=causal, scale=scale)
        worst_o = max(worst_o, (o.float() - o0.float()).abs().max().item())
        worst_l = max(worst_l, (lse - lse0).abs().max().item())
    assert worst_o <= 1e-2 and worst_l <= 1e-3, (worst_o, worst_l)


@pytest.mark.parametrize("causal", [False, True])
def test_rect_square_is_fa_fwd(fa, causal):
    q, k, v = make_qkv(2, 3, 777, 128, seed=41, device=DEV)
    o1, l1 = fa.attention(q, k, v, causal=causal)
    o2, l2 = fa.attention_rect(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_rect_guard_bands(fa, causal):
    B, H, Nq, Nk, d = 1, 4, 33, 5000, 128
    G = 4096
    q, k, v = _inputs(B, H, Nq, Nk, d, seed=42)
    n_o, n_l = B * H * Nq * d, B * H * Nq
    obuf = torch.full((n_o + 2 * G,), -512.0, dtype=torch.bfloat16, device=DEV)
    lbuf = torch.full((n_l + 2 * G,), -512.0, dtype=torch.float32, device=DEV)
    o = obuf[G:G + n_o].view(B, H, Nq, d)
    lse = lbuf[G:G + n_l].view(B, H, Nq)
    fa.fa_fwd_rect(q, k, v, o, lse, causal=causal, scale=0.1)
    torch.cuda.synchronize()
    assert (obuf[:G] == -512.0).all() and (obuf[G + n_o:] == -512.0).all()
    assert (lbuf[:G] == -512.0).all() and (lbuf[G + n_l:] == -512.0).all()
    assert_close(compare(o, lse, *_oracle(q, k, v, 0.1, causal)), "rect guarded")


def test_rect_causal_rows_past_the_keys_see_every_key(fa):
    # top-left: with Nq > Nk, rows from Nk - 1 on are the non-causal result
    q, k, v = _inputs(1, 2, 400, 150, 64, seed=43)
    oc, lc = fa.attention_rect(q, k, v, causal=True)
    on, ln = fa.attention_rect(q, k, v, causal=False)
    torch.cuda.synchronize()
    assert torch.equal(oc[:, :, 149:], on[:, :, 149:])
    assert torch.equal(lc[:, :, 149:], ln[:, :, 149:])
    assert not torch.equal(oc[:, :, :149], on[:, :, :149])
