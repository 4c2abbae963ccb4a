"""GPU parity of fa_bwd: dQ, dK, dV against the fp64 backward oracle.

The GPU path runs as a training step would: fa_fwd_rect gives O and LSE,
then fa_bwd takes them with the upstream gradient dO.  The oracle computes
the exact gradients of the forward definition from the same bf16 Q, K, V and
dO alone (none of its inputs comes from the GPU).  Every element of every
gradient is compared (tolerances in tests/parity.py); at full size the
oracle covers sampled heads.  The shapes cover one tile, ragged query and key
tails, more keys than queries and the reverse, a single query row and a
single key, both head sizes and both masks.
"""
import numpy as np
import pytest
import torch

from exact_attention_20_gb300 import build as fa_build
from exact_attention_20_gb300.inputs import make_grad, make_qkv
from tests.parity import (GRAD_EXACT_PEAKY_MAX_REL, GRAD_EXACT_PEAKY_MEAN_REL, assert_grads_close,
                          compare_grad, round_bf16, to_f64)

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
    do = make_grad(B, H, Nq, d, seed=seed + 2, device=DEV)
    return q, k, v, do


def _gpu(fa, q, k, v, do, causal, scale):
    o, lse = fa.attention_rect(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return dq, dk, dv


def _stats(got, want):
    return {name: compare_grad(g, w) for name, g, w in zip(("dq", "dk", "dv"), got, want)}


SHAPES = [
    (1, 1, 64, 128, 128),       # one step, one key block
    (1, 2, 256, 256, 64),       # several steps and key blocks
    (2, 3, 300, 300, 128),      # ragged query and key tails
    (1, 2, 200, 333, 128),      # more keys than queries
    (1, 2, 333, 200, 64),       # more queries than keys
]


@pytest.mark.parametrize("B,H,Nq,Nk,d", SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_every_element(fa, B, H, Nq, Nk, d, causal):
    q, k, v, do = _inputs(B, H, Nq, Nk, d, seed=50)
    scale = d ** -0.5
    got = _gpu(fa, q, k, v, do, causal, scale)
    want = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
    stats = _stats(got, want)
    print(f"\nbwd {B}x{H} {Nq}x{Nk} d{d} causal={causal}: " +
          ", ".join(f"{n} max {s['max_rel']:.2e} mean {s['mean_rel']:.2e}" for n, s in stats.items()))
    assert_grads_close(stats, f"bwd {Nq}x{Nk} d{d} causal={causal}")


def test_bwd_one_query_row(fa):
    q, k, v, do = _inputs(1, 2, 1, 130, 128, seed=50)
    got = _gpu(fa, q, k, v, do, False, 128 ** -0.5)
    want = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), 128 ** -0.5, False)
    assert_grads_close(_stats(got, want), "one query row")


@pytest.mark.parametrize("Nq,Nk,causal", [(130, 1, False), (130, 1, True), (1, 130, True)])
def test_bwd_single_visible_key(fa, Nq, Nk, causal):
    # Every row sees one key (one key in all; or, causal, one query row, which
    # sees key 0 only): the softmax is the constant 1 and O = v_0 whatever Q and
    # K are.  The exact dQ and dK are 0 (the GPU leaves the fp32 rounding of
    # dP - D, dP and D being summed in different orders), dV_0 is the sum of
    # dO's rows and every other dV row is 0.
    q, k, v, do = _inputs(1, 2, Nq, Nk, 64, seed=56)
    dq, dk, dv = _gpu(fa, q, k, v, do, causal, 0.125)
    bound = 1e-5 * do.float().abs().max().item() * v.float().abs().max().item()
    assert dq.float().abs().max().item() <= bound and dk.float().abs().max().item() <= bound
    want = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), 0.125, causal)
    assert_grads_close({"dv0": compare_grad(dv[:, :, :1], want[2][:, :, :1])}, "single key")
    assert torch.count_nonzero(dv[:, :, 1:]) == 0


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_b4_h16_n1024_d64(fa, causal):
    q, k, v, do = _inputs(4, 16, 1024, 1024, 64, seed=51)
    got = _gpu(fa, q, k, v, do, causal, 0.125)
    want = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), 0.125, causal)
    stats = _stats(got, want)
    print(f"\nbwd B4-H16-N1024-d64 causal={causal}: {stats}")
    assert_grads_close(stats, "B4-H16-N1024-d64")


@pytest.mark.parametrize("name,B,H,N,d,values", [
    ("B1-H32-N4096-d128", 1, 32, 4096, 128, "normal"),
    ("B2-H8-N3001-d128-outliers", 2, 8, 3001, 128, "outliers"),
])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_full_size_sampled_heads(fa, name, B, H, N, d, values, causal):
    q, k, v, do = _inputs(B, H, N, N, d, seed=52, values=values)
    scale = d ** -0.5
    dq, dk, dv = _gpu(fa, q, k, v, do, causal, scale)
    for b, h in [(0, 0), (B - 1, H - 1)]:
        args = [to_f64(t[b, h]) for t in (q, k, v, do)]
        got = (dq[b, h], dk[b, h], dv[b, h])
        exact = _stats(got, oracle.attention_backward(*args, scale, causal))
        print(f"\nbwd {name} head {b},{h} causal={causal} vs exact: {exact}")
        if values == "normal":
            assert_grads_close(exact, f"{name} head {b},{h}")
            continue
        # peaky softmax: the kernel against the recompute-from-L backward on the
        # oracle's own O stored in bf16, and the exact gradient under looser bounds
        o_ref, lse_ref = oracle.attention(args[0], args[1], args[2], scale, causal)
        alg = oracle.tiled_attention_backward(args[0], args[1], args[2], round_bf16(o_ref), lse_ref,
                                              args[3], scale, causal, Br=512, Bc=512)
        at_bf16_o = _stats(got, alg)
        print(f"bwd {name} head {b},{h} causal={causal} vs bf16-O recompute: {at_bf16_o}")
        assert_grads_close(at_bf16_o, f"{name} head {b},{h} (bf16 O)")
        assert_grads_close(exact, f"{name} head {b},{h} (exact)", GRAD_EXACT_PEAKY_MAX_REL,
                           GRAD_EXACT_PEAKY_MEAN_REL)


def test_bwd_outputs_inside_guard_bands(fa):
    B, H, Nq, Nk, d = 1, 2, 77, 150, 128
    q, k, v, do = _inputs(B, H, Nq, Nk, d, seed=53)
    o, lse = fa.attention_rect(q, k, v, causal=True)
    G = 4096
    bufs = {}
    views = {}
    for name, n in (("dq", B * H * Nq * d), ("dk", B * H * Nk * d), ("dv", B * H * Nk * d)):
        bufs[name] = torch.full((n + 2 * G,), -512.0, dtype=torch.bfloat16, device=DEV)
        rows = Nq if name == "dq" else Nk
        views[name] = bufs[name][G:G + n].view(B, H, rows, d)
    fa.fa_bwd(q, k, v, o, lse, do, views["dq"], views["dk"], views["dv"], causal=True)
    torch.cuda.synchronize()
    for name, buf in bufs.items():
        assert (buf[:G] == -512.0).all() and (buf[-G:] == -512.0).all(), name
    want = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), d ** -0.5, True)
    assert_grads_close(_stats((views["dq"], views["dk"], views["dv"]), want), "guarded")


def test_bwd_keys_past_every_query_get_zero_gradients(fa):
    # causal, Nk > Nq: key blocks beyond the last query row are seen by no row
    q, k, v, do = _inputs(1, 2, 100, 600, 64, seed=54)
    dq, dk, dv = _gpu(fa, q, k, v, do, True, 0.125)
    assert torch.count_nonzero(dk[:, :, 100:]) == 0 and torch.count_nonzero(dv[:, :, 100:]) == 0
    assert torch.count_nonzero(dv[:, :, :100]) > 0


def test_bwd_repeated_calls_agree(fa):
    # dK and dV are summed in a fixed order; dQ's fp32 sum may differ in its last bits
    q, k, v, do = _inputs(1, 4, 512, 512, 128, seed=55)
    a = _gpu(fa, q, k, v, do, False, 0.1)
    b = _gpu(fa, q, k, v, do, False, 0.1)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert (a[0].float() - b[0].float()).abs().max().item() <= 2.0 ** -6 * a[0].float().abs().max().item()
