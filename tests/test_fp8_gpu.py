"""GPU parity of the FP8 path: the quantiser and the FP8 forward.

The quantiser is byte and integer work: its e4m3 codes and fp32 scales must
equal the oracle's exactly (the division x / s is fp32 on both sides).  The
FP8 forward is compared, element by element, with the oracle's attention on
the dequantised inputs, which the oracle quantises itself from the same bf16
tensors.  Beyond that definition the kernel rounds P to e4m3 before P.V
(relative error up to 2^-4 per weight), which sets the tolerance on O; the
LSE comes from unrounded sums and keeps the bf16 path's bound.
"""
import numpy as np
import pytest
import torch

from exact_attention_20_gb300 import build as fa_build
from exact_attention_20_gb300.inputs import make_qkv
from tests.parity import BF16_FINE, round_bf16, to_f64

import oracle
from oracle import fp8 as ofp8

pytestmark = pytest.mark.gpu
DEV = "cuda"

# O tolerance: P in e4m3 moves each weight of the average by up to 2^-4
# relative (round to nearest), so the output by at most 2^-4 of the spread of
# the value rows it averages, and the weights' errors are independent, so
# over many keys they mostly cancel.  The bounds are in units of max |V|:
# 2^-5 for the maximum and 2^-9 for the mean, about twice the largest
# errors measured on these workloads (1.5 % and 0.07 % of max |V|).
# As for the bf16 path, the plain difference is bounded where |O| < 2 and
# the error beyond the output's own bf16 rounding where |O| >= 2; the mean
# is the plain one.
FP8_MAX_DO = 2.0 ** -5
FP8_MEAN_DO = 2.0 ** -9
FP8_MAX_DLSE = 1e-3


@pytest.fixture(scope="module")
def fa():
    fa_build.build()
    from exact_attention_20_gb300 import fa as mod
    mod.lib()
    return mod


def _codes_bytes(vals):
    """float64 e4m3 values -> their bytes (exact: every value is on the grid)."""
    t = torch.from_numpy(np.ascontiguousarray(vals, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


@pytest.mark.parametrize("B,H,N,d", [(1, 2, 256, 128), (2, 3, 300, 128), (1, 2, 1000, 64), (1, 1, 5, 128)])
@pytest.mark.parametrize("values", ["normal", "outliers"])
def test_quantiser_is_bit_exact(fa, B, H, N, d, values):
    x, _, _ = make_qkv(B, H, N, d, seed=60, values=values, device=DEV)
    x[0, 0, : min(N, 128)] = 0  # an all-zero block: scale 1, codes 0
    xf = to_f64(x)
    # mode 0: one scale per 128 rows, row layout
    x8, s = fa.quantize_fp8(x, 0)
    codes, scales = ofp8.quantize_blocks(xf, 128)
    assert np.array_equal(s.cpu().numpy(), scales)
    assert np.array_equal(x8.cpu().numpy(), _codes_bytes(codes))
    # mode 1: one scale per head, transposed, keys padded with zeros
    vt8, sv = fa.quantize_fp8(x, 1)
    codes_v, scales_v = ofp8.quantize_blocks(xf, N)
    assert np.array_equal(sv.cpu().numpy(), scales_v[..., 0])
    n_pad = vt8.shape[-1]
    want = np.zeros((B, H, d, n_pad), dtype=np.uint8)
    want[..., :N] = np.swapaxes(_codes_bytes(codes_v), -1, -2)
    assert np.array_equal(vt8.cpu().numpy(), want)


def _oracle_fp8(q, k, v, scale, causal):
    qf, kf, vf = to_f64(q), to_f64(k), to_f64(v)
    n = qf.shape[-2]
    q8, sq = ofp8.quantize_blocks(qf, 128)
    k8, sk = ofp8.quantize_blocks(kf, 128)
    v8, sv = ofp8.quantize_blocks(vf, n)
    return ofp8.attention_fp8(q8, sq, k8, sk, v8, sv, scale, causal), ofp8.dequantize_blocks(v8, sv, n)


def _compare(o, lse, o_ref, lse_ref, v_deq, label):
    og, lg = to_f64(o), to_f64(lse)
    vmax = np.abs(v_deq).max()
    d_raw = np.abs(og - o_ref)
    excess = d_raw - np.abs(round_bf16(o_ref) - o_ref)
    d_o = np.where(np.abs(o_ref) < BF16_FINE, d_raw, excess) / vmax
    d_l = np.abs(lg - lse_ref)
    stats = {"max_do_rel_vmax": float(d_o.max()), "mean_do_rel_vmax": float(d_raw.mean() / vmax),
             "max_dlse": float(d_l.max()), "nan": bool(np.isnan(og).any())}
    print(f"\nfp8 {label}: {stats}")
    assert not stats["nan"], label
    assert stats["max_do_rel_vmax"] <= FP8_MAX_DO, (label, stats)
    assert stats["mean_do_rel_vmax"] <= FP8_MEAN_DO, (label, stats)
    assert stats["max_dlse"] <= FP8_MAX_DLSE, (label, stats)
    return stats


@pytest.mark.parametrize("B,H,N", [(1, 2, 256), (2, 3, 300), (1, 4, 1000), (1, 1, 1), (1, 2, 129), (1, 4, 100), (1, 320, 100)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_every_element(fa, B, H, N, causal):
    q, k, v = make_qkv(B, H, N, 128, seed=61, device=DEV)
    scale = 128 ** -0.5
    o, lse = fa.attention_fp8(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    (o_ref, lse_ref), v_deq = _oracle_fp8(q, k, v, scale, causal)
    _compare(o, lse, o_ref, lse_ref, v_deq, f"{B}x{H}x{N} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_headline_sampled_heads(fa, causal):
    q, k, v = make_qkv(1, 32, 4096, 128, seed=62, device=DEV)
    scale = 128 ** -0.5
    o, lse = fa.attention_fp8(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    for h in (0, 31):
        (o_ref, lse_ref), v_deq = _oracle_fp8(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], scale, causal)
        _compare(o[:, h:h + 1], lse[:, h:h + 1], o_ref, lse_ref, v_deq, f"headline head {h} causal={causal}")


def test_fp8_forward_outliers(fa):
    q, k, v = make_qkv(2, 8, 3001, 128, seed=63, values="outliers", device=DEV)
    scale = 128 ** -0.5
    o, lse = fa.attention_fp8(q, k, v, causal=True, scale=scale)
    torch.cuda.synchronize()
    (o_ref, lse_ref), v_deq = _oracle_fp8(q[:1, :2], k[:1, :2], v[:1, :2], scale, True)
    _compare(o[:1, :2], lse[:1, :2], o_ref, lse_ref, v_deq, "outliers B2-H8-N3001 (2 heads)")


def test_fp8_close_to_bf16_forward(fa):
    # context, not the parity bar: FP8 against the exact bf16-input result
    q, k, v = make_qkv(1, 4, 1024, 128, seed=64, device=DEV)
    o8, _ = fa.attention_fp8(q, k, v, causal=False)
    o16, _ = fa.attention(q, k, v, causal=False)
    torch.cuda.synchronize()
    err = (o8.float() - o16.float()).abs()
    print(f"\nfp8 vs bf16 forward: max {err.max().item():.3g} mean {err.mean().item():.3g}")
    assert err.mean().item() < 0.05 * o16.float().abs().mean().item() + 1e-3
