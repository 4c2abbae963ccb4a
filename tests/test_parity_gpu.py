"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small and medium workloads are compared on every element; the 32K-token
causal workload is compared on sampled rows that the oracle evaluates one by
one, plus properties that hold at any size.  Edge lengths cover empty-ish,
single-tile, tile-boundary and ragged sequences for both head dimensions.
"""
import numpy as np
import pytest
import torch

from exact_attention_20_gb300 import build as fa_build
from exact_attention_20_gb300.inputs import WORKLOADS, make_qkv, make_workload
from tests.parity import assert_close, compare, oracle_full, oracle_sampled, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def fa():
    fa_build.build()
    from exact_attention_20_gb300 import fa as mod
    mod.lib()
    return mod


def run(fa, q, k, v, causal, scale):
    o, lse = fa.attention(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o, lse


FULL = ["B1-H2-N256-d64", "B4-H16-N1024-d64", "B2-H8-N3001-d128-outliers", "B1-H32-N4096-d128"]


@pytest.mark.parametrize("name,causal", [(n, c) for n in FULL for c in WORKLOADS[n].causal])
def test_workload_every_element(fa, name, causal):
    w = WORKLOADS[name]
    q, k, v = make_workload(name, seed=0, device=DEV)
    o, lse = run(fa, q, k, v, causal, w.scale)
    o_ref, lse_ref = oracle_full(q, k, v, w.scale, causal)
    st = compare(o, lse, o_ref, lse_ref)
    print(name, "causal" if causal else "non-causal", st)
    assert_close(st, name)


def test_long_context_sampled_rows(fa):
    name = "B1-H32-N32768-d128"
    w = WORKLOADS[name]
    q, k, v = make_workload(name, seed=0, device=DEV)
    o, lse = run(fa, q, k, v, True, w.scale)
    # properties at any size: finite everywhere; causal row 0 is exactly V[0]
    assert torch.isfinite(lse).all()
    assert torch.isfinite(o.float()).all()
    assert torch.equal(o[:, :, 0], v[:, :, 0])
    s00 = (q[:, :, 0].float() * k[:, :, 0].float()).sum(-1) * w.scale
    assert (lse[:, :, 0] - s00).abs().max().item() <= 1e-3
    rng = np.random.default_rng(5)
    fixed = [0, 1, 127, 128, 129, 255, 256, 8191, 16384, 32639, 32640, w.N - 2, w.N - 1]
    sample = []
    for h in (0, 13, 31):
        rows = sorted(set(fixed) | set(rng.integers(0, w.N, 24).tolist()))
        sample.append((0, h, rows))
    refs = oracle_sampled(q, k, v, w.scale, True, sample)
    for (b, h, rows), (o_ref, lse_ref) in zip(sample, refs):
        st = compare(o[b, h, rows], lse[b, h, rows], o_ref, lse_ref)
        print(name, "head", h, st)
        assert_close(st, f"{name} head {h}")


EDGE_N = [1, 2, 3, 64, 127, 128, 129, 255, 256, 257, 383, 384, 385, 640, 1000]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", EDGE_N)
def test_edge_lengths(fa, N, d, causal):
    q, k, v = make_qkv(1, 2, N, d, seed=N + d, device=DEV)
    scale = d ** -0.5
    o, lse = run(fa, q, k, v, causal, scale)
    st = compare(o, lse, *oracle_full(q, k, v, scale, causal))
    assert_close(st, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("B,H,N,d", [(3, 5, 300, 64), (2, 3, 129, 128), (1, 1, 2048, 128), (5, 1, 513, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_batch_head_indexing(fa, B, H, N, d, causal):
    q, k, v = make_qkv(B, H, N, d, seed=B * 100 + H, device=DEV)
    o, lse = run(fa, q, k, v, causal, 0.1)
    assert_close(compare(o, lse, *oracle_full(q, k, v, 0.1, causal)), f"{B}x{H}x{N}x{d}")


# Keys of 1.5 in the last tile raise each row's maximum there by about 20
# (d = 128) or 10 (d = 64) log2 units: below the bf16 path's rescale threshold
# of 32, so P grows past 1 against the old reference and nothing is rescaled.
# Keys of 5.0 raise it by about 65 or 46 and keys of 8.0 by about 105 or 74:
# the reference moves, the tile is exponentiated again and the accumulator
# rescaled.
@pytest.mark.parametrize("k_last", [1.5, 5.0, 8.0])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_max_in_last_key_tile(fa, d, causal, k_last):
    # the largest scores of every row sit in the last key tile, so a missing
    # rescale of the accumulator fails loudly (Break It #2 of the gtadkapally lesson)
    N = 1000
    q, k, v = make_qkv(1, 2, N, d, seed=77, device=DEV)
    q = q.float().abs().to(torch.bfloat16)
    k = k.clone()
    k[:, :, N - 8:, :] = k_last
    o, lse = run(fa, q, k, v, causal, d ** -0.5)
    assert_close(compare(o, lse, *oracle_full(q, k, v, d ** -0.5, causal)), "max-last")


@pytest.mark.parametrize("k_last", [1.5, 5.0, 8.0])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_max_jumps_in_some_rows_only(fa, d, causal, k_last):
    # even rows see a score jump in the last key tile (see above for its
    # size), odd rows see their smallest scores there: within one warp some
    # rows move their reference maximum and others keep it
    N = 777
    q, k, v = make_qkv(1, 2, N, d, seed=78, device=DEV)
    sign = torch.ones(N, device=DEV)
    sign[1::2] = -1.0
    q = (q.float().abs() * sign[None, None, :, None]).to(torch.bfloat16)
    k = k.clone()
    k[:, :, N - 5:, :] = k_last
    o, lse = run(fa, q, k, v, causal, d ** -0.5)
    assert_close(compare(o, lse, *oracle_full(q, k, v, d ** -0.5, causal)), "jump-some")


@pytest.mark.parametrize("scale", [0.01, 1.0, 3.0])
def test_scale_values(fa, scale):
    q, k, v = make_qkv(1, 2, 500, 64, seed=3, device=DEV)
    o, lse = run(fa, q, k, v, False, scale)
    assert_close(compare(o, lse, *oracle_full(q, k, v, scale, False)), f"scale={scale}")


def test_identical_keys_give_mean_of_visible_values(fa):
    B, H, N, d = 1, 2, 300, 64
    q, k, v = make_qkv(B, H, N, d, seed=4, device=DEV)
    k = k[:, :, :1, :].expand(B, H, N, d).contiguous()
    o, lse = run(fa, q, k, v, True, 0.125)
    vf = to_f64(v)
    mean = np.cumsum(vf, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    d_o = np.abs(to_f64(o) - mean)
    assert d_o.max() <= 1e-2 and d_o.mean() <= 1e-3


@pytest.mark.parametrize("B,H,N,d", [(2, 3, 129, 64), (2, 3, 1000, 128), (2, 3, 256, 128),
                                     (4, 40, 1000, 64), (1, 33, 2304, 128), (1, 10, 4096, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_guard_bands_untouched(fa, B, H, N, d, causal):
    # the last three shapes have more work items than SMs: (4, 40, 1000) and
    # (1, 10, 4096) have items split across CTAs and merged (with 152 SMs,
    # (1, 10, 4096) causal has ranges of about 18 steps against items of up to
    # 32, so some items have three parts); (1, 33, 2304) has short items, which
    # the plan keeps whole, two or three to a CTA
    G = 4096
    q, k, v = make_qkv(B, H, N, d, seed=9, device=DEV)
    n_o, n_l = B * H * N * d, B * H * N
    obuf = torch.full((n_o + 2 * G,), -512.0, dtype=torch.bfloat16, device=DEV)
    lbuf = torch.full((n_l + 2 * G,), -512.0, dtype=torch.float32, device=DEV)
    o = obuf[G:G + n_o].view(B, H, N, d)
    lse = lbuf[G:G + n_l].view(B, H, N)
    fa.fa_fwd(q, k, v, o, lse, causal=causal, scale=0.1)
    torch.cuda.synchronize()
    assert (obuf[:G] == -512.0).all() and (obuf[G + n_o:] == -512.0).all()
    assert (lbuf[:G] == -512.0).all() and (lbuf[G + n_l:] == -512.0).all()
    assert (o != -512.0).all() and (lse != -512.0).all()
    assert_close(compare(o, lse, *oracle_full(q, k, v, 0.1, causal)), "guarded")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_output_only_16_byte_aligned(fa, d, causal):
    # O 16 bytes past a 32-byte boundary: the epilogue must take its 16-byte
    # store path (the API promises 16-byte alignment only)
    B, H, N = 2, 3, 300
    q, k, v = make_qkv(B, H, N, d, seed=12, device=DEV)
    n_o = B * H * N * d
    obuf = torch.full((n_o + 64,), -512.0, dtype=torch.bfloat16, device=DEV)
    assert obuf.data_ptr() % 32 == 0
    o = obuf[8:8 + n_o].view(B, H, N, d)
    assert o.data_ptr() % 32 == 16
    lse = torch.empty((B, H, N), dtype=torch.float32, device=DEV)
    fa.fa_fwd(q, k, v, o, lse, causal=causal, scale=d ** -0.5)
    torch.cuda.synchronize()
    assert (obuf[:8] == -512.0).all() and (obuf[8 + n_o:] == -512.0).all()
    assert_close(compare(o, lse, *oracle_full(q, k, v, d ** -0.5, causal)), "o16")


@pytest.mark.parametrize("causal", [False, True])
def test_bitwise_deterministic(fa, causal):
    q, k, v = make_workload("B2-H8-N3001-d128-outliers", seed=1, device=DEV)
    o1, l1 = run(fa, q, k, v, causal, 128 ** -0.5)
    o2, l2 = run(fa, q, k, v, causal, 128 ** -0.5)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_side_stream_and_ordering(fa):
    q, k, v = make_qkv(2, 4, 777, 128, seed=11, device=DEV)
    ref_o, ref_l = run(fa, q, k, v, True, 0.09)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.attention(q, k, v, causal=True, scale=0.09, stream=s)
        o2 = o.clone()
    s.synchronize()
    assert torch.equal(o2, ref_o) and torch.equal(lse, ref_l)


def test_host_buffers_end_to_end(fa):
    q, k, v = make_qkv(1, 4, 1024, 64, seed=12)
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    oh, lh = fa.attention_host(qh, kh, vh, causal=False, scale=0.125)
    od, ld = run(fa, q.to(DEV), k.to(DEV), v.to(DEV), False, 0.125)
    assert torch.equal(oh, od.cpu()) and torch.equal(lh, ld.cpu())


def test_watchdog_times_out_and_context_survives(fa):
    assert fa.device_status() == fa.FA_OK
    assert fa.watchdog_selftest(limit_ms=100) == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.device_status() == fa.FA_OK
    q, k, v = make_qkv(1, 2, 256, 64, seed=13, device=DEV)
    o, lse = run(fa, q, k, v, True, 0.125)
    assert_close(compare(o, lse, *oracle_full(q, k, v, 0.125, True)), "after watchdog")
    assert fa.device_status() == fa.FA_OK


def test_wrong_shapes_and_dtypes_raise(fa):
    q, k, v = make_qkv(1, 2, 128, 64, device=DEV)
    with pytest.raises(TypeError):
        fa.attention(q.float(), k, v)
    with pytest.raises(ValueError):
        fa.attention(q, k[:, :, :64], v)
    with pytest.raises(ValueError):
        fa.attention(q.transpose(2, 3), k, v)
    with pytest.raises(fa.FAError):
        fa.attention(make_qkv(1, 1, 16, 32, device=DEV)[0], *make_qkv(1, 1, 16, 32, device=DEV)[1:])


def test_plan_reports_the_work_division(fa):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    grid, nsplit = fa.plan(1, 32, 4096, 128, False)  # 512 items of 256 rows
    assert grid == min(sms, 256) and 0 < nsplit <= grid
    assert fa.plan(1, 2, 300, 64, True) == (4, 0)     # 4 items: one CTA each
