"""The C-ABI library builds, loads without a GPU, exports every declared symbol,
and rejects bad arguments before touching CUDA (no compute call here)."""
import os
import re

import pytest
import torch

from exact_attention_20_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_gb300.h")


@pytest.fixture(scope="module")
def fa():
    fa_build.build()
    from exact_attention_20_gb300 import fa as mod
    mod.lib()
    return mod


def declared_functions():
    with open(HEADER) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    return sorted(set(re.findall(r"\b(fa_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert names == ["fa_bwd", "fa_fwd", "fa_fwd_fp8", "fa_fwd_noalloc", "fa_fwd_plan", "fa_fwd_rect",
                     "fa_get_device_status", "fa_quantize_fp8", "fa_release_stream", "fa_strerror", "fa_version",
                     "fa_watchdog_selftest"]


def test_library_exports_every_declared_symbol(fa):
    lib = fa.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(fa.SIGNATURES)


def test_version_and_strerror(fa):
    assert fa.version() == 100
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        msg = fa.strerror(code)
        assert msg.startswith("FA_")
    assert fa.strerror(12345) == "unknown fa status code"


# Fake, 256-byte aligned, far-apart addresses: every call below fails its host
# checks before any CUDA call, so nothing is dereferenced.
A = 1 << 40
STEP = 1 << 36
Q, K, V, O, L = (A + i * STEP for i in range(5))


@pytest.mark.parametrize("B,H,N,d,causal,scale", [
    (0, 1, 128, 64, 0, 0.125), (1, 0, 128, 64, 0, 0.125), (1, 1, 0, 64, 0, 0.125),
    (1, 1, -5, 64, 0, 0.125), (1, 1, 128, 32, 0, 0.125), (1, 1, 128, 96, 0, 0.125),
    (1, 1, 128, 256, 0, 0.125), (1, 1, 128, 64, 2, 0.125), (1, 1, 128, 64, -1, 0.125),
    (1, 1, 128, 64, 0, 0.0), (1, 1, 128, 64, 0, -0.5), (1, 1, 128, 64, 0, float("inf")),
    (1, 1, 128, 64, 0, float("nan")), (1 << 12, 1 << 12, 1 << 10, 128, 0, 0.1),
])
def test_invalid_arguments(fa, B, H, N, d, causal, scale):
    assert fa.fa_fwd_raw(Q, K, V, O, L, B, H, N, d, causal, scale) == fa.FA_ERR_INVALID_ARG


def test_null_pointers(fa):
    for i in range(5):
        ptrs = [Q, K, V, O, L]
        ptrs[i] = 0
        assert fa.fa_fwd_raw(*ptrs, 1, 2, 256, 64, 0, 0.125) == fa.FA_ERR_NULL


def test_misaligned_pointers(fa):
    for i in range(4):
        ptrs = [Q, K, V, O, L]
        ptrs[i] += 8
        assert fa.fa_fwd_raw(*ptrs, 1, 2, 256, 64, 0, 0.125) == fa.FA_ERR_ALIGN
    assert fa.fa_fwd_raw(Q, K, V, O, L + 2, 1, 2, 256, 64, 0, 0.125) == fa.FA_ERR_ALIGN


def test_aliasing_outputs(fa):
    nbytes = 1 * 2 * 256 * 64 * 2
    assert fa.fa_fwd_raw(Q, K, V, Q, L, 1, 2, 256, 64, 0, 0.125) == fa.FA_ERR_ALIAS
    assert fa.fa_fwd_raw(Q, K, V, K + nbytes - 16, L, 1, 2, 256, 64, 0, 0.125) == fa.FA_ERR_ALIAS
    assert fa.fa_fwd_raw(Q, K, V, O, V + 64, 1, 2, 256, 64, 0, 0.125) == fa.FA_ERR_ALIAS
    assert fa.fa_fwd_raw(Q, K, V, O, O + nbytes - 4, 1, 2, 256, 64, 0, 0.125) == fa.FA_ERR_ALIAS
    # touching but not overlapping is fine for the host checks; the call then
    # goes on to the device, so only where there is none (fake pointers)
    if not torch.cuda.is_available():
        rc = fa.fa_fwd_raw(Q, K, V, Q + nbytes, L, 1, 2, 256, 64, 0, 0.125)
        assert rc != fa.FA_ERR_ALIAS


@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on fake pointers")
def test_valid_call_without_a_device_fails_loudly(fa):
    rc = fa.fa_fwd_raw(Q, K, V, O, L, 1, 2, 256, 64, 0, 0.125)
    assert rc in (fa.FA_ERR_LAUNCH, fa.FA_ERR_DEVICE)


def test_binding_refuses_cpu_tensors(fa):
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.attention(q, q, q)


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU-only check")
def test_binding_has_no_cpu_fallback(fa, monkeypatch):
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "LIB_PATH", "/nonexistent/libfa_gb300.so")
    with pytest.raises(RuntimeError):
        fa.lib()


def test_plan_query_checks_its_arguments(fa):
    import ctypes

    a, b = ctypes.c_int(0), ctypes.c_int(0)
    pa, pb = ctypes.addressof(a), ctypes.addressof(b)
    assert fa.lib().fa_fwd_plan(1, 32, 4096, 4096, 128, 0, None, pb) == fa.FA_ERR_NULL
    assert fa.lib().fa_fwd_plan(1, 32, 4096, 4096, 128, 0, pa, None) == fa.FA_ERR_NULL
    for args in ((0, 1, 128, 128, 64, 0), (1, 1, 0, 128, 64, 0), (1, 1, 128, 0, 64, 0),
                 (1, 1, 128, 128, 96, 0), (1, 1, 128, 128, 64, 2),
                 (1 << 12, 1 << 12, 1 << 12, 1, 128, 0), (1, 1, 1, 1 << 30, 128, 0)):
        assert fa.lib().fa_fwd_plan(*args, pa, pb) == fa.FA_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU-only check")
def test_plan_query_without_a_device_fails_loudly(fa):
    with pytest.raises(fa.FAError):
        fa.plan(1, 32, 4096, 128, False)


def test_noalloc_entry_checks_arguments_like_fa_fwd(fa):
    # the host checks run before any CUDA call, with the same codes as fa_fwd
    raw = fa.lib().fa_fwd_noalloc
    assert raw(Q, K, V, O, L, 0, 1, 128, 64, 0, 0.125, None) == fa.FA_ERR_INVALID_ARG
    assert raw(Q, K, V, O, L, 1, 1, 128, 96, 0, 0.125, None) == fa.FA_ERR_INVALID_ARG
    assert raw(None, K, V, O, L, 1, 2, 256, 64, 0, 0.125, None) == fa.FA_ERR_NULL
    assert raw(Q + 8, K, V, O, L, 1, 2, 256, 64, 0, 0.125, None) == fa.FA_ERR_ALIGN
    assert raw(Q, K, V, Q, L, 1, 2, 256, 64, 0, 0.125, None) == fa.FA_ERR_ALIAS


@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on fake pointers")
def test_noalloc_entry_without_a_device_fails_loudly(fa):
    rc = fa.lib().fa_fwd_noalloc(Q, K, V, O, L, 1, 2, 256, 64, 0, 0.125, None)
    assert rc in (fa.FA_ERR_LAUNCH, fa.FA_ERR_DEVICE)


def test_noalloc_scratch_size_is_stated_in_the_header():
    import re as _re

    with open(HEADER) as f:
        text = f.read()
    ctas = int(_re.search(r"#define FA_NOALLOC_MAX_CTAS (\d+)", text).group(1))
    assert ctas == 160
    assert "42,278,912 bytes" in text and (ctas * 2 * 256 * 129 + 2048) * 4 == 42278912


def test_rect_entry_checks_arguments(fa):
    raw = fa.lib().fa_fwd_rect
    # q, o: [1][2][64][64]; k, v: [1][2][512][64] -- sizes in bytes
    qb, kb = 1 * 2 * 64 * 64 * 2, 1 * 2 * 512 * 64 * 2
    assert raw(Q, K, V, O, L, 1, 2, 0, 512, 64, 0, 0.125, None) == fa.FA_ERR_INVALID_ARG
    assert raw(Q, K, V, O, L, 1, 2, 64, 0, 64, 0, 0.125, None) == fa.FA_ERR_INVALID_ARG
    assert raw(Q, None, V, O, L, 1, 2, 64, 512, 64, 0, 0.125, None) == fa.FA_ERR_NULL
    assert raw(Q, K + 8, V, O, L, 1, 2, 64, 512, 64, 0, 0.125, None) == fa.FA_ERR_ALIGN
    # o overlapping the tail of k counts with k's own (longer) extent
    assert raw(Q, K, V, K + kb - 16, L, 1, 2, 64, 512, 64, 0, 0.125, None) == fa.FA_ERR_ALIAS
    assert raw(Q, K, V, Q + qb - 16, L, 1, 2, 64, 512, 64, 0, 0.125, None) == fa.FA_ERR_ALIAS
    if not torch.cuda.is_available():  # past the host checks the call reaches the device
        rc = raw(Q, K, V, Q + qb, L, 1, 2, 64, 512, 64, 0, 0.125, None)  # just past q: no alias
        assert rc != fa.FA_ERR_ALIAS


def test_bwd_entry_checks_arguments(fa):
    raw = fa.lib().fa_bwd
    # q, o, do, dq: [1][2][64][64]; k, v, dk, dv: [1][2][512][64]
    qb, kb = 1 * 2 * 64 * 64 * 2, 1 * 2 * 512 * 64 * 2
    DO, DQ, DK, DV = (A + i * STEP for i in range(5, 9))
    args = [Q, K, V, O, L, DO, DQ, DK, DV]

    def call(*ptrs, B=1, H=2, Nq=64, Nk=512, d=64, causal=0, scale=0.125):
        return raw(*ptrs, B, H, Nq, Nk, d, causal, scale, None)

    assert call(*args, Nq=0) == fa.FA_ERR_INVALID_ARG
    assert call(*args, Nk=-1) == fa.FA_ERR_INVALID_ARG
    assert call(*args, d=96) == fa.FA_ERR_INVALID_ARG
    assert call(*args, causal=3) == fa.FA_ERR_INVALID_ARG
    assert call(*args, scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert call(*args, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert call(*args, B=65536, H=1, Nq=1, Nk=1) == fa.FA_ERR_INVALID_ARG   # more heads than the grid takes
    # with the mask the key blocks take the grid's y dimension: at most 65535 of 128 keys
    assert call(*args, B=1, H=1, Nq=1, Nk=65535 * 128 + 1, causal=1) == fa.FA_ERR_INVALID_ARG
    for i in range(9):
        bad = list(args)
        bad[i] = None
        assert call(*bad) == fa.FA_ERR_NULL, i
    for i in range(9):
        bad = list(args)
        bad[i] = args[i] + (2 if i == 4 else 8)
        assert call(*bad) == fa.FA_ERR_ALIGN, i
    # every output against every input and the other outputs
    bad = list(args)
    bad[6] = O + qb - 16                      # dq over the tail of o
    assert call(*bad) == fa.FA_ERR_ALIAS
    bad = list(args)
    bad[7] = V + kb - 16                      # dk over the tail of v
    assert call(*bad) == fa.FA_ERR_ALIAS
    bad = list(args)
    bad[8] = DK + 16                          # dv over dk
    assert call(*bad) == fa.FA_ERR_ALIAS
    bad = list(args)
    bad[8] = L                                # dv over lse
    assert call(*bad) == fa.FA_ERR_ALIAS


def test_fp8_entries_check_arguments(fa):
    fwd, quant = fa.lib().fa_fwd_fp8, fa.lib().fa_quantize_fp8
    Q8, K8, V8, SQ, SK, SV = (A + i * STEP for i in range(9, 15))
    args = [Q8, K8, V8, SQ, SK, SV, O, L]

    def call(*ptrs, B=1, H=2, N=256, d=128, causal=0, scale=0.125):
        return fwd(*ptrs, B, H, N, d, causal, scale, None)

    assert call(*args, d=64) == fa.FA_ERR_INVALID_ARG      # the FP8 path takes d = 128
    assert call(*args, N=0) == fa.FA_ERR_INVALID_ARG
    assert call(*args, causal=2) == fa.FA_ERR_INVALID_ARG
    assert call(*args, scale=-1.0) == fa.FA_ERR_INVALID_ARG
    for i in range(8):
        bad = list(args)
        bad[i] = None
        assert call(*bad) == fa.FA_ERR_NULL, i
        bad = list(args)
        bad[i] = args[i] + (2 if i >= 3 and i != 6 else 8)
        assert call(*bad) == fa.FA_ERR_ALIGN, i
    bad = list(args)
    bad[6] = Q8 + 64                                        # o over the codes of q
    assert call(*bad) == fa.FA_ERR_ALIAS
    bad = list(args)
    bad[7] = SV                                             # lse over v's scales
    assert call(*bad) == fa.FA_ERR_ALIAS
    assert quant(Q, Q8, SQ, 1, 2, 256, 96, 0, None) == fa.FA_ERR_INVALID_ARG
    assert quant(Q, Q8, SQ, 1, 2, 256, 128, 2, None) == fa.FA_ERR_INVALID_ARG
    assert quant(None, Q8, SQ, 1, 2, 256, 128, 0, None) == fa.FA_ERR_NULL
    assert quant(Q, Q8 + 8, SQ, 1, 2, 256, 128, 0, None) == fa.FA_ERR_ALIGN
    assert quant(Q, Q + 64, SQ, 1, 2, 256, 128, 0, None) == fa.FA_ERR_ALIAS
