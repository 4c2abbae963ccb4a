"""Streams and device memory of the forward's boundary (GPU).

- A call that splits work items on a fresh non-blocking stream: the stream's
  workspace is allocated and its arrival counters cleared on that stream, so
  the kernel that follows on it sees them cleared; its output is compared
  with the oracle on sampled heads and bit for bit with the same call on the
  current stream.
- fa_release_stream frees a stream's workspaces, and the next call on the
  stream allocates them again.
- Nothing of size N x N is allocated: one causal call at 32,768 tokens (B1,
  H32, d128) on a fresh stream takes at most the documented per-stream
  workspace from the device (about 40 MB), against 4.3 GB for one head's
  fp32 score matrix ("FlashAttention and kernels.", "Build It", where the
  peak memory of each call is measured).
"""
import numpy as np
import pytest
import torch

from exact_attention_20_gb300 import build as fa_build
from exact_attention_20_gb300.inputs import make_workload
from tests.parity import assert_close, compare, oracle_sampled

pytestmark = pytest.mark.gpu
DEV = "cuda"
MiB = 1 << 20


@pytest.fixture(scope="module")
def fa():
    fa_build.build()
    from exact_attention_20_gb300 import fa as mod
    mod.lib()
    return mod


def _workspace_bytes():
    sms = min(torch.cuda.get_device_properties(0).multi_processor_count, 256)
    return (2 * sms * 256 * 129 + 2048) * 4


@pytest.mark.parametrize("causal", [False, True])
def test_split_items_on_a_fresh_nonblocking_stream(fa, causal):
    name = "B1-H32-N4096-d128"
    q, k, v = make_workload(name, seed=3, device=DEV)
    assert fa.plan(1, 32, 4096, 128, causal)[1] > 0, "the call must split items"
    o_ref, l_ref = fa.attention(q, k, v, causal=causal, scale=128 ** -0.5)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()  # from torch's pool: created non-blocking
    # keep the legacy default stream busy meanwhile, so that a clear queued
    # there would still be pending when the kernel on `s` starts
    busy = torch.empty(256 * MiB, dtype=torch.uint8, device=DEV)
    with torch.cuda.stream(torch.cuda.default_stream()):
        for _ in range(20):
            busy.add_(1)
    with torch.cuda.stream(s):
        o, lse = fa.attention(q, k, v, causal=causal, scale=128 ** -0.5, stream=s)
    s.synchronize()
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    rng = np.random.default_rng(7)
    sample = [(0, h, sorted(rng.choice(4096, 48, replace=False).tolist()) + [0, 127, 128, 255, 4095])
              for h in (0, 17, 31)]
    for (b, h, rows), (o64, l64) in zip(sample, oracle_sampled(q, k, v, 128 ** -0.5, causal, sample)):
        st = compare(o[b, h, rows], lse[b, h, rows], o64, l64)
        assert_close(st, f"fresh stream head {h} causal={causal}")
    fa.release_stream(s)


def test_release_stream_frees_and_reallocates(fa):
    q, k, v = make_workload("B1-H32-N4096-d128", seed=4, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = fa.attention(q, k, v, causal=False, scale=128 ** -0.5, stream=s)
    s.synchronize()
    free_with = torch.cuda.mem_get_info()[0]
    fa.release_stream(s)
    free_without = torch.cuda.mem_get_info()[0]
    assert free_without - free_with >= _workspace_bytes() - 4 * MiB
    with torch.cuda.stream(s):
        o2, l2 = fa.attention(q, k, v, causal=False, scale=128 ** -0.5, stream=s)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    fa.release_stream(s)
    fa.release_stream(s)  # releasing twice is harmless


def test_no_quadratic_allocation_at_32k_tokens(fa):
    name = "B1-H32-N32768-d128"
    q, k, v = make_workload(name, seed=0, device=DEV)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    torch_before = torch.cuda.max_memory_allocated()
    free_before = torch.cuda.mem_get_info()[0]
    with torch.cuda.stream(s):
        fa.fa_fwd(q, k, v, o, lse, causal=True, scale=128 ** -0.5, stream=s)
    s.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    taken = free_before - free_after
    print(f"\n32K causal: device memory taken by the call {taken / MiB:.1f} MiB; "
          f"torch peak unchanged: {torch.cuda.max_memory_allocated() == torch_before}; "
          f"one head's fp32 N x N scores would be {32768 ** 2 * 4 / MiB:.0f} MiB")
    assert torch.cuda.max_memory_allocated() == torch_before
    assert taken <= _workspace_bytes() + 8 * MiB
    assert torch.isfinite(o.float()).all() and torch.equal(o[:, :, 0], v[:, :, 0])
    fa.release_stream(s)
