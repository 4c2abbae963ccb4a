"""Thin ctypes binding of libfa_gb300.so: argument marshalling only.

Every step of the attention forward and backward runs in the CUDA library; this module
checks tensor metadata, passes raw device pointers and sizes through the C
ABI declared in include/fa_gb300.h, and turns status codes into exceptions.
There is no CPU fallback: without the built library, or on a device other
than a GB300, every compute call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa_gb300.so")

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_NULL = -2
FA_ERR_ALIGN = -3
FA_ERR_ALIAS = -4
FA_ERR_DEVICE = -5
FA_ERR_LAUNCH = -6
FA_ERR_DEVICE_TIMEOUT = -7
FA_ERR_SCRATCH = -8

# every function declared in include/fa_gb300.h, with its ctypes signature
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _P]),
    "fa_fwd_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _P]),
    "fa_fwd_plan": (_I, [_I, _I, _I, _I, _I, _I, _P, _P]),
    "fa_fwd_rect": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P]),
    "fa_quantize_fp8": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "fa_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _P]),
    "fa_strerror": (ctypes.c_char_p, [_I]),
    "fa_get_device_status": (_I, [_P]),
    "fa_release_stream": (_I, [_P]),
    "fa_watchdog_selftest": (_I, [_P, _P, _P, _P, _P, _I, _P]),
    "fa_version": (_I, []),
}

_lib = None


class FAError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        super().__init__(strerror(code) if _lib is not None else f"fa status {code}")


def lib() -> ctypes.CDLL:
    """Loads the CUDA library (once); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; build it with `python -m exact_attention_20_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def strerror(code: int) -> str:
    return lib().fa_strerror(int(code)).decode()


def version() -> int:
    return lib().fa_version()


def fa_fwd_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, d: int,
               causal: int, scale: float, stream: int = 0) -> int:
    """Direct call of the C entry point with integer addresses; returns the status code."""
    return lib().fa_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, stream)


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(name, t, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


def fa_fwd(q, k, v, o, lse, causal: bool = False, scale: float | None = None, stream=None) -> None:
    """O and LSE into caller-owned tensors. q, k, v, o: bf16 [B, H, N, d]; lse: fp32 [B, H, N]."""
    _call("fa_fwd", q, k, v, o, lse, causal, scale, stream)


def fa_fwd_noalloc(q, k, v, o, lse, causal: bool = False, scale: float | None = None,
                   stream=None) -> None:
    """fa_fwd through the entry point that allocates no device memory at any call.

    For callers that cannot let the library allocate once they run (a fixed
    memory budget reserved at start-up, or no tolerance for an allocation
    blocking on other streams).  The split-item parts go to one static
    scratch per device, so calls that overlap on the GPU race on it; calls on
    one stream are ordered.  The first call on a device does that device's
    set-up and should come before any stream capture.
    """
    _call("fa_fwd_noalloc", q, k, v, o, lse, causal, scale, stream)


def _call(entry, q, k, v, o, lse, causal, scale, stream) -> None:
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _check(name, t, torch.bfloat16, (B, H, N, d), dev)
    _check("lse", lse, torch.float32, (B, H, N), dev)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(dev):
        rc = getattr(lib(), entry)(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                   _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc)


def fa_fwd_rect(q, k, v, o, lse, causal: bool = False, scale: float | None = None,
                stream=None) -> None:
    """O and LSE for Nq query rows over Nk keys (top-left causal mask).

    q, o: bf16 [B, H, Nq, d]; k, v: bf16 [B, H, Nk, d]; lse: fp32 [B, H, Nq].
    """
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B, H, Nq, d] and k [B, H, Nk, d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    _check("q", q, torch.bfloat16, (B, H, Nq, d), dev)
    _check("k", k, torch.bfloat16, (B, H, Nk, d), dev)
    _check("v", v, torch.bfloat16, (B, H, Nk, d), dev)
    _check("o", o, torch.bfloat16, (B, H, Nq, d), dev)
    _check("lse", lse, torch.float32, (B, H, Nq), dev)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(dev):
        rc = lib().fa_fwd_rect(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                               lse.data_ptr(), B, H, Nq, Nk, d, int(bool(causal)), float(scale),
                               _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc)


def attention_rect(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Allocating form of fa_fwd_rect: returns (O, LSE)."""
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    fa_fwd_rect(q, k, v, o, lse, causal=causal, scale=scale, stream=stream)
    return o, lse


def fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal: bool = False, scale: float | None = None,
           stream=None) -> None:
    """dQ, dK, dV into caller-owned tensors, from the forward's O and LSE.

    q, o, do, dq: bf16 [B, H, Nq, d]; k, v, dk, dv: bf16 [B, H, Nk, d];
    lse: fp32 [B, H, Nq] (the forward's natural-log logsumexp).  Same mask
    and scale as the forward that produced O and LSE.
    """
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B, H, Nq, d] and k [B, H, Nk, d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("tensors must be on a CUDA device")
    for name, t in (("q", q), ("o", o), ("do", do), ("dq", dq)):
        _check(name, t, torch.bfloat16, (B, H, Nq, d), dev)
    for name, t in (("k", k), ("v", v), ("dk", dk), ("dv", dv)):
        _check(name, t, torch.bfloat16, (B, H, Nk, d), dev)
    _check("lse", lse, torch.float32, (B, H, Nq), dev)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(dev):
        rc = lib().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d,
                          int(bool(causal)), float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc)


def attention_backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None,
                       stream=None):
    """Allocating form of fa_bwd: returns (dQ, dK, dV)."""
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    fa_bwd(q, k, v, o, lse, do, dq, dk, dv, causal=causal, scale=scale, stream=stream)
    return dq, dk, dv


def quantize_fp8(x, mode: int, stream=None):
    """bf16 x [B, H, N, d] to e4m3 codes (uint8) and fp32 scales.

    mode 0 (Q, K): codes [B, H, N, d], scales [B, H, ceil(N/128)], one per 128 rows.
    mode 1 (V): codes transposed [B, H, d, ceil(N/128)*128] (padding keys 0),
    scales [B, H], one per head.
    """
    if x.dim() != 4 or x.dtype != torch.bfloat16 or not x.is_contiguous() or x.device.type != "cuda":
        raise ValueError("x must be a contiguous bf16 CUDA tensor [B, H, N, d]")
    B, H, N, d = x.shape
    nblk = (N + 127) // 128
    if mode == 0:
        x8 = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
        scales = torch.empty((B, H, nblk), dtype=torch.float32, device=x.device)
    elif mode == 1:
        x8 = torch.empty((B, H, d, nblk * 128), dtype=torch.uint8, device=x.device)
        scales = torch.empty((B, H), dtype=torch.float32, device=x.device)
    else:
        raise ValueError("mode is 0 (Q, K) or 1 (V)")
    with torch.cuda.device(x.device):
        rc = lib().fa_quantize_fp8(x.data_ptr(), x8.data_ptr(), scales.data_ptr(), B, H, N, d, mode,
                                   _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc)
    return x8, scales


def fa_fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, causal: bool = False,
               scale: float | None = None, stream=None) -> None:
    """The forward on FP8 operands (the layouts of quantize_fp8), into caller-owned O and LSE."""
    B, H, N, d = q8.shape
    dev = q8.device
    nblk = (N + 127) // 128
    _check("q8", q8, torch.uint8, (B, H, N, d), dev)
    _check("k8", k8, torch.uint8, (B, H, N, d), dev)
    _check("vt8", vt8, torch.uint8, (B, H, d, nblk * 128), dev)
    _check("q_scale", q_scale, torch.float32, (B, H, nblk), dev)
    _check("k_scale", k_scale, torch.float32, (B, H, nblk), dev)
    _check("v_scale", v_scale, torch.float32, (B, H), dev)
    _check("o", o, torch.bfloat16, (B, H, N, d), dev)
    _check("lse", lse, torch.float32, (B, H, N), dev)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with torch.cuda.device(dev):
        rc = lib().fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), q_scale.data_ptr(),
                              k_scale.data_ptr(), v_scale.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
                              N, d, int(bool(causal)), float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc)


def attention_fp8(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Quantises bf16 q, k, v to FP8 and runs the FP8 forward; returns (O, LSE)."""
    q8, sq = quantize_fp8(q, 0, stream)
    k8, sk = quantize_fp8(k, 0, stream)
    vt8, sv = quantize_fp8(v, 1, stream)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    fa_fwd_fp8(q8, k8, vt8, sq, sk, sv, o, lse, causal=causal, scale=scale, stream=stream)
    return o, lse


def attention(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Allocates O (bf16) and LSE (fp32) next to q and runs the forward; returns (O, LSE)."""
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    fa_fwd(q, k, v, o, lse, causal=causal, scale=scale, stream=stream)
    return o, lse


def attention_host(q, k, v, causal: bool = False, scale: float | None = None, device="cuda",
                   stream=None, out=None, workspace=None):
    """End-to-end call from host memory: copies q, k, v (pinned host bf16) to the
    device, runs the forward, and copies O and LSE back into host tensors.

    ``workspace`` may hold preallocated device tensors (q, k, v, o, lse) and
    ``out`` preallocated pinned host tensors (o, lse), so that repeated calls
    allocate nothing.  Returns (o_host, lse_host); synchronises the stream.
    """
    dev = torch.device(device)
    B, H, N, d = q.shape
    if workspace is None:
        workspace = tuple(torch.empty_like(t, device=dev) for t in (q, k, v)) + (
            torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev),
            torch.empty((B, H, N), dtype=torch.float32, device=dev))
    qd, kd, vd, od, lsed = workspace
    if out is None:
        out = (torch.empty((B, H, N, d), dtype=torch.bfloat16, pin_memory=True),
               torch.empty((B, H, N), dtype=torch.float32, pin_memory=True))
    oh, lseh = out
    s = torch.cuda.current_stream(dev) if stream is None else stream
    with torch.cuda.stream(s):
        qd.copy_(q, non_blocking=True)
        kd.copy_(k, non_blocking=True)
        vd.copy_(v, non_blocking=True)
        fa_fwd(qd, kd, vd, od, lsed, causal=causal, scale=scale, stream=s)
        oh.copy_(od, non_blocking=True)
        lseh.copy_(lsed, non_blocking=True)
    s.synchronize()
    return oh, lseh


def plan(B: int, H: int, N: int, d: int, causal: bool = False,
         n_keys: int | None = None) -> tuple[int, int]:
    """(attention grid, split items) that fa_fwd uses for these sizes on the current device.

    N query rows and ``n_keys`` keys (default N, as fa_fwd).  Split items are
    computed in parts and merged inside the same launch.
    """
    grid, nsplit = ctypes.c_int(0), ctypes.c_int(0)
    nk = N if n_keys is None else n_keys
    rc = lib().fa_fwd_plan(int(B), int(H), int(N), int(nk), int(d), int(bool(causal)),
                           ctypes.addressof(grid), ctypes.addressof(nsplit))
    if rc != FA_OK:
        raise FAError(rc)
    return grid.value, nsplit.value


KERNELS_PER_CALL = 1  # an fa_fwd call at the bench sizes is one kernel launch (so is a decode call up to 2048 heads)
BWD_KERNELS_PER_CALL = 3  # fa_bwd: prep (D, L, zero dQ accumulator), the backward kernel, dQ conversion


def device_status(stream=None) -> int:
    """FA_OK, or FA_ERR_DEVICE_TIMEOUT if a kernel gave up on a wait (clears the record)."""
    return lib().fa_get_device_status(_stream_handle(stream))


def release_stream(stream=None) -> None:
    """Frees the library's workspaces for `stream` (after synchronising it)."""
    rc = lib().fa_release_stream(_stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc)


def watchdog_selftest(limit_ms: int = 100, device="cuda") -> int:
    """Runs the deliberate-starvation self-test; returns the status the library reports."""
    dev = torch.device(device)
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device=dev)
    k, v, o = torch.zeros_like(q), torch.zeros_like(q), torch.zeros_like(q)
    lse = torch.zeros((1, 1, 128), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        return lib().fa_watchdog_selftest(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                          lse.data_ptr(), int(limit_ms),
                                          torch.cuda.current_stream(dev).cuda_stream)
