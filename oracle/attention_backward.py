"""Plain, slow, fp64 CPU oracle for the exact attention backward pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` may use it.  It shares no code with the CUDA path.

What is computed, and where the pages define it
-----------------------------------------------
For one head with scores s_ij = scale * q_i . k_j over the visible keys
(j < N_k and, causal, j <= i: the top-left mask), P = softmax(s) per row,
O = P V, and an upstream gradient dO = dLoss/dO:

* ``attention_backward`` — the gradients of O with respect to Q, K and V by
  the plain chain rule: dV = P^T dO; dP = dO V^T; the softmax Jacobian gives
  dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik); dQ = scale * dS K and
  dK = scale * dS^T Q.  The row term is written out as the sum over the row
  of P * dP, the textbook form, not through the shortcut below.  Source:
  "FlashAttention and kernels." (gtadkapally.com), section "The backward
  pass: recompute instead of remember" (the five tile products and the
  softmax backward, elementwise).
* ``rowdot`` — the shortcut that section derives: sum_j P_ij dP_ij equals
  dO_i . O_i, one dot product per query row (called D there).
* ``tiled_attention_backward`` — the algorithm that section describes: from
  the saved O and the natural-log logsumexp L of the forward pass, walk the
  tiles again, recompute each tile's probabilities as P = exp(S - L) (no
  running maximum), and accumulate dV += P^T dO, dK += scale dS^T Q and
  dQ += scale dS K tile by tile with dS = P (dP - D).  The same recompute
  is described in "FlashAttention 2 from PyTorch to Triton" (dev.to, Lewis
  Won), section "What I am building" (P = exp(S - L) because
  exp(S - m) / l = exp(S - m - log l)), and in "Kernels and FlashAttention:
  When the Same Math Runs 7.6x Faster" (prathameshsaraf.com), section 2.9.
  It is a second CPU path used only to pin the first one.

Readings where the pages are silent (listed in the design notes): the
gradient flows through the softmax only (masked scores are constants, -inf,
and carry none); L is the logsumexp of the scaled, masked row, so P is
exp(S - L) with S already scaled; dQ and dK carry the factor scale because
the scores are scale * Q K^T.

Parity status: every function here is pinned by
tests/test_oracle_backward_pins.py (central finite differences of the
forward oracle, a closed form for two keys, invariants of the softmax
Jacobian, and the two CPU paths against each other).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "attention_backward",
    "rowdot",
    "tiled_attention_backward",
]


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def _visible(n_keys: int, rows: np.ndarray, causal: bool) -> np.ndarray:
    """Boolean [len(rows), n_keys]: key j is visible to query i iff (not causal or j <= i)."""
    j = np.arange(n_keys)[None, :]
    if causal:
        return j <= rows[:, None]
    return np.ones((rows.shape[0], n_keys), dtype=bool)


def _softmax_rows(s: np.ndarray) -> np.ndarray:
    """Safe softmax of every row of s (masked entries are -inf and come out 0)."""
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=1, keepdims=True)


def _head_backward(q, k, v, do, scale: float, causal: bool, row_block: int):
    """Gradients for one head; q, do: [N_q, d]; k: [N_k, d]; v: [N_k, d_v]."""
    n_q = q.shape[0]
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r0 in range(0, n_q, row_block):
        rows = np.arange(r0, min(n_q, r0 + row_block))
        vis = _visible(k.shape[0], rows, causal)
        if not np.all(vis.any(axis=1)):
            raise ValueError("a query row has no visible key; its result is undefined")
        s = np.where(vis, scale * (q[rows] @ k.T), -np.inf)
        p = _softmax_rows(s)                              # P, [rows, N_k]
        dv += p.T @ do[rows]                              # dV = P^T dO
        dp = do[rows] @ v.T                               # dP = dO V^T
        row_term = np.sum(p * dp, axis=1, keepdims=True)  # sum_k P_ik dP_ik
        ds = p * (dp - row_term)                          # softmax Jacobian applied to dP
        dq[rows] = scale * (ds @ k)                       # dQ = scale dS K
        dk += scale * (ds.T @ q[rows])                    # dK = scale dS^T Q
    return dq, dk, dv


def attention_backward(q, k, v, do, scale: float, causal: bool, row_block: int = 512):
    """dQ, dK, dV of O = softmax(scale Q K^T [causal]) V for the upstream gradient dO.

    q, do: [..., N_q, d]; k: [..., N_k, d]; v: [..., N_k, d_v]; leading axes
    are independent heads.  Returns float64 (dq, dk, dv) shaped like q, k, v.
    Query rows are taken ``row_block`` at a time so that long sequences fit
    in host memory; dK and dV are sums over rows, so this only splits the sum.
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    if q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1] or v.shape[:-1] != k.shape[:-1]:
        raise ValueError("q must be [..., N_q, d], k [..., N_k, d] and v [..., N_k, d_v]")
    if do.shape[:-1] != q.shape[:-1] or do.shape[-1] != v.shape[-1]:
        raise ValueError("do must be [..., N_q, d_v]")
    lead = q.shape[:-2]
    n_q, d = q.shape[-2:]
    n_k, dv_ = k.shape[-2], v.shape[-1]
    qf, kf = q.reshape(-1, n_q, d), k.reshape(-1, n_k, d)
    vf, dof = v.reshape(-1, n_k, dv_), do.reshape(-1, n_q, dv_)
    dq, dk, dv = np.empty_like(qf), np.empty_like(kf), np.empty_like(vf)
    for h in range(qf.shape[0]):
        dq[h], dk[h], dv[h] = _head_backward(qf[h], kf[h], vf[h], dof[h], scale, causal, row_block)
    return dq.reshape(q.shape), dk.reshape(k.shape), dv.reshape(v.shape)


def rowdot(do, o) -> np.ndarray:
    """D_i = dO_i . O_i for every query row (the shortcut for sum_j P_ij dP_ij)."""
    return np.sum(_f64(do) * _f64(o), axis=-1)


def tiled_attention_backward(q, k, v, o, lse, do, scale: float, causal: bool,
                             Br: int = 64, Bc: int = 64):
    """The recompute-from-L backward for one head, key blocks outer, query blocks inner.

    q, o, do: [N_q, d]; k, v: [N_k, d]; lse: [N_q] natural-log logsumexp of
    the scaled, masked score rows (the forward's second output).
    D = rowdot(dO, O) once; then for each key block and each query block:
    S = scale Q K^T (masked -inf), P = exp(S - L), dV += P^T dO,
    dP = dO V^T, dS = P (dP - D), dQ += scale dS K, dK += scale dS^T Q.
    """
    q, k, v, o, do = _f64(q), _f64(k), _f64(v), _f64(o), _f64(do)
    lse = _f64(lse)
    n_q, n_k = q.shape[0], k.shape[0]
    D = rowdot(do, o)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for j0 in range(0, n_k, Bc):
        cols = np.arange(j0, min(n_k, j0 + Bc))
        for i0 in range(0, n_q, Br):
            rows = np.arange(i0, min(n_q, i0 + Br))
            s = scale * (q[rows] @ k[cols].T)
            if causal:
                s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)
            p = np.exp(s - lse[rows][:, None])           # exact probabilities from L
            dv[cols] += p.T @ do[rows]
            dp = do[rows] @ v[cols].T
            ds = p * (dp - D[rows][:, None])
            dq[rows] += scale * (ds @ k[cols])
            dk[cols] += scale * (ds.T @ q[rows])
    return dq, dk, dv
