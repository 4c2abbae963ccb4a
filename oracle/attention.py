"""Plain, slow, fp64 CPU oracle for the fused exact attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code with the CUDA path; it receives plain numpy arrays (bf16 values
already widened, exactly, to float) and computes everything in float64.

What is computed, and where the pages define it
-----------------------------------------------
* ``attention`` / ``attention_rows`` — the plain definition of scaled
  dot-product attention, O = softmax(scale * Q K^T [causal]) V, with the row
  maximum subtracted before exponentiation, plus the per-row logsumexp
  L = m + ln(l).  Sources: "4 Triton and Custom Kernels" (aisyseng.dev),
  section 4.7, Eq. 4.1; "FlashAttention and kernels." (gtadkapally.com),
  sections "Softmax, the safe way" and "FlashAttention's forward pass" (the
  logsumexp written per row for the backward pass); "FlashAttention 2 from
  PyTorch to Triton" (dev.to, Lewis Won), section "What I am building" (L is
  the natural-log logsumexp of the scaled scores).  The causal mask keeps key
  j for query i when j <= i (same pages, "causal mask" glossary entry of the
  gtadkapally lesson; top-left convention of "How to profile and optimise
  kernels", Round 4, "Causal tile-skipping").
* ``softmax_safe`` — the three-pass safe softmax ("Softmax, the safe way").
* ``online_max_sum`` / ``merge_max_sum`` — the one-pass running maximum and
  running sum, and the merge of two partial states ("Online softmax: keep a
  running max and a running sum", same lesson; "Kernels and FlashAttention:
  When the Same Math Runs 7.6x Faster" (prathameshsaraf.com), section 2.7).
* ``tiled_attention`` — the FlashAttention-2 recurrence over query blocks of
  Br rows and key blocks of Bc keys: m_new = max(m, rowmax(S_blk)),
  alpha = exp(m - m_new), l = alpha*l + rowsum(P), O = alpha*O + P V_blk,
  divide by l once at the end ("From a sum to an output row" and
  "FlashAttention's forward pass" of the gtadkapally lesson; section 2.8 of
  the prathameshsaraf post; section 4.8 of the aisyseng chapter, worked
  example "Online softmax across two blocks").  It is a second CPU path used
  only to pin the first one; it is never the primary reference.
* ``merge_partials`` — combining normalised partial results computed over
  disjoint key ranges through their logsumexps (the Flash-Decoding merge in
  "FlashAttention-2, -3, and what came after" of the gtadkapally lesson,
  which reuses the (m, l, o) merge rule).

Readings where the pages are silent (all listed in the design notes):
masked scores are excluded (equivalently -inf); a row with no visible key has
no defined result and is rejected here (the pages leave it to "an explicit
caller policy", section 4.8 of the aisyseng chapter); LSE is in natural-log
units and float64.

Parity status: every function here is pinned by tests/test_oracle_pins.py
(the pages' worked examples, closed forms, invariants and brute force).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "softmax_safe",
    "online_max_sum",
    "merge_max_sum",
    "attention",
    "attention_rows",
    "attention_weights",
    "tiled_attention",
    "merge_partials",
]


# ---------------------------------------------------------------------------
# Softmax building blocks
# ---------------------------------------------------------------------------

def softmax_safe(x) -> np.ndarray:
    """Three passes over a 1-D row: m = max(x); l = sum(exp(x - m)); exp(x - m) / l.

    "FlashAttention and kernels.", section "Softmax, the safe way".
    """
    x = np.asarray(x, dtype=np.float64)
    m = np.max(x)                     # pass 1
    e = np.exp(x - m)
    l = np.sum(e)                     # pass 2
    return e / l                      # pass 3


def online_max_sum(x) -> tuple[float, float]:
    """One pass, one element at a time: the running max m and the running sum l.

    Start at m = -inf, l = 0; for each x: m_new = max(m, x),
    l = l * exp(m - m_new) + exp(x - m_new).  "FlashAttention and kernels.",
    section "Online softmax: keep a running max and a running sum".
    """
    m = -math.inf
    l = 0.0
    for xi in np.asarray(x, dtype=np.float64).ravel():
        xi = float(xi)
        m_new = max(m, xi)
        l = l * math.exp(m - m_new) + math.exp(xi - m_new)
        m = m_new
    return m, l


def merge_max_sum(a: tuple[float, float], b: tuple[float, float]) -> tuple[float, float]:
    """Combine two partial (m, l) states measured against their own maxima.

    Both sums are moved onto the larger maximum by one factor each, the same
    rescale the online update applies ("FlashAttention and kernels.", the
    merge rule of "Online softmax" used by Flash-Decoding).
    """
    (ma, la), (mb, lb) = a, b
    m = max(ma, mb)
    if m == -math.inf:
        return m, 0.0
    return m, la * math.exp(ma - m) + lb * math.exp(mb - m)


# ---------------------------------------------------------------------------
# The definition: materialise S, safe softmax per row, multiply by V
# ---------------------------------------------------------------------------

def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def _visible(n_keys: int, rows: np.ndarray, causal: bool) -> np.ndarray:
    """Boolean [len(rows), n_keys]: key j is visible to query i iff j < N_k and (not causal or j <= i)."""
    j = np.arange(n_keys)[None, :]
    if causal:
        return j <= rows[:, None]
    return np.ones((rows.shape[0], n_keys), dtype=bool)


def _head_rows(q, k, v, scale: float, causal: bool, rows: np.ndarray):
    """Definition for a set of query rows of one head.

    q: [N_q, d], k: [N_k, d], v: [N_k, d_v] (float64); rows: int indices into q.
    Returns (O [len(rows), d], LSE [len(rows)]) in float64.
    """
    s = scale * (q[rows] @ k.T)                      # scores s_ij = scale * q_i . k_j
    vis = _visible(k.shape[0], rows, causal)
    if not np.all(vis.any(axis=1)):
        raise ValueError("a query row has no visible key; its result is undefined")
    s = np.where(vis, s, -np.inf)                   # masked keys take no part
    m = np.max(s, axis=1, keepdims=True)            # row maximum (safe softmax)
    e = np.exp(s - m)                               # exp(-inf) = 0 for masked keys
    l = np.sum(e, axis=1, keepdims=True)            # row sum
    o = (e @ v) / l                                 # weighted average of value rows
    lse = m[:, 0] + np.log(l[:, 0])                 # natural-log logsumexp of the scaled row
    return o, lse


def attention_weights(q, k, scale: float, causal: bool) -> np.ndarray:
    """softmax(scale * q k^T [causal]) for one head, [N, N] float64 (masked entries are 0)."""
    q, k = _f64(q), _f64(k)
    rows = np.arange(q.shape[0])
    s = scale * (q @ k.T)
    vis = _visible(k.shape[0], rows, causal)
    s = np.where(vis, s, -np.inf)
    return np.stack([softmax_safe(row) for row in s])


def attention(q, k, v, scale: float, causal: bool, row_block: int = 256):
    """O and LSE for q [..., N_q, d], k [..., N_k, d] and v [..., N_k, d_v].

    Leading axes are independent heads.  N_q and N_k may differ; causal then
    keeps key j for query i when j <= i, the top-left mask ("How to profile
    and optimise kernels", Round 4: non-square causal attention is checked
    against an explicit top-left mask).  Returns (O float64 [..., N_q, d_v],
    LSE float64 [..., N_q]).  S is materialised ``row_block`` query rows at a
    time so that long sequences fit in host memory; every row is still
    computed by the plain definition.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.shape[:-2] != k.shape[:-2] or q.shape[-1] != k.shape[-1] or v.shape[:-1] != k.shape[:-1]:
        raise ValueError("q must be [..., N_q, d], k [..., N_k, d] and v [..., N_k, d_v]")
    lead = q.shape[:-2]
    n_q, d = q.shape[-2:]
    n_k = k.shape[-2]
    dv = v.shape[-1]
    qf = q.reshape(-1, n_q, d)
    kf = k.reshape(-1, n_k, d)
    vf = v.reshape(-1, n_k, dv)
    o = np.empty((qf.shape[0], n_q, dv))
    lse = np.empty(qf.shape[:2], dtype=np.float64)
    for h in range(qf.shape[0]):
        for r0 in range(0, n_q, row_block):
            rows = np.arange(r0, min(n_q, r0 + row_block))
            o[h, rows], lse[h, rows] = _head_rows(qf[h], kf[h], vf[h], scale, causal, rows)
    return o.reshape(*lead, n_q, dv), lse.reshape(*lead, n_q)


def attention_rows(q_head, k_head, v_head, scale: float, causal: bool, rows):
    """The definition evaluated only for the listed query rows of one head.

    Used to check sampled outputs of very long sequences one row at a time.
    """
    rows = np.asarray(rows, dtype=np.int64)
    return _head_rows(_f64(q_head), _f64(k_head), _f64(v_head), scale, causal, rows)


# ---------------------------------------------------------------------------
# The FlashAttention-2 recurrence (second CPU path, for pinning only)
# ---------------------------------------------------------------------------

def tiled_attention(q, k, v, scale: float, causal: bool, Br: int = 64, Bc: int = 64,
                    trace: bool = False):
    """Online-softmax attention for one head, query blocks outer, key blocks inner.

    q: [N_q, d], k: [N_k, d], v: [N_k, d_v]; causal keeps key j for query i
    when j <= i (top-left).

    For each query block, m = -inf, l = 0, acc = 0; for each key block:
    m_new = max(m, rowmax(S)), P = exp(S - m_new), alpha = exp(m - m_new),
    l = alpha*l + rowsum(P), acc = alpha*acc + P V, m = m_new.  After the last
    block O = acc / l and L = m + ln(l).  Masked scores are -inf.  A key
    block that is entirely masked for a row that has not yet seen any visible
    key is skipped for that row (alpha = 1, P = 0), as section 4.8 of the
    aisyseng chapter prescribes for all-masked blocks; once m is finite the
    plain update already gives P = 0 and alpha = 1 for such a block.

    With ``trace=True`` also returns the list of (m, l, acc) after each key
    block for every query block (copies), for checking printed traces.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    n_q, d = q.shape
    n_k = k.shape[0]
    O = np.empty((n_q, v.shape[1]))
    L = np.empty(n_q, dtype=np.float64)
    states = []
    for i0 in range(0, n_q, Br):
        rows = np.arange(i0, min(n_q, i0 + Br))
        qb = q[rows]
        m = np.full(rows.shape[0], -np.inf)
        l = np.zeros(rows.shape[0])
        acc = np.zeros((rows.shape[0], v.shape[1]))
        block_trace = []
        for j0 in range(0, n_k, Bc):
            cols = np.arange(j0, min(n_k, j0 + Bc))
            s = scale * (qb @ k[cols].T)
            if causal:
                s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)
            m_blk = np.max(s, axis=1)
            m_new = np.maximum(m, m_blk)
            live = np.isfinite(m_new)                    # rows that have seen a visible key
            m_use = np.where(live, m_new, 0.0)
            p = np.exp(s - m_use[:, None])               # exp(-inf) = 0
            alpha = np.where(live, np.exp(m - m_use), 1.0)
            l = alpha * l + np.sum(p, axis=1)
            acc = alpha[:, None] * acc + p @ v[cols]
            m = m_new
            if trace:
                block_trace.append((m.copy(), l.copy(), acc.copy()))
        O[rows] = acc / l[:, None]
        L[rows] = m + np.log(l)
        states.append(block_trace)
    if trace:
        return O, L, states
    return O, L


# ---------------------------------------------------------------------------
# Merge of partial results over disjoint key ranges
# ---------------------------------------------------------------------------

def merge_partials(outputs, lses):
    """Combine normalised partial results (O_r, LSE_r) over disjoint key ranges.

    Each O_r = sum_{j in range r} exp(s_j - LSE_r) v_j is already normalised
    within its range.  The whole row is LSE = ln(sum_r exp(LSE_r)) and
    O = sum_r exp(LSE_r - LSE) O_r; the largest LSE_r is subtracted first so
    that nothing overflows (the merge rule carried by Flash-Decoding in
    "FlashAttention and kernels.").  outputs: sequence of [..., d]; lses:
    sequence of [...] float arrays.
    """
    lses = [np.asarray(x, dtype=np.float64) for x in lses]
    outputs = [np.asarray(x, dtype=np.float64) for x in outputs]
    m = np.max(np.stack(lses), axis=0)
    w = [np.exp(x - m) for x in lses]
    total = np.sum(np.stack(w), axis=0)
    lse = m + np.log(total)
    o = sum(wi[..., None] * oi for wi, oi in zip(w, outputs)) / total[..., None]
    return o, lse
