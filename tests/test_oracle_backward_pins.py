"""Pins for the fp64 backward oracle.

None of these re-types the oracle's gradient formulas.  The gradients are
checked against central finite differences of the forward oracle (itself
pinned by test_oracle_pins.py), against a closed form for two keys, against
invariants the softmax Jacobian fixes (rows of dS sum to zero, so the key
gradients sum to zero; the value gradients share out dO exactly; a single
visible key carries no query gradient), against a uniform-attention case
written with pure-Python loops, and the two CPU paths (the plain chain rule
and the pages' recompute-from-L tile walk) against each other.
"""
import math

import numpy as np
import pytest

import oracle
from oracle.attention import attention as forward_attention
from oracle.attention import attention_weights as forward_weights


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _problem(nq, nk, d, dv, seed):
    return (_rand((nq, d), seed), _rand((nk, d), seed + 1), _rand((nk, dv), seed + 2),
            _rand((nq, dv), seed + 3))


def _loss(q, k, v, do, scale, causal):
    o, _ = forward_attention(q, k, v, scale, causal)
    return float(np.sum(o * do))


def _central_differences(q, k, v, do, scale, causal, h=1e-5):
    """d(sum O * dO) / d(each input element), by (f(x + h) - f(x - h)) / 2h."""
    grads = []
    for which in range(3):
        args = [q.copy(), k.copy(), v.copy()]
        x = args[which]
        g = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            x0 = x[idx]
            x[idx] = x0 + h
            fp = _loss(*args, do, scale, causal)
            x[idx] = x0 - h
            fm = _loss(*args, do, scale, causal)
            x[idx] = x0
            g[idx] = (fp - fm) / (2 * h)
        grads.append(g)
    return grads


@pytest.mark.parametrize("nq,nk,d,dv", [(5, 7, 3, 3), (6, 6, 4, 2), (7, 4, 2, 3), (1, 5, 3, 2)])
@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_finite_differences(nq, nk, d, dv, causal):
    q, k, v, do = _problem(nq, nk, d, dv, seed=nq * 31 + nk)
    scale = 0.7
    dq, dk, dv_ = oracle.attention_backward(q, k, v, do, scale, causal)
    fq, fk, fv = _central_differences(q, k, v, do, scale, causal)
    for name, got, want in (("dq", dq, fq), ("dk", dk, fk), ("dv", dv_, fv)):
        assert got.shape == want.shape, name
        assert np.max(np.abs(got - want)) <= 2e-8, name


def test_two_keys_closed_form():
    # d = 1, one query over two keys: O = w0 v0 + w1 v1, w = softmax(scale q k_j).
    q, k0, k1, v0, v1, g, scale = 0.8, 1.3, -0.4, 2.0, -1.5, 0.9, 0.6
    w0 = 1.0 / (1.0 + math.exp(-scale * q * (k0 - k1)))
    w1 = 1.0 - w0
    want_dq = g * scale * w0 * w1 * (k0 - k1) * (v0 - v1)
    want_dk0 = g * scale * q * w0 * w1 * (v0 - v1)
    dq, dk, dv = oracle.attention_backward(
        np.array([[q]]), np.array([[k0], [k1]]), np.array([[v0], [v1]]), np.array([[g]]),
        scale, False)
    assert abs(dq[0, 0] - want_dq) <= 1e-15
    assert abs(dk[0, 0] - want_dk0) <= 1e-15 and abs(dk[1, 0] + want_dk0) <= 1e-15
    assert abs(dv[0, 0] - g * w0) <= 1e-15 and abs(dv[1, 0] - g * w1) <= 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_key_and_value_gradient_sums(causal):
    # Every row of dS sums to zero, so sum_j dK_j = scale sum_i q_i sum_j dS_ij = 0;
    # every row of P sums to one, so sum_j dV_j = sum_i dO_i.
    q, k, v, do = _problem(40, 40, 8, 8, seed=7)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.35, causal)
    assert np.max(np.abs(dk.sum(axis=0))) <= 1e-12
    assert np.max(np.abs(dv.sum(axis=0) - do.sum(axis=0))) <= 1e-12


def test_first_causal_row_has_no_query_gradient():
    # Row 0 sees key 0 only: its output is v_0 whatever q_0 and k_0 are.
    q, k, v, do = _problem(9, 9, 4, 4, seed=8)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5, True)
    assert np.max(np.abs(dq[0])) == 0.0
    q2, k2, v2, do2 = _problem(1, 1, 4, 4, seed=9)
    dq2, dk2, dv2 = oracle.attention_backward(q2, k2, v2, do2, 0.5, False)
    assert np.max(np.abs(dq2)) == 0.0 and np.max(np.abs(dk2)) == 0.0
    assert np.array_equal(dv2, do2)


@pytest.mark.parametrize("causal", [False, True])
def test_shifting_all_keys_or_values_leaves_gradients(causal):
    # k_j + c adds scale q_i . c to a whole row of scores: P is unchanged, so are
    # O and every gradient.  v_j + c adds c to every output row and dO_i . c to
    # every dP_ij of row i, which the softmax Jacobian removes.
    q, k, v, do = _problem(12, 15, 5, 5, seed=10)
    c = _rand((5,), 11)
    base = oracle.attention_backward(q, k, v, do, 0.4, causal)
    for shifted in (oracle.attention_backward(q, k + c, v, do, 0.4, causal),
                    oracle.attention_backward(q, k, v + c, do, 0.4, causal)):
        for a, b in zip(base, shifted):
            assert np.max(np.abs(a - b)) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_attention_closed_form(causal):
    # q = 0: every visible key gets weight 1 / (number visible).  Pure-Python loops:
    # dV_j = sum over rows i that see j of dO_i / n_i; dK = 0 (dK = scale dS^T Q);
    # dQ_i = scale / n_i * sum_j (dO_i . (v_j - vbar_i)) k_j over the visible j.
    nq, nk, d, scale = 6, 6, 3, 0.8
    _, k, v, do = _problem(nq, nk, d, d, seed=12)
    q = np.zeros((nq, d))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale, causal)
    want_dv = [[0.0] * d for _ in range(nk)]
    want_dq = [[0.0] * d for _ in range(nq)]
    for i in range(nq):
        seen = list(range(i + 1)) if causal else list(range(nk))
        n = len(seen)
        vbar = [sum(v[j][c] for j in seen) / n for c in range(d)]
        for j in seen:
            for c in range(d):
                want_dv[j][c] += do[i][c] / n
            w = sum(do[i][c] * (v[j][c] - vbar[c]) for c in range(d))
            for c in range(d):
                want_dq[i][c] += scale / n * w * k[j][c]
    assert np.max(np.abs(dv - np.array(want_dv))) <= 1e-13
    assert np.max(np.abs(dq - np.array(want_dq))) <= 1e-13
    assert np.max(np.abs(dk)) == 0.0


@pytest.mark.parametrize("causal", [False, True])
def test_rowdot_is_the_softmax_row_term(causal):
    # sum_j P_ij dP_ij = dO_i . O_i, with P and O from the forward oracle.
    q, k, v, do = _problem(20, 20, 6, 6, seed=13)
    p = forward_weights(q, k, 0.45, causal)
    o, _ = forward_attention(q, k, v, 0.45, causal)
    want = np.array([sum(p[i, j] * float(do[i] @ v[j]) for j in range(20)) for i in range(20)])
    assert np.max(np.abs(oracle.rowdot(do, o) - want)) <= 1e-12


@pytest.mark.parametrize("nq,nk", [(37, 37), (50, 23), (9, 70)])
@pytest.mark.parametrize("Br,Bc", [(1, 1), (16, 8), (64, 64), (5, 13)])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_recompute_equals_definition(nq, nk, Br, Bc, causal):
    q, k, v, do = _problem(nq, nk, 5, 5, seed=14)
    scale = 0.6
    o, lse = forward_attention(q, k, v, scale, causal)
    want = oracle.attention_backward(q, k, v, do, scale, causal)
    got = oracle.tiled_attention_backward(q, k, v, o, lse, do, scale, causal, Br=Br, Bc=Bc)
    for a, b in zip(got, want):
        assert np.max(np.abs(a - b)) <= 1e-12


def test_heads_are_independent_and_rows_blocked():
    q, k, v, do = (_rand((2, 3, 30, 4), s) for s in (15, 16, 17, 18))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.5, True, row_block=7)
    for b in range(2):
        for h in range(3):
            one = oracle.attention_backward(q[b, h], k[b, h], v[b, h], do[b, h], 0.5, True)
            for a, o in zip((dq[b, h], dk[b, h], dv[b, h]), one):
                assert np.max(np.abs(a - o)) <= 1e-12
