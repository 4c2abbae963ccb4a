"""Pins for the fp64 oracle: the pages' worked examples, closed forms, invariants
and brute force.  None of these re-types the oracle's own formula: each value
comes from a page (tests/golden/, cited there), from algebra that fixes the
answer independently, or from a pure-Python evaluation of the textbook
softmax without any of the oracle's steps (no max shift, no blocking, no
numpy linear algebra).
"""
import math

import numpy as np
import pytest

import oracle


def _tol(decimals):
    return 0.5 * 10.0 ** (-decimals) + 1e-12


# ---------------------------------------------------------------------------
# E1-E4: values printed on the pages
# ---------------------------------------------------------------------------

def test_e1_four_token_trace(golden):
    g = golden("four_token_trace.json")
    q = np.array(g["q"], float)
    k = np.array(g["k"], float)
    v = np.array(g["v"], float)
    scale = 1.0 / math.sqrt(g["head_dim"])
    pr, tol = g["printed"], _tol(g["printed_decimals"])

    # The query sits at position four: embed it as the last of four query rows
    # so that the causal mask is exercised and keeps all four keys.
    qs = np.vstack([np.zeros((3, 2)), q])
    for causal in (False, True):
        o, lse = oracle.attention_rows(qs, k, v, scale, causal, [3])
        assert np.max(np.abs(o[0] - pr["output"])) <= tol
        assert abs(math.exp(lse[0]) - pr["sum"]) <= tol   # LSE = ln(sum of exponentials)
    w = oracle.attention_weights(qs, k, scale, causal=True)[3]
    assert np.max(np.abs(w - pr["weights"])) <= tol
    # closed form: o = [sigmoid(1/sqrt 2), 1/2]
    o, _ = oracle.attention_rows(q, k, v, scale, False, [0])
    assert abs(o[0, 0] - 1.0 / (1.0 + math.exp(-1.0 / math.sqrt(2)))) <= 1e-14
    assert abs(o[0, 1] - 0.5) <= 1e-14


def test_e2_two_block_online(golden):
    g = golden("two_block_online.json")
    s = np.array(g["scaled_scores"], float)
    v = np.array(g["v"], float)
    pr = g["printed"]
    # scores are realised as q . k with d = 1, q = 1 and scale = 1
    q = np.ones((1, 1))
    k = s[:, None]
    o, lse, states = oracle.tiled_attention(q, k, v, 1.0, False, Br=1, Bc=g["block_size"], trace=True)
    (m1, l1, acc1), (m2, l2, acc2) = states[0]
    assert m1[0] == pr["after_block_1"]["m"] and l1[0] == pr["after_block_1"]["l"]
    np.testing.assert_allclose(acc1[0], pr["after_block_1"]["o"], rtol=0, atol=1e-15)
    assert abs(m2[0] - pr["after_block_2"]["m"]) <= 1e-15
    assert abs(l2[0] - pr["after_block_2"]["l"]) <= 1e-14
    np.testing.assert_allclose(acc2[0], pr["after_block_2"]["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(o[0], pr["output"], rtol=0, atol=1e-14)
    # the plain definition agrees, and so do the printed weights
    o_def, _ = oracle.attention_rows(q, k, v, 1.0, False, [0])
    np.testing.assert_allclose(o_def[0], pr["output"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(oracle.softmax_safe(s), pr["weights"], rtol=0, atol=1e-15)


def test_e3_eight_score_row(golden):
    g = golden("eight_score_row.json")
    s = np.array(g["scores"], float)
    pr, tol = g["printed"], _tol(g["printed_decimals"])
    np.testing.assert_allclose(oracle.softmax_safe(s), pr["P"], rtol=0, atol=tol)
    m, l = oracle.online_max_sum(s)
    assert m == pr["m"] and abs(l - pr["l"]) <= tol
    # tile by tile through the FA2 recurrence: state after each tile of four
    q = np.ones((1, 1))
    v = np.eye(8)                      # O row = softmax weights themselves
    o, lse, states = oracle.tiled_attention(q, s[:, None], v, 1.0, False, Br=1, Bc=g["tile"], trace=True)
    (m1, l1, _), (m2, l2, _) = states[0]
    assert m1[0] == pr["after_tile_1"]["m"] and abs(l1[0] - pr["after_tile_1"]["l"]) <= tol
    assert m2[0] == pr["after_tile_2"]["m"] and abs(l2[0] - pr["after_tile_2"]["l"]) <= tol
    np.testing.assert_allclose(o[0], pr["P"], rtol=0, atol=tol)
    np.testing.assert_allclose(np.exp(s - m), pr["exponentials"], rtol=0, atol=tol)
    assert abs(lse[0] - (pr["m"] + math.log(pr["l"]))) <= 1e-4


def test_e4_four_values(golden):
    g = golden("four_values.json")
    pr, tol = g["printed"], _tol(g["printed_decimals"])
    m, l = oracle.online_max_sum(g["x"])
    assert m == pr["m"] and abs(l - pr["l"]) <= tol
    np.testing.assert_allclose(np.exp(np.array(g["x"], float) - m), pr["terms"], rtol=0, atol=tol)


# ---------------------------------------------------------------------------
# E5: online against safe softmax, whole and merged from uneven chunks
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("scale", [1, 10, 100])
def test_e5_online_vs_safe(scale):
    rng = np.random.default_rng(0)
    x = rng.normal(size=10_000) * scale
    m, l = oracle.online_max_sum(x)
    p_online = np.exp(x - m) / l
    p_safe = oracle.softmax_safe(x)
    # the online sum carries 10,000 sequential rescales: fp64 rounding only
    assert np.max(np.abs(p_online - p_safe)) <= 1e-13
    assert m == np.max(x)
    # seven uneven chunks, each reduced on its own, then merged
    cuts = [0, 3, 100, 1234, 1235, 5000, 7777, 10_000]
    state = (-math.inf, 0.0)
    for a, b in zip(cuts[:-1], cuts[1:]):
        state = oracle.merge_max_sum(state, oracle.online_max_sum(x[a:b]))
    assert state[0] == m
    assert abs(state[1] - l) <= 1e-12 * l
    # and the sum against a compensated textbook sum of the shifted terms
    assert abs(l - math.fsum(math.exp(xi - m) for xi in x)) <= 1e-12 * l


# ---------------------------------------------------------------------------
# Brute force: pure-Python textbook softmax, no max shift, no numpy algebra
# ---------------------------------------------------------------------------

def _brute(q, k, v, scale, causal):
    n_q, d = len(q), len(q[0])
    out, lses = [], []
    for i in range(n_q):
        keys = [j for j in range(len(k)) if (not causal or j <= i)]
        w = [math.exp(scale * math.fsum(q[i][c] * k[j][c] for c in range(d))) for j in keys]
        tot = math.fsum(w)
        out.append([math.fsum(w[t] * v[j][c] for t, j in enumerate(keys)) / tot
                    for c in range(len(v[0]))])
        lses.append(math.log(tot))
    return np.array(out), np.array(lses)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 1), (2, 3), (3, 2), (5, 4), (7, 3), (8, 4)])
def test_brute_force_tiny(n, d, causal):
    rng = np.random.default_rng(1000 * n + d)
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    scale = 0.7
    o_b, lse_b = _brute(q.tolist(), k.tolist(), v.tolist(), scale, causal)
    o, lse = oracle.attention(q, k, v, scale, causal)
    np.testing.assert_allclose(o, o_b, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_b, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n_q,n_k", [(1, 7), (3, 8), (8, 3), (5, 1), (2, 9), (6, 4)])
def test_brute_force_rectangular(n_q, n_k, causal):
    # N_q != N_k with the top-left causal mask (key j visible to query i iff
    # j <= i), "How to profile and optimise kernels", Round 4
    rng = np.random.default_rng(100 * n_q + n_k)
    q = rng.normal(size=(n_q, 3))
    k, v = rng.normal(size=(n_k, 3)), rng.normal(size=(n_k, 2))
    o_b, lse_b = _brute(q.tolist(), k.tolist(), v.tolist(), 0.6, causal)
    o, lse = oracle.attention(q, k, v, 0.6, causal)
    np.testing.assert_allclose(o, o_b, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_b, rtol=0, atol=1e-13)


def test_rectangular_causal_limits():
    # top-left causal: with N_q < N_k the keys from N_q on are never visible,
    # so dropping them changes nothing; with N_q > N_k every row from N_k - 1
    # on sees every key, as without the mask
    rng = np.random.default_rng(31)
    q = rng.normal(size=(2, 5, 4))
    k, v = rng.normal(size=(2, 12, 4)), rng.normal(size=(2, 12, 4))
    o, lse = oracle.attention(q, k, v, 0.5, True)
    o_t, lse_t = oracle.attention(q, k[:, :5], v[:, :5], 0.5, True)
    np.testing.assert_allclose(o, o_t, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, lse_t, rtol=0, atol=1e-14)
    q2 = rng.normal(size=(2, 12, 4))
    k2, v2 = rng.normal(size=(2, 5, 4)), rng.normal(size=(2, 5, 4))
    o_c, lse_c = oracle.attention(q2, k2, v2, 0.5, True)
    o_n, lse_n = oracle.attention(q2, k2, v2, 0.5, False)
    np.testing.assert_allclose(o_c[:, 4:], o_n[:, 4:], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse_c[:, 4:], lse_n[:, 4:], rtol=0, atol=1e-14)
    assert np.abs(o_c[:, :4] - o_n[:, :4]).max() > 1e-3  # the mask does act on the first rows


def test_brute_force_batched_heads_keep_their_own_data():
    rng = np.random.default_rng(7)
    q, k, v = (rng.normal(size=(2, 3, 5, 4)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, 0.5, True)
    for b in range(2):
        for h in range(3):
            o_b, lse_b = _brute(q[b, h].tolist(), k[b, h].tolist(), v[b, h].tolist(), 0.5, True)
            np.testing.assert_allclose(o[b, h], o_b, rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[b, h], lse_b, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# I1-I7: invariants and closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_i1_rows_sum_to_one(causal):
    rng = np.random.default_rng(11)
    q, k = rng.normal(size=(40, 8)) * 3, rng.normal(size=(40, 8)) * 3
    w = oracle.attention_weights(q, k, 0.5, causal)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    if causal:
        assert np.all(np.triu(w, 1) == 0)
    # the logsumexp rebuilds the same weights: exp(s - L)
    v = np.eye(40)
    o, lse = oracle.attention(q, k, v, 0.5, causal)
    np.testing.assert_allclose(o, w, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_i2_identical_keys_give_mean_of_visible_values(causal):
    rng = np.random.default_rng(12)
    n, d = 33, 6
    q = rng.normal(size=(n, d)) * 4
    k = np.tile(rng.normal(size=(1, d)), (n, 1))
    v = rng.normal(size=(n, d))
    o, lse = oracle.attention(q, k, v, 0.3, causal)
    for i in range(n):
        hi = i + 1 if causal else n
        np.testing.assert_allclose(o[i], v[:hi].mean(axis=0), rtol=0, atol=1e-12)
        s = 0.3 * float(q[i] @ k[0])
        assert abs(lse[i] - (s + math.log(hi))) <= 1e-12


def test_i3_causal_row_zero_is_first_value_row():
    rng = np.random.default_rng(13)
    q, k, v = (rng.normal(size=(17, 5)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, 0.8, True)
    np.testing.assert_array_equal(o[0], v[0])
    assert lse[0] == pytest.approx(0.8 * float(q[0] @ k[0]), abs=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_i4_online_equals_two_pass_all_block_sizes(causal):
    rng = np.random.default_rng(14)
    for n in range(1, 9):
        for d in (1, 2, 4):
            q, k, v = (rng.normal(size=(n, d)) * 2 for _ in range(3))
            o_ref, lse_ref = oracle.attention(q, k, v, 0.9, causal)
            for br in range(1, n + 1):
                for bc in range(1, n + 1):
                    o, lse = oracle.tiled_attention(q, k, v, 0.9, causal, Br=br, Bc=bc)
                    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
                    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_i5_key_tile_size_invariance(causal):
    rng = np.random.default_rng(15)
    q, k, v = (rng.normal(size=(200, 16)) * 2 for _ in range(3))
    ref = oracle.tiled_attention(q, k, v, 0.25, causal, Br=64, Bc=1)
    for bc in (3, 16, 64, 128):
        o, lse = oracle.tiled_attention(q, k, v, 0.25, causal, Br=64, Bc=bc)
        np.testing.assert_allclose(o, ref[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref[1], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_i6_max_in_last_tile_and_constant_shift(causal):
    rng = np.random.default_rng(16)
    n, d = 100, 8
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    # the largest scores sit in the last key block (Break It #2 of the
    # gtadkapally lesson): keys 96..99 point along every query's direction
    k[96:] = 6.0 * np.sign(q.sum(axis=0))[None, :] + 0.1 * k[96:]
    o_ref, lse_ref = oracle.attention(q, k, v, 0.5, causal)
    o, lse = oracle.tiled_attention(q, k, v, 0.5, causal, Br=32, Bc=16)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
    # adding c to every score leaves O unchanged and moves L by c: append a
    # constant feature, q' = [q, c/scale], k' = [k, 1]
    c = 37.5
    q2 = np.hstack([q, np.full((n, 1), c / 0.5)])
    k2 = np.hstack([k, np.ones((n, 1))])
    o2, lse2 = oracle.attention(q2, k2, v, 0.5, causal)
    np.testing.assert_allclose(o2, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse2, lse_ref + c, rtol=0, atol=1e-11)


def test_i7_two_key_hand_case():
    s0, s1, v0, v1 = 0.3, -1.1, 2.0, -5.0
    q = np.array([[1.0], [1.0]])
    k = np.array([[s0], [s1]])
    v = np.array([[v0], [v1]])
    o, lse = oracle.attention(q, k, v, 1.0, False)
    expect = (math.exp(s0) * v0 + math.exp(s1) * v1) / (math.exp(s0) + math.exp(s1))
    assert abs(o[0, 0] - expect) <= 1e-15 and abs(o[1, 0] - expect) <= 1e-15
    assert abs(lse[0] - math.log(math.exp(s0) + math.exp(s1))) <= 1e-15
    oc, lsec = oracle.attention(q, k, v, 1.0, True)
    assert oc[0, 0] == v0 and abs(oc[1, 0] - expect) <= 1e-15
    assert abs(lsec[0] - s0) <= 1e-15


@pytest.mark.parametrize("n", [1, 5, 64])
def test_causal_row_equals_last_row_of_its_prefix(n):
    rng = np.random.default_rng(17 + n)
    q, k, v = (rng.normal(size=(n, 4)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, 0.6, True)
    for i in range(n):
        o_p, lse_p = oracle.attention_rows(q[: i + 1], k[: i + 1], v[: i + 1], 0.6, False, [i])
        np.testing.assert_allclose(o[i], o_p[0], rtol=0, atol=1e-14)
        assert abs(lse[i] - lse_p[0]) <= 1e-14


def test_large_scores_do_not_overflow():
    # scores in the thousands (the +-40 outlier workload reaches this): the
    # shifted exponentials stay finite and a dominant key is reproduced
    q = np.array([[40.0] * 8])
    k = np.array([[40.0] * 8, [39.0] * 8, [-40.0] * 8])
    v = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]])
    o, lse = oracle.attention_rows(q, k, v, 1.0, False, [0])
    assert np.all(np.isfinite(o)) and np.isfinite(lse[0])
    np.testing.assert_allclose(o[0], v[0], rtol=0, atol=1e-100)
    assert lse[0] == pytest.approx(12800.0, abs=1e-9)


def test_rows_entry_point_matches_full():
    rng = np.random.default_rng(18)
    q, k, v = (rng.normal(size=(300, 8)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, 0.35, True, row_block=64)
    rows = [0, 1, 63, 64, 65, 200, 299]
    o_r, lse_r = oracle.attention_rows(q, k, v, 0.35, True, rows)
    np.testing.assert_array_equal(o_r, o[rows])
    np.testing.assert_array_equal(lse_r, lse[rows])


def test_row_without_visible_key_is_rejected():
    # the pages leave a row with no permitted key to an explicit caller policy;
    # the oracle refuses it rather than inventing a value
    q = np.zeros((1, 2))
    with pytest.raises(ValueError):
        oracle.attention_rows(q, np.zeros((0, 2)), np.zeros((0, 2)), 1.0, False, [0])


# ---------------------------------------------------------------------------
# Merge of partial results over key ranges (split-key exchange step)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("splits", [[0, 50, 100], [0, 1, 2, 99, 100], [0, 33, 34, 70, 100]])
def test_merge_partials_equals_unsplit(splits):
    rng = np.random.default_rng(19)
    q, k, v = (rng.normal(size=(100, 8)) * 2 for _ in range(3))
    o_ref, lse_ref = oracle.attention(q, k, v, 0.4, False)
    outs, lses = [], []
    for a, b in zip(splits[:-1], splits[1:]):
        o_r, lse_r = oracle.attention_rows(q, k[a:b], v[a:b], 0.4, False, np.arange(100))
        outs.append(o_r)
        lses.append(lse_r)
    o, lse = oracle.merge_partials(outs, lses)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
