"""Planted mistakes in the backward oracle: each must fail at least one pin.

A copy of oracle/attention_backward.py is edited in memory, loaded as a
separate module and the pins of test_oracle_backward_pins.py are run against
it (the forward oracle they use stays the real one).  The real oracle is
never modified.
"""
import importlib
import os
import types

import pytest

from tests import test_oracle_backward_pins as pins
from tests.test_oracle_mutations import _pin_calls as _forward_pin_calls  # same collector

real = importlib.import_module("oracle.attention_backward")

SRC_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "oracle", "attention_backward.py")

MUTATIONS = {
    "row_term_dropped": ("ds = p * (dp - row_term)  ", "ds = p * dp  "),
    "row_term_sign": ("ds = p * (dp - row_term)  ", "ds = p * (dp + row_term)  "),
    "dv_scaled": ("dv += p.T @ do[rows]", "dv += scale * (p.T @ do[rows])"),
    "dp_with_keys": ("dp = do[rows] @ v.T  ", "dp = do[rows] @ k.T[:do.shape[1]]  "),
    "dq_scale_dropped": ("dq[rows] = scale * (ds @ k)", "dq[rows] = (ds @ k)"),
    "dq_with_values": ("dq[rows] = scale * (ds @ k)", "dq[rows] = scale * (ds @ v[:, :k.shape[1]])"),
    "dk_scale_dropped": ("dk += scale * (ds.T @ q[rows])", "dk += (ds.T @ q[rows])"),
    "dk_from_p": ("dk += scale * (ds.T @ q[rows])", "dk += scale * (p.T @ q[rows])"),
    "scores_unscaled": ("s = np.where(vis, scale * (q[rows] @ k.T), -np.inf)",
                        "s = np.where(vis, (q[rows] @ k.T), -np.inf)"),
    "causal_off_by_one": ("return j <= rows[:, None]", "return j < rows[:, None] + (rows[:, None] == 0)"),
    "softmax_not_normalised": ("return e / np.sum(e, axis=1, keepdims=True)", "return e"),
    "rowdot_wrong_operand": ("return np.sum(_f64(do) * _f64(o), axis=-1)",
                             "return np.sum(_f64(do) * _f64(do), axis=-1)"),
    "tiled_lse_sign": ("p = np.exp(s - lse[rows][:, None])", "p = np.exp(lse[rows][:, None] - s)"),
    "tiled_lse_dropped": ("p = np.exp(s - lse[rows][:, None])", "p = np.exp(s)"),
    "tiled_D_dropped": ("ds = p * (dp - D[rows][:, None])", "ds = p * dp"),
    "tiled_causal_flipped": ("s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)",
                             "s = np.where(cols[None, :] >= rows[:, None], s, -np.inf)"),
    "tiled_dk_dropped_scale": ("dk[cols] += scale * (ds.T @ q[rows])", "dk[cols] += (ds.T @ q[rows])"),
    "tiled_dq_transposed": ("dq[rows] += scale * (ds @ k[cols])", "dq[rows] += scale * (ds @ k[cols][::-1])"),
}


def _mutant(name):
    old, new = MUTATIONS[name]
    with open(SRC_PATH) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mod = types.ModuleType(f"oracle_backward_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def _pin_calls():
    import tests.test_oracle_mutations as fm
    saved = fm.pins
    fm.pins = pins
    try:
        return _forward_pin_calls()
    finally:
        fm.pins = saved


def test_real_backward_oracle_passes_every_pin_call():
    calls = _pin_calls()
    assert len(calls) > 40
    for fname, fn, kw in calls:
        fn(**kw)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_backward_mutant_is_caught(name, monkeypatch):
    mutant = _mutant(name)
    shim = types.ModuleType("oracle_shim")
    for attr in real.__all__:
        setattr(shim, attr, getattr(mutant, attr))
    monkeypatch.setattr(pins, "oracle", shim)
    caught = []
    for fname, fn, kw in _pin_calls():
        try:
            fn(**kw)
        except Exception:  # assertion or numerical failure both count as caught
            caught.append(fname)
    assert caught, f"mutation {name} passed every pin"
