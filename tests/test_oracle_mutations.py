"""Planted mistakes: each mutant of the oracle must fail at least one pin.

A copy of oracle/attention.py is edited in memory (a dropped term, a wrong
sign or index, a transposed operand, a wrong log base ...), loaded as a
separate module, and the pin suite of test_oracle_pins.py is run against it.
The real oracle is never modified.  This shows that the pins constrain every
step of the oracle, not only that the oracle passes them.
"""
import importlib
import inspect
import os
import types

import pytest

real = importlib.import_module("oracle.attention")  # the module, not the function of that name
from tests import test_oracle_pins as pins

SRC_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "oracle", "attention.py")

MUTATIONS = {
    "transposed_scores": ("s = scale * (q[rows] @ k.T)", "s = scale * (k[rows] @ q.T)"),
    "scale_dropped": ("s = scale * (q[rows] @ k.T)", "s = (q[rows] @ k.T)"),
    "causal_off_by_one": ("return j <= rows[:, None]", "return j < rows[:, None]"),
    "causal_flipped": ("return j <= rows[:, None]", "return j >= rows[:, None]"),
    "causal_bottom_right": ("return j <= rows[:, None]", "return j <= rows[:, None] + (n_keys - rows.size)"),
    "max_shift_dropped": ("e = np.exp(s - m)  ", "e = np.exp(s)  "),
    "sum_wrong_axis": ("l = np.sum(e, axis=1, keepdims=True)", "l = np.sum(e, axis=0, keepdims=True)"),
    "no_normalisation": ("o = (e @ v) / l  ", "o = (e @ v)  "),
    "keys_as_values": ("o = (e @ v) / l  ", "o = (e @ k) / l  "),
    "lse_log2": ("lse = m[:, 0] + np.log(l[:, 0])", "lse = m[:, 0] + np.log2(l[:, 0])"),
    "lse_without_max": ("lse = m[:, 0] + np.log(l[:, 0])", "lse = np.log(l[:, 0])"),
    "tiled_alpha_dropped_on_acc": ("acc = alpha[:, None] * acc + p @ v[cols]", "acc = acc + p @ v[cols]"),
    "tiled_alpha_dropped_on_l": ("l = alpha * l + np.sum(p, axis=1)", "l = l + np.sum(p, axis=1)"),
    "tiled_alpha_sign": ("alpha = np.where(live, np.exp(m - m_use), 1.0)",
                         "alpha = np.where(live, np.exp(m_use - m), 1.0)"),
    "tiled_causal_off_by_one": ("s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)",
                                "s = np.where(cols[None, :] < rows[:, None], s, -np.inf)"),
    "tiled_lse_log2": ("L[rows] = m + np.log(l)", "L[rows] = m + np.log2(l)"),
    "online_rescale_dropped": ("l = l * math.exp(m - m_new) + math.exp(xi - m_new)",
                               "l = l + math.exp(xi - m_new)"),
    "merge_rescale_dropped": ("return m, la * math.exp(ma - m) + lb * math.exp(mb - m)",
                              "return m, la + lb"),
    "partials_weight_sign": ("w = [np.exp(x - m) for x in lses]", "w = [np.exp(m - x) for x in lses]"),
    "safe_softmax_no_division": ("return e / l                      # pass 3",
                                 "return e                          # pass 3"),
}


def _mutant(name):
    old, new = MUTATIONS[name]
    with open(SRC_PATH) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def _golden_loader():
    import json
    from tests.conftest import GOLDEN

    def load(fname):
        with open(os.path.join(GOLDEN, fname)) as f:
            return json.load(f)

    return load


def _pin_calls():
    """Every pin test with concrete arguments, as zero-argument callables."""
    calls = []
    for fname, fn in inspect.getmembers(pins, inspect.isfunction):
        if not fname.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        grids = [m.args for m in marks if m.name == "parametrize"]
        combos = [{}]
        for argnames, values in grids:
            names = [a.strip() for a in argnames.split(",")]
            new = []
            for c in combos:
                for val in values:
                    vals = val if len(names) > 1 else (val,)
                    d = dict(c)
                    d.update(zip(names, vals))
                    new.append(d)
            combos = new
        params = inspect.signature(fn).parameters
        for c in combos:
            kw = dict(c)
            if "golden" in params:
                kw["golden"] = _golden_loader()
            calls.append((fname, fn, kw))
    return calls


def test_real_oracle_passes_every_pin_call():
    for fname, fn, kw in _pin_calls():
        fn(**kw)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(name, monkeypatch):
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
