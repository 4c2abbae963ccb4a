"""Planted mistakes in the FP8 oracle: each must fail at least one pin.

A copy of oracle/fp8.py is edited in memory, loaded as a separate module and
the pins of test_oracle_fp8_pins.py run against it.
"""
import importlib
import os
import types

import pytest

real_attention = importlib.import_module("oracle.attention")  # the module, not the function
from tests import test_oracle_fp8_pins as pins
from tests.test_oracle_mutations import _pin_calls as _collect

SRC_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "fp8.py")

MUTATIONS = {
    "ties_away_from_zero": ("up = (frac > 0.5) | ((frac == 0.5) & (np.mod(r, 2.0) == 1.0))", "up = frac >= 0.5"),
    "truncate": ("up = (frac > 0.5) | ((frac == 0.5) & (np.mod(r, 2.0) == 1.0))", "up = frac > 2.0"),
    "no_saturation": ("mag = np.minimum(r * step, E4M3_MAX)", "mag = r * step"),
    "two_mantissa_bits": ("step = np.where(normal, 2.0 ** (e - 3), _SUB_STEP)",
                          "step = np.where(normal, 2.0 ** (e - 2), _SUB_STEP)"),
    "subnormal_step": ("step = np.where(normal, 2.0 ** (e - 3), _SUB_STEP)",
                       "step = np.where(normal, 2.0 ** (e - 3), 2.0 * _SUB_STEP)"),
    "scale_to_240": ("s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0))",
                     "s = np.where(amax > 0, amax / np.float32(240.0), np.float32(1.0))"),
    "zero_block_scale_0": ("s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0))",
                           "s = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(0.5))"),
    "multiply_by_scale": ("codes[..., r0:r1, :] = e4m3_round((blk / s[..., None, None]).astype(np.float32))",
                          "codes[..., r0:r1, :] = e4m3_round((blk * s[..., None, None]).astype(np.float32))"),
    "dequant_wrong_block": ("s = np.repeat(np.asarray(scales, dtype=np.float64), rows_per_scale, axis=-1)[..., : codes.shape[-2]]",
                            "s = np.repeat(np.asarray(scales, dtype=np.float64)[..., ::-1], rows_per_scale, axis=-1)[..., : codes.shape[-2]]"),
    "v_unscaled": ("    v = dequantize_blocks(v8, sv, v_rows)", "    v = np.asarray(v8, dtype=np.float64)"),
}


def _mutant(name):
    old, new = MUTATIONS[name]
    with open(SRC_PATH) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mod = types.ModuleType(f"oracle_fp8_mutant_{name}")
    mod.__dict__["__package__"] = "oracle"
    src = src.replace("from .attention import attention", "")
    mod.__dict__["attention"] = real_attention.attention
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def _pin_calls():
    import tests.test_oracle_mutations as fm
    saved = fm.pins
    fm.pins = pins
    try:
        return _collect()
    finally:
        fm.pins = saved


def test_real_fp8_oracle_passes_every_pin_call():
    calls = _pin_calls()
    assert len(calls) >= 9
    for _, fn, kw in calls:
        fn(**kw)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_fp8_mutant_is_caught(name, monkeypatch):
    monkeypatch.setattr(pins, "fp8", _mutant(name))
    caught = []
    for fname, fn, kw in _pin_calls():
        try:
            fn(**kw)
        except Exception:
            caught.append(fname)
    assert caught, f"mutation {name} passed every pin"
