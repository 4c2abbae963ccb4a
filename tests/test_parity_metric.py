"""The comparison helper itself (CPU): what it accepts and what it rejects."""
import numpy as np
import pytest
import torch

from tests.parity import assert_close, compare


PAD = np.zeros(4000)  # exact values, so that the mean reflects a whole tensor


def _bf16(x):
    return torch.tensor(np.concatenate([np.asarray(x, float), PAD])).to(torch.bfloat16)


def _ref(x):
    return np.concatenate([np.asarray(x, float), PAD])


def test_correctly_rounded_large_values_pass():
    # 4.0162 has no bf16 neighbour within 1e-2; its nearest bf16 (4.03125) passes
    ref = _ref([4.0162, -5.37, 0.3])
    st = compare(_bf16([4.0162, -5.37, 0.3]), torch.zeros(1), ref, np.zeros(1))
    assert st["max_do_raw"] > 1e-2
    assert st["max_do"] <= 1e-12
    assert_close(st)


def test_one_ulp_flip_below_four_passes_only_near_a_midpoint():
    # 2.0078 sits near the midpoint of 2.0 and 2.015625: either neighbour is fine
    ref = _ref([2.0078])
    assert_close(compare(_bf16([2.0]), torch.zeros(1), ref, np.zeros(1)))
    # 2.0005 is far from the midpoint: returning the far neighbour is 0.0146
    # worse than the nearest bf16 value
    ref = _ref([2.0005])
    with pytest.raises(AssertionError):
        assert_close(compare(_bf16([2.015625]), torch.zeros(1), ref, np.zeros(1)))


def test_errors_are_caught():
    ref = _ref([0.5, 0.25])
    assert_close(compare(_bf16([0.5, 0.25]), torch.zeros(1), ref, np.zeros(1)))
    with pytest.raises(AssertionError):
        assert_close(compare(_bf16([0.5, 0.27]), torch.zeros(1), ref, np.zeros(1)))
    with pytest.raises(AssertionError):
        assert_close(compare(_bf16([0.5, 0.25]), torch.tensor([0.002]), ref, np.zeros(1)))
    with pytest.raises(AssertionError):
        assert_close(compare(_bf16([0.5, float("nan")]), torch.zeros(1), ref, np.zeros(1)))
    # a small bias on every element breaks the mean bar before the max bar
    ref = np.linspace(-1, 1, 1000)
    biased = torch.tensor(ref + 0.003).to(torch.bfloat16)
    with pytest.raises(AssertionError):
        assert_close(compare(biased, torch.zeros(1), ref, np.zeros(1)))
