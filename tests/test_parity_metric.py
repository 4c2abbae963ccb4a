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
    assert st["max_excess_from2"] <= 1e-12
    assert_close(st)


def test_far_neighbour_at_large_values_fails():
    # at |O| >= 2 the far bf16 neighbour of a value close to a grid point is
    # about one spacing (0.0156 at [2, 4)) worse than the nearest one
    ref = _ref([2.0005])
    assert_close(compare(_bf16([2.0]), torch.zeros(1), ref, np.zeros(1)))
    with pytest.raises(AssertionError):
        assert_close(compare(_bf16([2.015625]), torch.zeros(1), ref, np.zeros(1)))


def test_plain_bound_below_two():
    # below 2 the plain difference is held to 1e-2: 1.99 returned as 1.976
    # (one grid step of 2^-7 below the nearest value 1.9921875) is 0.014 off
    ref = _ref([1.99])
    assert_close(compare(_bf16([1.99]), torch.zeros(1), ref, np.zeros(1)))
    bad = torch.tensor(np.concatenate([[1.9765625], PAD])).to(torch.bfloat16)
    assert bad[0].item() == 1.9765625
    with pytest.raises(AssertionError):
        assert_close(compare(bad, torch.zeros(1), ref, np.zeros(1)))
    # the far neighbour of 0.5001 (0.50390625) is within 1e-2: the plain bound
    # holds it, the mean catches a systematic far neighbour (next test)
    ref = _ref([0.5001])
    assert_close(compare(_bf16([0.50390625]), torch.zeros(1), ref, np.zeros(1)))


def test_far_neighbour_everywhere_breaks_the_mean():
    # a kernel that returned the far bf16 neighbour of every element would be
    # about one spacing off on each: at |O| ~ 0.75 that is 2^-8 = 0.0039 per
    # element, above the 1e-3 bound on the plain mean
    ref = np.linspace(0.5, 0.99, 4001) + 1e-5
    rn = torch.tensor(ref).to(torch.bfloat16).double().numpy()
    spacing = 2.0 ** (np.floor(np.log2(rn)) - 7)  # bf16 keeps 8 significant bits
    far = torch.tensor(np.where(rn >= ref, rn - spacing, rn + spacing)).to(torch.bfloat16)
    assert np.all(np.abs(far.double().numpy() - ref) > np.abs(rn - ref))
    st = compare(far, torch.zeros(1), ref, np.zeros(1))
    assert st["max_do_raw_below2"] <= 1e-2
    with pytest.raises(AssertionError):
        assert_close(st)
    assert_close(compare(torch.tensor(ref).to(torch.bfloat16), torch.zeros(1), ref, np.zeros(1)))


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
