"""The comparison rules of tests/parity.py on hand-made cases (CPU): what
they accept and what they must reject."""
import numpy as np
import pytest

import oracle
import parity


def test_e4m3_boundary_rule_relative_window():
    # 1.5 * 2^-9 is the midpoint between the subnormal codes 1 (2^-9) and
    # 2 (2^-8); RNE gives code 2 at the midpoint, code 1 just below it.
    mid = 1.5 * 2.0 ** -9
    below = mid * (1 - 2.0 ** -10)          # within 2^-8 of the midpoint
    assert oracle.to_e4m3([below])[0] == 1
    ref = np.array([below])
    assert parity.check_e4m3(np.array([2], np.uint8), np.array([1], np.uint8), ref) == 1
    # far from the midpoint, with no large values to raise the floor: rejected
    far = np.array([mid * 0.9])
    with pytest.raises(AssertionError):
        parity.check_e4m3(np.array([2], np.uint8), np.array([1], np.uint8), far)


def test_e4m3_boundary_rule_rms_floor():
    """A value from a cancellation near zero, in a tensor whose values are
    ~8: the window is 2^-8 of 1% of the RMS, so a code that a fp32 result
    0.4% below the midpoint rounds the other way is accepted; a code two
    steps away, or one step away far from any midpoint, is not."""
    mid = 1.5 * 2.0 ** -9
    r = mid * (1 - 4e-3)
    big = np.full(99, 8.0)
    ref = np.concatenate([[r], big])
    want = oracle.to_e4m3(ref)
    got = want.copy()
    got[0] = 2
    assert want[0] == 1
    assert parity.check_e4m3(got, want, ref) == 1
    got[0] = 3  # not adjacent
    with pytest.raises(AssertionError):
        parity.check_e4m3(got, want, ref)
    # one step away from a value in the middle of its code interval
    ref2 = ref.copy()
    ref2[1] = 8.25  # between the adjacent codes of 8 and 9, a quarter step from 8
    want2 = oracle.to_e4m3(ref2)
    got2 = want2.copy()
    got2[1] = want2[1] + 1
    with pytest.raises(AssertionError):
        parity.check_e4m3(got2, want2, ref2)


def test_bf16_rule_and_unfloored_report():
    ref = np.array([1.0, -2.0, 1e-6, 3.0])
    got = oracle.to_bf16_bits(ref * np.array([1.01, 1.0, 3.0, 1.0]))
    st = parity.check_bf16(got, ref)          # 1e-6 tripled: inside the RMS floor
    assert st["n_above_2e-2_unfloored"] == 1  # ... but reported unfloored
    assert st["max_rel_unfloored"] == pytest.approx(2.0, rel=1e-2)
    with pytest.raises(AssertionError):
        parity.check_bf16(oracle.to_bf16_bits(ref * np.array([1.05, 1, 1, 1])), ref)
