"""The parity rule itself (tests/tolerance.py), on constructed values: what it
accepts and what it rejects, so that a change to the rule shows up here."""
from __future__ import annotations

import numpy as np
import pytest

from tolerance import bf16_ulp, check_bf16


def bits(values) -> np.ndarray:
    """bf16 bit patterns of exactly representable values."""
    a = np.asarray(values, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def test_ulp_is_the_bf16_spacing():
    assert bf16_ulp(np.array([1.0]))[0] == 2.0 ** -7
    assert bf16_ulp(np.array([0.75]))[0] == 2.0 ** -8
    assert bf16_ulp(np.array([-3.0]))[0] == 2.0 ** -6
    assert bf16_ulp(np.array([0.0]))[0] == 2.0 ** -133


def test_one_ulp_passes_two_ulps_fail_without_a_scale():
    ref = np.full(1000, 1.0)
    one = np.full(1000, 1.0 + 2.0 ** -7)
    check_bf16(bits(one), bits(ref))
    two = np.full(1000, 1.0 + 2.0 ** -6)
    with pytest.raises(AssertionError, match="within 1 ulp"):
        check_bf16(bits(two), bits(ref))


def test_half_a_percent_may_be_off_by_more_than_an_ulp():
    ref = np.full(1000, 1.9375)
    got = ref.copy()
    got[:5] = 1.9375 + 2.0 ** -6  # 0.5 % of the elements: two ulps, inside the 1e-2 bound
    check_bf16(bits(got), bits(ref))
    got[:6] = 1.9375 + 2.0 ** -6  # 0.6 %
    with pytest.raises(AssertionError, match="within 1 ulp"):
        check_bf16(bits(got), bits(ref))


def test_bound_violation_is_reported_even_when_rare():
    ref = np.full(1000, 1.0)
    got = ref.copy()
    got[0] = 1.0625  # 6 %: outside 1e-3 + 1e-2
    with pytest.raises(AssertionError, match="outside"):
        check_bf16(bits(got), bits(ref))


def test_bound_is_taken_at_the_output_itself():
    """1e-3 + 1e-2 |ref|: near zero the absolute term decides, elsewhere the
    relative one, both at the oracle value of the output (no operand scale)."""
    n = 1000
    # near zero: 2^-10 (~9.8e-4) off a value of 2^-12 is inside, 2^-9 is not
    ref = np.full(n, 2.0 ** -12)
    got = ref.copy()
    got[0] = 2.0 ** -12 + 2.0 ** -10
    st = check_bf16(bits(got), bits(ref))
    assert st["n_outside"] == 0
    got[0] = 2.0 ** -12 + 2.0 ** -9
    with pytest.raises(AssertionError, match="outside"):
        check_bf16(bits(got), bits(ref))
    # two ulps at 0.25 are 1.6 %: outside, even though the element's parts
    # may be larger than the output
    ref2 = np.full(n, 0.25)
    got2 = ref2.copy()
    got2[0] = 0.25 + 2.0 ** -8
    with pytest.raises(AssertionError, match="outside"):
        check_bf16(bits(got2), bits(ref2))


def test_allowance_is_explicit_and_counted():
    ref = np.full(1000, 1.0)
    got = ref.copy()
    got[:2] = 1.0625
    st = check_bf16(bits(got), bits(ref), allow_outside=2)
    assert st["n_outside"] == 2
    with pytest.raises(AssertionError, match="outside"):
        check_bf16(bits(got), bits(ref), allow_outside=1)
