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


def test_operand_scale_reads_the_ulp_of_the_larger_part():
    """out = bf16(bf16(R) + ys) with R = -0.125, ys = 0.0859375: out = -0.0390625.
    One ulp of the larger part (2^-10 at 0.125) is four ulps of out (2^-12):
    accepted at the operand scale, rejected at the output's own ulp."""
    n = 1000
    ref = np.full(n, -0.0390625)
    got = np.full(n, -0.0390625 - 2.0 ** -10)
    scale = np.full(n, 0.125)
    check_bf16(bits(got), bits(ref), scale=scale)
    with pytest.raises(AssertionError, match="within 1 ulp"):
        check_bf16(bits(got), bits(ref))
    # same-sign parts: the scale is |out| itself and the clause is the plain one
    ref2 = np.full(n, 0.25)
    got2 = np.full(n, 0.25 + 2.0 ** -8)  # two ulps of 0.25
    with pytest.raises(AssertionError, match="within 1 ulp"):
        check_bf16(bits(got2), bits(ref2), scale=np.full(n, 0.25))
