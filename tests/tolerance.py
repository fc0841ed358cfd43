"""The parity rule for the BF16 outputs of the MoE block, read literally.

The rule: at least 99.5% of the elements lie within one BF16 ulp of the
oracle value, and every element lies within relative error 1e-2, with
absolute error 1e-3 near zero.

Both clauses are measured at the oracle value ref of each element:
  - one ulp is the BF16 spacing at |ref|;
  - the bound is |err| <= 1e-3 + 1e-2 * |ref|.
The bound uses the usual closeness form: absolute 1e-3 near zero, relative
1e-2 elsewhere, both at the output itself.

check_bf16 always reports how many elements lie outside the bound
(n_outside). By default it asserts that there are none. A test of a path
that does not meet the every-element clause has to pass its own allowance,
and has to say why.
"""
from __future__ import annotations

import numpy as np

FRAC_WITHIN_ULP = 0.995
REL = 1e-2
ABS = 1e-3


def bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_ulp(ref: np.ndarray) -> np.ndarray:
    """ulp of each bf16 value (2^(e-7) for |v| in [2^e, 2^(e+1)); subnormals
    and zero use the subnormal spacing 2^-133)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    u = np.exp2(e - 7)
    return np.where(a >= 2.0 ** -126, u, 2.0 ** -133)


def stats_bf16(got_bits, ref_bits) -> dict:
    """The rule's statistics for one comparison (no assertion)."""
    got = bits_to_f64(got_bits)
    ref = bits_to_f64(ref_bits)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return {"n": 0, "frac_within_ulp": 1.0, "n_exact": 0, "n_outside": 0, "max_abs_err": 0.0}
    assert np.isfinite(got).all(), "non-finite values"
    err = np.abs(got - ref)
    within = err <= bf16_ulp(ref)
    outside = err > ABS + REL * np.abs(ref)
    st = {"n": int(err.size), "frac_within_ulp": float(within.mean()), "n_exact": int((err == 0).sum()),
          "n_outside": int(outside.sum()), "max_abs_err": float(err.max())}
    if outside.any():
        i = np.flatnonzero(outside.ravel())[:5]
        st["outside_examples"] = list(zip(got.ravel()[i].tolist(), ref.ravel()[i].tolist()))
    return st


def check_bf16(got_bits, ref_bits, what: str = "out", allow_outside: int = 0) -> dict:
    """Assert the rule: the 1-ulp fraction >= 99.5 % and at most
    `allow_outside` elements (0 = the rule as stated) outside
    1e-3 + 1e-2 |ref|.  Returns the statistics."""
    st = stats_bf16(got_bits, ref_bits)
    assert st["frac_within_ulp"] >= FRAC_WITHIN_ULP, f"{what}: only {st['frac_within_ulp']:.5f} within 1 ulp ({st})"
    assert st["n_outside"] <= allow_outside, f"{what}: {st['n_outside']} elements outside 1e-3 + 1e-2 |ref| ({st})"
    return st
