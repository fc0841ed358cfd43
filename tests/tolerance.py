"""The parity rule for floating-point outputs of the MoE block.

Stated for the block's BF16 outputs: at least 99.5% of the elements within one
BF16 ulp of the oracle value, and every element within relative error 1e-2
with absolute error 1e-3 near zero.  The second clause is read with the usual
closeness semantics (numpy/torch isclose): |err| <= 1e-3 + 1e-2 * |ref|, so
the absolute term takes over as |ref| approaches zero.  The ulp is that of the
oracle (reference) value.
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


def check_bf16(got_bits, ref_bits, what: str = "out") -> dict:
    """Apply the rule; raise AssertionError with a summary on failure."""
    got = bits_to_f64(got_bits)
    ref = bits_to_f64(ref_bits)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return {"n": 0}
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref)
    within = err <= bf16_ulp(ref)
    frac = float(within.mean())
    bound = ABS + REL * np.abs(ref)
    bad = err > bound
    stats = {"n": int(err.size), "frac_within_ulp": frac, "n_exact": int((err == 0).sum()),
             "n_bound_violations": int(bad.sum()), "max_abs_err": float(err.max())}
    assert frac >= FRAC_WITHIN_ULP, f"{what}: only {frac:.5f} within 1 ulp ({stats})"
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} elements outside 1e-3 + 1e-2|ref|: "
            f"idx {i.tolist()} got {got.ravel()[i].tolist()} ref {ref.ravel()[i].tolist()} ({stats})")
    return stats
