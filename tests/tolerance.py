"""The parity rule for floating-point outputs of the MoE block.

Stated for the block's BF16 outputs: at least 99.5% of the elements within one
BF16 ulp of the oracle value, and every element within relative error 1e-2
with absolute error 1e-3 near zero.

Reading of the second clause: |err| <= 1e-3 + 1e-2 * s, the usual closeness
form, where s is the magnitude the relative error is measured against.  For
an output out = bf16(bf16(R) + ys) (routed part R, shared part ys), s is the
largest of |out|, |R| and |ys|: an output is "near zero" when the two parts
cancel, and then its error is that of the parts (one bf16 ulp of R or ys
under any valid fp32 summation order), not a fraction of the tiny result.
Without cancellation s = |out| and the clause is the plain relative bound.

The first clause's ulp is read at the same s: the ulp of the largest of
|out|, |R| and |ys|.  Each part may differ from the oracle's exact sums by
one of its own ulps under a valid fp32 order, and one such difference in a
large shared-expert activation moves every output of its token by about an
ulp of ys; where the parts add with the same sign, s = |out| and the clause
is the plain one.
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


def operand_scale(res: dict) -> np.ndarray:
    """max(|bf16(R)|, |ys|) per output element from the oracle's
    intermediates (y [n, k, H], tw [n, k], ys [n, H]); R is re-summed in fp32
    in rank order exactly as the block defines it."""
    y = bits_to_f64(res["y"]).astype(np.float32)
    tw = res["tw"].astype(np.float32)
    R = np.zeros(y.shape[::2], dtype=np.float32)
    for j in range(y.shape[1]):
        R = (R + (tw[:, j:j + 1] * y[:, j, :]).astype(np.float32)).astype(np.float32)
    Rb = (np.ascontiguousarray(R).view(np.uint32) + 0x7FFF + ((np.ascontiguousarray(R).view(np.uint32) >> 16) & 1)) >> 16
    Rb = bits_to_f64(Rb.astype(np.uint16))
    return np.maximum(np.abs(Rb), np.abs(bits_to_f64(res["ys"])))


def check_bf16(got_bits, ref_bits, what: str = "out", scale=None) -> dict:
    """Apply the rule; raise AssertionError with a summary on failure.
    `scale` (optional, same shape) is the operand magnitude of each element
    (see the module docstring); the ulp and the relative term are taken at
    max(|ref|, scale)."""
    got = bits_to_f64(got_bits)
    ref = bits_to_f64(ref_bits)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return {"n": 0}
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref)
    ulp_at = ref if scale is None else np.maximum(np.abs(ref), np.asarray(scale, np.float64))
    within = err <= bf16_ulp(ulp_at)
    frac = float(within.mean())
    mag = np.abs(ref) if scale is None else np.maximum(np.abs(ref), np.asarray(scale, np.float64))
    bound = ABS + REL * mag
    bad = err > bound
    literal = err > ABS + REL * np.abs(ref)
    stats = {"n": int(err.size), "frac_within_ulp": frac, "n_exact": int((err == 0).sum()),
             "n_bound_violations": int(bad.sum()), "n_outside_plain_relative": int(literal.sum()),
             "max_abs_err": float(err.max())}
    assert frac >= FRAC_WITHIN_ULP, f"{what}: only {frac:.5f} within 1 ulp ({stats})"
    if bad.any():
        i = np.flatnonzero(bad.ravel())[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} elements outside 1e-3 + 1e-2 s: "
            f"idx {i.tolist()} got {got.ravel()[i].tolist()} ref {ref.ravel()[i].tolist()} ({stats})")
    return stats
