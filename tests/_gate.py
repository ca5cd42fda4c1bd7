"""The parity gate shared by the tests.

The stated bound is err = |C - Cref| / (|alpha| * D) elementwise, where D is
the oracle's sum of |a_ik| * |b_kj|.  It bounds the error of the product; the
beta * Cin term adds none of its own except the rounding of the final fp32
result.  Every kernel of the library stores RN(beta * c + RN(alpha * acc)):
given its accumulator, the result differs from the exact alpha * acc +
beta * c by at most 2^-24 * |alpha * acc| (covered by the product's bound)
plus 2^-24 * |beta * c|.  So the gate is

    |C - Cref| - 2^-24 * |beta * Cin|  <=  tol * |alpha| * D,

which is the stated formula unchanged when beta = 0, and, where D = 0 (a
zero row or column of the product), requires the result to be beta * Cin
rounded once to fp32.  err' = |C - Cref| / (|alpha| * D + |beta * Cin|), the
beta-augmented error, is reported beside it and never gated on.
"""
import numpy as np

# FP8 (E4M3 operands): every product of two E4M3 values is exact in fp32 and
# the tensor cores accumulate in fp32, so a full-precision accumulation would
# stay near K / 32 * 2^-24 of D.  The gate allows the accumulator of one MMA
# to keep as few as 14 mantissa bits (2^-14 ~ 6e-5 of D per MMA of 32 terms)
# over K / 32 MMAs with random signs: sqrt(280) * 6e-5 ~ 1e-3 at K = 8960,
# doubled.  Dropped or doubled K blocks are caught separately, on
# non-negative operands, where one block of K = 8960 is 1.4e-2 of D.
TOL = {"fp32": 1e-6, "tf32": 2e-3, "bf16": 8e-3, "fp8": 2e-3}

# One rounding of an fp32 result (unit roundoff of binary32).
U32 = 2.0 ** -24


def _beta_c(beta, Cin, shape):
    if beta == 0.0 or Cin is None:
        return np.zeros(shape)
    return np.abs(beta * np.asarray(Cin, dtype=np.float64))


def errors(C, Cref, D, alpha=1.0, beta=0.0, Cin=None):
    """The gated error: (|C - Cref| - 2^-24 |beta Cin|)+ / (|alpha| D); inf
    where D = 0 and the difference exceeds that one rounding, or where only
    one side is NaN."""
    C = np.asarray(C, dtype=np.float64)
    Cref = np.asarray(Cref, dtype=np.float64)
    scale = abs(alpha) * np.asarray(D, dtype=np.float64)
    excess = np.maximum(np.abs(C - Cref) - U32 * _beta_c(beta, Cin, C.shape), 0.0)
    bad_nan = np.isnan(C) != np.isnan(Cref)
    with np.errstate(divide="ignore", invalid="ignore"):
        err = np.where(scale > 0, excess / np.where(scale > 0, scale, 1.0), np.where(excess > 0, np.inf, 0.0))
    err = np.where(bad_nan, np.inf, np.nan_to_num(err, nan=0.0))
    return err


def errors_augmented(C, Cref, D, alpha=1.0, beta=0.0, Cin=None):
    """err' = |C - Cref| / (|alpha| D + |beta Cin|), reported, not gated."""
    C = np.asarray(C, dtype=np.float64)
    Cref = np.asarray(Cref, dtype=np.float64)
    scale = abs(alpha) * np.asarray(D, dtype=np.float64) + _beta_c(beta, Cin, C.shape)
    diff = np.abs(C - Cref)
    with np.errstate(divide="ignore", invalid="ignore"):
        err = np.where(scale > 0, diff / np.where(scale > 0, scale, 1.0), np.where(diff > 0, np.inf, 0.0))
    return np.nan_to_num(err, nan=0.0)


def max_err(C, Cref, D, alpha=1.0, beta=0.0, Cin=None):
    e = errors(C, Cref, D, alpha, beta, Cin)
    return float(e.max()) if e.size else 0.0


def assert_within(mode, C, Cref, D, alpha=1.0, beta=0.0, Cin=None, what=""):
    """Gate on the stated bound; returns the worst gated error."""
    e = errors(C, Cref, D, alpha, beta, Cin)
    if e.size == 0:
        return 0.0
    worst = float(e.max())
    if not worst <= TOL[mode]:
        idx = np.unravel_index(int(np.argmax(e)), e.shape)
        aug = float(errors_augmented(C, Cref, D, alpha, beta, Cin).max())
        raise AssertionError(
            f"{what} {mode}: max err {worst:.3e} > {TOL[mode]:.1e} at {idx}: "
            f"got {np.asarray(C)[idx]!r}, want {np.asarray(Cref)[idx]!r} (err' {aug:.3e})")
    return worst
