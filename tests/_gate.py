"""The parity gate shared by the tests.

err = |C - Cref| / (|alpha| * D + |beta * Cin|) elementwise, where D is the
oracle's sum of |a_ik| * |b_kj|.  With beta = 0 and |alpha| <= 1 this is at
least the bare |C - Cref| / D of the stated bound, so gating on it is never
looser.  The beta * Cin term keeps the fp32 rounding of the final
alpha * acc + beta * c sum from being measured against a tiny D (for example
K = 1); where the whole denominator is zero the result must be exact.
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


def errors(C, Cref, D, alpha=1.0, beta=0.0, Cin=None):
    C = np.asarray(C, dtype=np.float64)
    Cref = np.asarray(Cref, dtype=np.float64)
    scale = abs(alpha) * np.asarray(D, dtype=np.float64)
    if beta != 0.0:
        scale = scale + np.abs(beta * np.asarray(Cin, dtype=np.float64))
    diff = np.abs(C - Cref)
    bad_nan = np.isnan(C) != np.isnan(Cref)
    with np.errstate(divide="ignore", invalid="ignore"):
        err = np.where(scale > 0, diff / np.where(scale > 0, scale, 1.0), np.where(diff > 0, np.inf, 0.0))
    err = np.where(bad_nan, np.inf, np.nan_to_num(err, nan=0.0))
    return err


def max_err(C, Cref, D, alpha=1.0, beta=0.0, Cin=None):
    e = errors(C, Cref, D, alpha, beta, Cin)
    return float(e.max()) if e.size else 0.0


def assert_within(mode, C, Cref, D, alpha=1.0, beta=0.0, Cin=None, what=""):
    e = errors(C, Cref, D, alpha, beta, Cin)
    if e.size == 0:
        return 0.0
    worst = float(e.max())
    if not worst <= TOL[mode]:
        idx = np.unravel_index(int(np.argmax(e)), e.shape)
        raise AssertionError(
            f"{what} {mode}: max err {worst:.3e} > {TOL[mode]:.1e} at {idx}: "
            f"got {np.asarray(C)[idx]!r}, want {np.asarray(Cref)[idx]!r}")
    return worst
