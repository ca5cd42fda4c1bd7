"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties the oracle to a fact fixed by mathematics or by an independent
routine: exact rational arithmetic on tiny shapes, identity and permutation
matrices, integer products, a rank-one closed form, torch's float64 matmul,
the TF32 and bfloat16 formats from their definitions, and a hand-computed
example.  A wrong sign, a dropped term, a transposed operand or a missing
rounding step in the oracle fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import _gate

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TRANS = [(False, False), (False, True), (True, False), (True, True)]


# ---------------------------------------------------------------- formats
def _tf32_by_definition(x: float, rule: str) -> float:
    """TF32 from its definition: fp32's exponent range, 10 fraction bits.

    The spacing of TF32 values near |x| is 2^(e - 10) with e the binade of |x|
    (never below fp32's smallest normal binade, -126).  Truncation keeps the
    multiple of the spacing below |x|; nearest-away rounds half up in magnitude.
    """
    if x == 0.0 or math.isinf(x) or math.isnan(x):
        return x
    f = Fraction(x)
    mag = abs(f)
    e = max(math.frexp(x)[1] - 1, -126)
    q = Fraction(2) ** (e - 10)
    if rule == "truncate":
        n = mag // q
    else:
        n = (mag / q + Fraction(1, 2)).__floor__()
    r = n * q
    if r >= Fraction(2) ** 128:
        return math.copysign(math.inf, x)
    return math.copysign(float(r), x)


def _special_patterns():
    pats = [0x00000000, 0x80000000, 0x00000001, 0x00001000, 0x00001fff, 0x00002000,
            0x007fffff, 0x00800000, 0x3f800000, 0x3f801000, 0x3f802000, 0x3f803000,
            0x3f800fff, 0x3f801001, 0xbf801000, 0xbf803000, 0x7f7fffff, 0x7f7ff000,
            0x7f7fefff, 0xff7fffff, 0x3fffffff, 0x3ffff000, 0x4b7ff000]
    return np.array(pats, dtype=np.uint32)


@pytest.mark.parametrize("rule", ["truncate", "nearest_away"])
def test_tf32_reduction_matches_definition(rule):
    rng = np.random.default_rng(7)
    pats = rng.integers(0, 2**32, size=4000, dtype=np.uint64).astype(np.uint32)
    pats = np.concatenate([pats, _special_patterns()])
    x = pats.view(np.float32)
    x = x[np.isfinite(x)]
    got = oracle.tf32(x, rule)
    for xi, gi in zip(x.tolist(), got.tolist()):
        want = _tf32_by_definition(xi, rule)
        assert (gi == want and math.copysign(1, gi) == math.copysign(1, want)), (rule, xi, gi, want)


def test_tf32_passes_inf_and_nan():
    x = np.array([np.inf, -np.inf, np.nan], dtype=np.float32)
    for rule in ("truncate", "nearest_away"):
        got = oracle.tf32(x, rule)
        assert got[0] == np.inf and got[1] == -np.inf and np.isnan(got[2])


def test_tf32_rules_differ_only_at_half_spacing():
    # 1 + 2^-11 is exactly half a TF32 spacing above 1: truncation keeps 1,
    # nearest-away goes up to 1 + 2^-10.
    x = np.array([1 + 2.0 ** -11, 1 + 2.0 ** -11 - 2.0 ** -23], dtype=np.float32)
    assert oracle.tf32(x, "truncate").tolist() == [1.0, 1.0]
    assert oracle.tf32(x, "nearest_away").tolist() == [1 + 2.0 ** -10, 1.0]


def test_bf16_widening_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.bf16_to_f64(bits)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_e4m3_decoding_exhaustive():
    """All 256 codes against torch's float8_e4m3fn widening (a library
    routine the oracle does not use), plus values fixed by the format."""
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_f64(codes)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.flatnonzero(nan).tolist() == [0x7F, 0xFF]  # S.1111.111 only: no infinities
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    fixed = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5,
             0x40: 2.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in fixed.items():
        assert got[c] == v, hex(c)
    assert np.signbit(got[0x80]) and got[0x80] == 0.0
    # positive codes 0 .. 0x7E are strictly increasing; negatives mirror them
    assert np.all(np.diff(got[:0x7F]) > 0)
    assert np.array_equal(got[0x80:0xFF], -got[:0x7F])


def test_e5m2_decoding_exhaustive():
    """All 256 codes against torch's float8_e5m2 widening, plus values the
    format fixes (IEEE-style infinities and NaNs at exponent 31)."""
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e5m2_to_f64(codes)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e5m2).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.flatnonzero(nan).tolist() == [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))
    fixed = {0x00: 0.0, 0x01: 2.0 ** -16, 0x03: 3 * 2.0 ** -16, 0x04: 2.0 ** -14, 0x3C: 1.0, 0x3E: 1.5,
             0x40: 2.0, 0x7B: 57344.0, 0x7C: np.inf, 0xBC: -1.0, 0xFC: -np.inf}
    for c, v in fixed.items():
        assert got[c] == v, hex(c)
    assert np.all(np.diff(got[:0x7D]) > 0)
    assert np.array_equal(got[0x80:0xFD], -got[:0x7D])
    # E5M2 is E4M3's range traded for precision: every E5M2 value of
    # magnitude in [2^-6, 448] with one mantissa bit to spare is also E4M3
    e4 = set(oracle.e4m3_to_f64(codes[:0x7F]).tolist())
    for v in got[:0x7C]:
        if 2.0 ** -6 <= v <= 448.0:
            assert v in e4, v


FP8_MODES = ["fp8", "fp8_e5m2", "fp8_e4m3_e5m2", "fp8_e5m2_e4m3"]
_FP8_TORCH = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
_FP8_SIDES = {"fp8": ("e4m3", "e4m3"), "fp8_e5m2": ("e5m2", "e5m2"), "fp8_e4m3_e5m2": ("e4m3", "e5m2"),
              "fp8_e5m2_e4m3": ("e5m2", "e4m3")}


# ---------------------------------------------------------------- helpers
def _operands(mode, a, b):
    """numpy operands for the oracle plus their exact values as Fractions."""
    if mode in _FP8_SIDES:
        fa, fb = _FP8_SIDES[mode]
        (ca, _), (cb, _) = si.to_fp8(torch.from_numpy(a), fa), si.to_fp8(torch.from_numpy(b), fb)
        def widen(c, f):
            return torch.from_numpy(c.copy()).view(_FP8_TORCH[f]).to(torch.float64).numpy()
        return ca, cb, widen(ca, fa), widen(cb, fb)
    if mode == "bf16":
        ab, bb = si.to_bf16(torch.from_numpy(a)), si.to_bf16(torch.from_numpy(b))
        qa, qb = ab.to(torch.float64).numpy(), bb.to(torch.float64).numpy()
        return si.bf16_bits(ab), si.bf16_bits(bb), qa, qb
    if mode == "tf32":
        qa = np.vectorize(lambda v: _tf32_by_definition(float(v), oracle.DEFAULT_TF32_RULE))(a)
        qb = np.vectorize(lambda v: _tf32_by_definition(float(v), oracle.DEFAULT_TF32_RULE))(b)
        return a, b, qa, qb
    return a, b, a.astype(np.float64), b.astype(np.float64)


def _op(x, t):
    return x.T if t else x


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"] + FP8_MODES)
@pytest.mark.parametrize("tA,tB", TRANS)
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.5, 1.0), (-2.0, 0.25)])
def test_bruteforce_exact_rational(mode, tA, tB, alpha, beta):
    rng = np.random.default_rng(hash((mode, tA, tB, alpha)) % 2**32)
    M, N, K = 5, 6, 7
    a = rng.uniform(-1, 1, size=(K, M) if tA else (M, K)).astype(np.float32)
    b = rng.uniform(-1, 1, size=(N, K) if tB else (K, N)).astype(np.float32)
    c = rng.standard_normal((M, N)).astype(np.float32)
    A, B, qa, qb = _operands(mode, a, b)
    got, D = oracle.gemm(mode, A, B, transA=tA, transB=tB, alpha=alpha, beta=beta, C=c)
    oa, ob = _op(qa, tA), _op(qb, tB)
    for i in range(M):
        for j in range(N):
            s = sum(Fraction(float(oa[i, k])) * Fraction(float(ob[k, j])) for k in range(K))
            d = sum(abs(Fraction(float(oa[i, k])) * Fraction(float(ob[k, j]))) for k in range(K))
            exact = Fraction(alpha) * s + Fraction(beta) * Fraction(float(c[i, j]))
            bound = 2 * (K + 2) * 2.0 ** -53 * (abs(alpha) * float(d) + abs(beta * float(c[i, j])))
            assert abs(Fraction(float(got[i, j])) - exact) <= Fraction(bound), (i, j)
            assert abs(Fraction(float(D[i, j])) - d) <= Fraction(2 * K * 2.0 ** -53 * float(d))


def test_golden_hand_computed_example():
    """A 2x3 by 3x2 product written out by hand (tests/golden)."""
    path = os.path.join(GOLDEN, "hand_2x3x2.txt")
    blocks = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = line.split(":", 1)
            blocks[key.strip()] = [float(v) for v in vals.split()]
    A = np.array(blocks["A"], dtype=np.float32).reshape(2, 3)
    B = np.array(blocks["B"], dtype=np.float32).reshape(3, 2)
    C = np.array(blocks["C"], dtype=np.float32).reshape(2, 2)
    alpha, beta = blocks["alpha"][0], blocks["beta"][0]
    want = np.array(blocks["expected"]).reshape(2, 2)
    for mode in ("fp32", "tf32"):
        got, _ = oracle.gemm(mode, A, B, alpha=alpha, beta=beta, C=C)
        assert np.array_equal(got, want), mode
    got, _ = oracle.gemm("bf16", si.bf16_bits(si.to_bf16(torch.from_numpy(A))),
                         si.bf16_bits(si.to_bf16(torch.from_numpy(B))), alpha=alpha, beta=beta, C=C)
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- structure
@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"] + FP8_MODES)
def test_identity_and_permutation(mode):
    rng = np.random.default_rng(3)
    M, N = 9, 11
    b = rng.standard_normal((M, N)).astype(np.float32)
    c = rng.standard_normal((M, N)).astype(np.float32)
    eye = np.eye(M, dtype=np.float32)
    A, B, _, qb = _operands(mode, eye, b)
    got, _ = oracle.gemm(mode, A, B)
    assert np.array_equal(got, qb)
    got, _ = oracle.gemm(mode, A, B, alpha=0.5, beta=1.0, C=c)
    assert np.array_equal(got, 0.5 * qb + c.astype(np.float64))
    perm = rng.permutation(M)
    P = np.zeros((M, M), dtype=np.float32)
    P[np.arange(M), perm] = 1.0
    A, B, _, qb = _operands(mode, P, b)
    got, _ = oracle.gemm(mode, A, B)
    assert np.array_equal(got, qb[perm])
    # B = P^T on the right permutes columns of A
    A2, B2, qa2, _ = _operands(mode, b.T.copy(), P.T.copy())
    got, _ = oracle.gemm(mode, A2, B2)
    assert np.array_equal(got, qa2[:, perm])


@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"] + FP8_MODES)
@pytest.mark.parametrize("tA,tB", TRANS)
def test_small_integers_are_exact(mode, tA, tB):
    M, N, K = 40, 33, 1024
    a = si.integers((K, M) if tA else (M, K), 11).numpy()
    b = si.integers((N, K) if tB else (K, N), 12).numpy()
    A, B, _, _ = _operands(mode, a, b)
    got, D = oracle.gemm(mode, A, B, transA=tA, transB=tB)
    want = _op(a.astype(np.int64), tA) @ _op(b.astype(np.int64), tB)
    assert np.array_equal(got, want.astype(np.float64))
    assert np.array_equal(D, np.abs(_op(a.astype(np.int64), tA)) @ np.abs(_op(b.astype(np.int64), tB)))


def test_rank_one_closed_form():
    M, N, K = 13, 17, 300
    u = (np.arange(M, dtype=np.float32) - 6) / 4
    v = (np.arange(N, dtype=np.float32) - 8) / 8
    A = np.repeat(u[:, None], K, axis=1)
    B = np.repeat(v[None, :], K, axis=0)
    c = np.full((M, N), 3.0, dtype=np.float32)
    got, D = oracle.gemm("fp32", A, B, alpha=2.0, beta=-1.0, C=c)
    want = 2.0 * K * np.outer(u.astype(np.float64), v.astype(np.float64)) - 3.0
    assert np.array_equal(got, want)
    assert np.array_equal(D, K * np.abs(np.outer(u, v)).astype(np.float64))


@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"] + FP8_MODES)
def test_transpose_flags_match_explicit_transpose(mode):
    rng = np.random.default_rng(5)
    M, N, K = 19, 23, 29
    a = rng.standard_normal((M, K)).astype(np.float32)
    b = rng.standard_normal((K, N)).astype(np.float32)
    A, B, _, _ = _operands(mode, a, b)
    ref, _ = oracle.gemm(mode, A, B)
    for tA, tB in TRANS:
        At = np.ascontiguousarray(A.T) if tA else A
        Bt = np.ascontiguousarray(B.T) if tB else B
        got, _ = oracle.gemm(mode, At, Bt, transA=tA, transB=tB)
        assert np.array_equal(got, ref), (tA, tB)


def test_leading_dimensions_and_row_sampling():
    rng = np.random.default_rng(6)
    M, N, K = 12, 10, 8
    big = rng.standard_normal((M, K + 5)).astype(np.float32)
    a = big[:, :K]                       # lda = K + 5
    b = rng.standard_normal((K, N)).astype(np.float32)
    full, _ = oracle.gemm("fp32", a, b)
    part, _ = oracle.gemm("fp32", a, b, rows=(3, 9))
    assert np.array_equal(part, full[3:9])
    assert np.array_equal(full, oracle.gemm("fp32", np.ascontiguousarray(a), b)[0])


def test_matches_torch_float64_matmul():
    M, N, K = 64, 48, 512
    a = si.normal((M, K), 21).numpy()
    b = si.normal((K, N), 22).numpy()
    got, D = oracle.gemm("fp32", a, b)
    want = (torch.from_numpy(a).double() @ torch.from_numpy(b).double()).numpy()
    assert np.max(np.abs(got - want) / D) < 1e-12


# ---------------------------------------------------------------- conventions
def test_k_zero_and_alpha_zero_give_beta_c():
    c = np.arange(6, dtype=np.float32).reshape(2, 3)
    got, D = oracle.gemm("fp32", np.zeros((2, 0), np.float32), np.zeros((0, 3), np.float32),
                         alpha=1.0, beta=2.0, C=c)
    assert np.array_equal(got, 2.0 * c) and not D.any()
    nanA = np.full((2, 4), np.nan, dtype=np.float32)
    got, _ = oracle.gemm("fp32", nanA, np.ones((4, 3), np.float32), alpha=0.0, beta=-1.0, C=c)
    assert np.array_equal(got, -c.astype(np.float64))


def test_beta_zero_does_not_read_c():
    a = np.ones((2, 2), np.float32)
    got, _ = oracle.gemm("fp32", a, a, beta=0.0, C=np.full((2, 2), np.nan, np.float32))
    assert np.array_equal(got, np.full((2, 2), 2.0))


# ---------------------------------------------------------------- error model
def test_tf32_error_is_of_the_expected_size():
    """TF32 operands cost about 2^-11 relative error per product; FP32 about 2^-24.

    "bare-metal-bard" (first paragraph) puts TF32's error at thousands of
    times FP32's; the ratio of the unit roundoffs is 2^13 = 8192.
    """
    M, N, K = 64, 64, 1024
    a = si.normal((M, K), 31).numpy()
    b = si.normal((K, N), 32).numpy()
    ref, D = oracle.gemm("fp32", a, b)
    tf, _ = oracle.gemm("tf32", a, b)
    e_tf32 = np.abs(tf - ref) / D
    assert 1e-6 < np.max(e_tf32) < _gate.TOL["tf32"]
    sgemm = (torch.from_numpy(a) @ torch.from_numpy(b)).numpy().astype(np.float64)
    e_fp32 = np.abs(sgemm - ref) / D
    assert np.max(e_fp32) < _gate.TOL["fp32"]
    ratio = np.median(e_tf32) / max(np.median(e_fp32), 1e-30)
    assert 1e2 < ratio < 1e5, ratio


def test_gate_rejects_one_dropped_term():
    """The gate is not vacuous: an oracle with one k-term dropped fails it."""
    M, N, K = 32, 32, 256
    a = si.uniform((M, K), 41).numpy()
    b = si.uniform((K, N), 42).numpy()
    ref, D = oracle.gemm("fp32", a, b)
    broken, _ = oracle.gemm("fp32", a[:, 1:].copy(), b[1:, :].copy())  # planted: k = 0 dropped
    assert _gate.max_err(broken, ref, D) > _gate.TOL["bf16"]
    with pytest.raises(AssertionError):
        _gate.assert_within("fp32", broken, ref, D)
    flipped, _ = oracle.gemm("fp32", a, b, alpha=-1.0)  # planted: wrong sign
    with pytest.raises(AssertionError):
        _gate.assert_within("bf16", flipped, ref, D)
    _gate.assert_within("fp32", ref.astype(np.float32), ref, D)


def test_gate_charges_beta_c_one_rounding_only():
    """With beta != 0 the gate stays the stated |C - Cref| / (|alpha| D): the
    beta * C term may add only the one fp32 rounding of the stored result.
    Where D = 0 the result must be beta * C rounded once; where |beta C| is
    large against D, an error of a few units of it fails, although the
    beta-augmented err' would hide it."""
    M, N, K = 8, 8, 4
    a = si.uniform((M, K), 45).numpy()
    b = si.uniform((K, N), 46).numpy()
    a[3, :] = 0.0  # a zero row: D = 0 there
    c = (si.normal((M, N), 47).numpy() * 1000.0).astype(np.float32)
    alpha, beta = 0.5, 0.75
    ref, D = oracle.gemm("fp32", a, b, alpha=alpha, beta=beta, C=c)
    assert np.all(D[3] == 0)
    once = ref.astype(np.float32)  # every element rounded once
    _gate.assert_within("fp32", once, ref, D, alpha, beta, c)
    off = once.astype(np.float64).copy()
    off[3, 2] = np.nextafter(np.nextafter(once[3, 2], np.float32(np.inf)), np.float32(np.inf))  # planted: 2 ulps
    with pytest.raises(AssertionError):
        _gate.assert_within("fp32", off, ref, D, alpha, beta, c)
    off = once.astype(np.float64).copy()
    off[1, 1] += 8 * _gate.U32 * abs(beta * c[1, 1])  # planted: 8 roundings of beta*c
    assert 8 * _gate.U32 * abs(beta * c[1, 1]) > _gate.TOL["fp32"] * alpha * D[1, 1]
    assert _gate.errors_augmented(off, ref, D, alpha, beta, c)[1, 1] < _gate.TOL["fp32"]
    with pytest.raises(AssertionError):
        _gate.assert_within("fp32", off, ref, D, alpha, beta, c)


def test_fp8_gate_catches_one_missing_k_block_on_nonnegative_operands():
    """At decode depth (K = 8960, 70 blocks of 128 bytes) a missing or doubled
    K block moves a random-sign result by less than the FP8 gate, so the FP8
    parity tests also run non-negative operands, where D = |Cref| and one
    block of 128 is 1/70 of every element.  Planted in the oracle's inputs."""
    K = 8960
    a8, _ = si.to_fp8_e4m3(si.uniform((2, K), 43, lo=0.0, hi=1.0))
    b8, _ = si.to_fp8_e4m3(si.uniform((24, K), 44, lo=0.0, hi=1.0))
    ref, D = oracle.gemm("fp8", a8, b8, transB=True)
    assert np.allclose(D, ref)
    dropped = a8.copy()
    dropped[:, 128 * 37:128 * 38] = 0  # planted: one K block missing
    broken, _ = oracle.gemm("fp8", dropped, b8, transB=True)
    assert _gate.max_err(broken, ref, D) > 5 * _gate.TOL["fp8"]
    with pytest.raises(AssertionError):
        _gate.assert_within("fp8", broken, ref, D)
    _gate.assert_within("fp8", ref.astype(np.float32), ref, D)


# ------------------------------------------------------------ block-scaled (MX / NVFP4)
# The E2M1 magnitudes as the OCP Microscaling specification tabulates them.
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_values():
    got = oracle.e2m1_to_f64(np.arange(16, dtype=np.uint8))
    assert got[:8].tolist() == E2M1_VALUES
    assert np.array_equal(got[8:], -got[:8]) and np.signbit(got[8])


def test_e8m0_scales():
    got = oracle.e8m0_to_f64(np.arange(256, dtype=np.uint8))
    assert got[127] == 1.0 and got[128] == 2.0 and got[126] == 0.5
    assert got[0] == 2.0 ** -127 and got[254] == 2.0 ** 127
    assert np.isnan(got[255]) and not np.isnan(got[:255]).any()
    assert np.all(got[1:255] / got[:254] == 2.0)


def test_ue4m3_scales_are_e4m3_magnitudes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.ue4m3_to_f64(codes)
    want = np.abs(torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy())
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def _fp8_values(codes, fmt):
    """Exact values of element codes, decoded without the oracle: torch's
    float8 widening, or the E2M1 table (two codes per byte, low nibble first)."""
    if fmt == "e2m1":
        lo, hi = codes & 15, codes >> 4
        nib = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)
        mag = np.array(E2M1_VALUES)[nib & 7]
        return np.where(nib & 8, -mag, mag)
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(codes.copy()).view(dt).to(torch.float64).numpy()


def _scale_values(codes, scale_fmt):
    if scale_fmt == "e8m0":
        return np.vectorize(lambda c: Fraction(2) ** (int(c) - 127))(codes)
    return np.abs(torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy())


def _random_codes(rng, rows, K, fmt):
    if fmt == "e2m1":
        return rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    codes = rng.integers(0, 256, size=(rows, K), dtype=np.uint8)
    nan = np.isnan(_fp8_values(codes, fmt)) | np.isinf(_fp8_values(codes, fmt))
    codes[nan] = 0x38 if fmt == "e4m3" else 0x3C  # 1.0 in place of the non-finite codes
    return codes


@pytest.mark.parametrize("fmt_a,fmt_b,block,scale_fmt", [
    ("e4m3", "e4m3", 32, "e8m0"), ("e5m2", "e4m3", 32, "e8m0"), ("e4m3", "e5m2", 32, "e8m0"),
    ("e2m1", "e2m1", 32, "e8m0"), ("e2m1", "e2m1", 16, "ue4m3")])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-0.75, 0.5)])
def test_block_scaled_exact_rational(fmt_a, fmt_b, block, scale_fmt, alpha, beta):
    """Every output against a Fraction evaluation of the definition, with
    elements and scales decoded without the oracle; K ends in a partial
    block, and every block has its own scale."""
    rng = np.random.default_rng(hash((fmt_a, fmt_b, block, alpha)) % 2 ** 32)
    M, N, K = 3, 4, 2 * block + 6
    nb = -(-K // block)
    A, B = _random_codes(rng, M, K, fmt_a), _random_codes(rng, N, K, fmt_b)
    if scale_fmt == "e8m0":
        SA, SB = (rng.integers(118, 137, size=(r, nb), dtype=np.uint8) for r in (M, N))
    else:
        SA, SB = (rng.integers(0x20, 0x58, size=(r, nb), dtype=np.uint8) for r in (M, N))
    c = rng.standard_normal((M, N)).astype(np.float32)
    got, D = oracle.gemm_block_scaled(fmt_a, fmt_b, A, SA, B, SB, block=block, scale_fmt=scale_fmt,
                                      alpha=alpha, beta=beta, C=c)
    va, vb = _fp8_values(A, fmt_a), _fp8_values(B, fmt_b)
    sa, sb = _scale_values(SA, scale_fmt), _scale_values(SB, scale_fmt)
    for i in range(M):
        for j in range(N):
            terms = [Fraction(sa[i, k // block]) * Fraction(float(va[i, k])) *
                     Fraction(sb[j, k // block]) * Fraction(float(vb[j, k])) for k in range(K)]
            exact = Fraction(alpha) * sum(terms) + Fraction(beta) * Fraction(float(c[i, j]))
            d = sum(abs(t) for t in terms)
            bound = 2 * (K + 2) * 2.0 ** -53 * (abs(alpha) * float(d) + abs(beta * float(c[i, j])))
            assert abs(Fraction(float(got[i, j])) - exact) <= Fraction(bound), (i, j)
            assert abs(Fraction(float(D[i, j])) - d) <= Fraction(2 * K * 2.0 ** -53 * float(d))


@pytest.mark.parametrize("mode,fa,fb", [("fp8", "e4m3", "e4m3"), ("fp8_e5m2", "e5m2", "e5m2"),
                                        ("fp8_e4m3_e5m2", "e4m3", "e5m2")])
def test_block_scaled_unit_scales_is_the_plain_product(mode, fa, fb):
    """Scales of 1 (E8M0 code 127) reduce MXFP8 to the per-tensor FP8
    product, which has its own pins."""
    rng = np.random.default_rng(7)
    M, N, K = 9, 11, 100
    A, B = _random_codes(rng, M, K, fa), _random_codes(rng, N, K, fb)
    ones_a = np.full((M, 4), 127, dtype=np.uint8)
    ones_b = np.full((N, 4), 127, dtype=np.uint8)
    got, D = oracle.gemm_block_scaled(fa, fb, A, ones_a, B, ones_b, block=32, scale_fmt="e8m0", alpha=0.5)
    ref, Dref = oracle.gemm(mode, A, B, transB=True, alpha=0.5)
    assert np.array_equal(got, ref) and np.array_equal(D, Dref)


def test_block_scale_applies_to_its_own_block_only():
    """A scale of 8 on block 1 of one row of A multiplies that block's
    share of the row's products and nothing else (a wrong block index, or
    a scale taken from the wrong row, fails)."""
    rng = np.random.default_rng(8)
    M, N, K, bs = 4, 5, 90, 32  # blocks 0..31, 32..63, 64..89
    A, B = _random_codes(rng, M, K, "e4m3"), _random_codes(rng, N, K, "e4m3")
    SA = np.full((M, 3), 127, dtype=np.uint8)
    SB = np.full((N, 3), 127, dtype=np.uint8)
    SA[2, 1] = 130  # 2^3
    got, D = oracle.gemm_block_scaled("e4m3", "e4m3", A, SA, B, SB, block=bs, scale_fmt="e8m0")
    inside = np.zeros_like(A)
    inside[:, 32:64] = A[:, 32:64]
    outside = A.copy()
    outside[:, 32:64] = 0
    p_in, _ = oracle.gemm("fp8", inside, B, transB=True)
    p_out, _ = oracle.gemm("fp8", outside, B, transB=True)
    want = p_in + p_out
    want[2] = 8.0 * p_in[2] + p_out[2]
    assert np.allclose(got, want, rtol=0, atol=1e-12 * D.max())
    # NVFP4-sized blocks: the same scale codes now cover 16 elements each
    SA16 = np.full((M, 6), 0x38, dtype=np.uint8)  # UE4M3 1.0
    SB16 = np.full((N, 6), 0x38, dtype=np.uint8)
    SA16[1, 5] = 0x40  # 2.0 on elements 80..89 of row 1
    A4 = _random_codes(rng, M, K, "e2m1")
    B4 = _random_codes(rng, N, K, "e2m1")
    got4, D4 = oracle.gemm_block_scaled("e2m1", "e2m1", A4, SA16, B4, SB16, block=16, scale_fmt="ue4m3")
    va, vb = _fp8_values(A4, "e2m1"), _fp8_values(B4, "e2m1")
    want4 = va @ vb.T
    want4[1] += (va[1, 80:] @ vb[:, 80:].T)  # doubled: the scale of 2 adds one more copy
    assert np.allclose(got4, want4, rtol=0, atol=1e-12 * max(D4.max(), 1.0))


def test_e2m1_packing_low_nibble_first():
    """Byte t holds elements 2t (low four bits) and 2t + 1 (high four bits)."""
    K = 8
    B = np.full((1, K // 2), 0x22, dtype=np.uint8)  # every element 1.0
    SB = np.full((1, 1), 127, dtype=np.uint8)
    SA = np.full((1, 1), 127, dtype=np.uint8)
    for k in range(K):
        A = np.zeros((1, K // 2), dtype=np.uint8)
        A[0, k // 2] = (7 << 4) if k % 2 else 5  # 6.0 high, or 3.0 low
        got, _ = oracle.gemm_block_scaled("e2m1", "e2m1", A, SA, B, SB, block=32, scale_fmt="e8m0")
        assert got[0, 0] == (6.0 if k % 2 else 3.0)


# ------------------------------------------------------------ fused epilogue
# Standard normal distribution function Phi at 1, 2 and -1 as tabulated
# (Abramowitz and Stegun, table 26.1, to 10 digits).  GELU(x) = x * Phi(x).
PHI_TABLE = {1.0: 0.8413447461, 2.0: 0.9772498681, -1.0: 0.1586552539}


def test_gelu_matches_the_tabulated_normal_distribution():
    """Pins GELU to x * Phi(x) with the exact Phi: the tanh approximation
    differs by 1.5e-4 at x = 1, a sign or factor error by far more."""
    for x, phi in PHI_TABLE.items():
        assert abs(oracle.gelu(x) - x * phi) < 1e-9, x
    assert oracle.gelu(0.0) == 0.0


def test_gelu_odd_part_is_the_identity():
    """GELU(x) - GELU(-x) = x (Phi(x) + Phi(-x) = 1), at any x."""
    for x in (0.1, 0.5, 1.7, 3.0, 6.0):
        assert abs(oracle.gelu(x) - oracle.gelu(-x) - x) < 1e-12 * max(1.0, x)


def test_dgelu_is_the_derivative_of_gelu():
    """GELU' against a central difference of GELU (brute force), and its
    limits: 1/2 at 0, 1 far right, 0 far left."""
    h = 1e-5
    for x in (-3.0, -1.2, -0.3, 0.0, 0.4, 1.0, 2.5):
        fd = (oracle.gelu(x + h) - oracle.gelu(x - h)) / (2 * h)
        assert abs(fd - oracle.dgelu(x)) < 1e-8, x
    assert oracle.dgelu(0.0) == 0.5
    assert abs(oracle.dgelu(12.0) - 1.0) < 1e-12 and abs(oracle.dgelu(-12.0)) < 1e-12


def test_epilogue_variants_elementwise():
    """none adds the bias to every row; gelu applies GELU after the bias;
    dgelu multiplies by GELU'(Z) and takes no bias."""
    Y = np.array([[0.5, -1.0, 2.0], [0.0, 1.0, -2.0]])
    bias = np.array([0.5, 0.0, -1.0], dtype=np.float32)
    Z = np.array([[1.0, -1.0, 0.0], [2.0, 0.0, -3.0]], dtype=np.float32)
    assert np.array_equal(oracle.epilogue("none", Y, bias), Y + bias.astype(np.float64))
    assert np.array_equal(oracle.epilogue("none", Y), Y)
    g = oracle.epilogue("gelu", Y, bias)
    assert abs(g[0, 0] - 1.0 * PHI_TABLE[1.0]) < 1e-9 and abs(g[0, 1] + PHI_TABLE[-1.0]) < 1e-9
    assert abs(g[0, 2] - PHI_TABLE[1.0]) < 1e-9 and abs(g[1, 1] - PHI_TABLE[1.0]) < 1e-9
    d = oracle.epilogue("dgelu", Y, Z=Z)
    for i in range(2):
        for j in range(3):
            assert d[i, j] == Y[i, j] * oracle.dgelu(float(Z[i, j]))
    with pytest.raises(ValueError):
        oracle.epilogue("dgelu", Y, bias, Z)


# ------------------------------------------------------------ attention (the fused-attention row)
def _bf(x):
    """bfloat16 bit patterns of float values (exact when they are bf16 values)."""
    return si.bf16_bits(si.to_bf16(torch.from_numpy(np.asarray(x, dtype=np.float32))))


def test_attention_zero_queries_average_the_visible_values():
    """q = 0 gives equal scores, so every query averages the values it sees:
    rows 0..i when causal, all rows otherwise."""
    rng = np.random.default_rng(71)
    P, T, D = 3, 9, 4
    q = np.zeros((P, T, D))
    k = rng.integers(-4, 5, size=(P, T, D)).astype(np.float32)
    v = rng.integers(-4, 5, size=(P, T, D)).astype(np.float64)
    O, W = oracle.attention(_bf(q), _bf(k), _bf(v), causal=True)
    for i in range(T):
        assert np.allclose(O[:, i], v[:, :i + 1].mean(axis=1), rtol=0, atol=1e-15)
        assert np.allclose(W[:, i], np.abs(v[:, :i + 1]).mean(axis=1), rtol=0, atol=1e-15)
    O, _ = oracle.attention(_bf(q), _bf(k), _bf(v), causal=False)
    assert np.allclose(O, np.repeat(v.mean(axis=1, keepdims=True), T, axis=1), rtol=0, atol=1e-15)


def test_attention_two_keys_closed_form():
    """T = 2, Dh = 1, scale 1: row 0 sees only key 0; row 1 weighs the keys
    e^1 : e^0, so O = (2e - 1) / (e + 1) and W = (2e + 1) / (e + 1)."""
    q = np.array([[[1.0], [1.0]]])
    k = np.array([[[1.0], [0.0]]])
    v = np.array([[[2.0], [-1.0]]])
    O, W = oracle.attention(_bf(q), _bf(k), _bf(v), causal=True, scale=1.0)
    e = math.e
    assert O[0, 0, 0] == 2.0 and W[0, 0, 0] == 2.0
    assert abs(O[0, 1, 0] - (2 * e - 1) / (e + 1)) < 1e-15
    assert abs(W[0, 1, 0] - (2 * e + 1) / (e + 1)) < 1e-15
    O, _ = oracle.attention(_bf(q), _bf(k), _bf(v), causal=False, scale=1.0)
    assert abs(O[0, 0, 0] - (2 * e - 1) / (e + 1)) < 1e-15  # non-causal row 0 sees both keys


def test_attention_constant_values_and_a_dominant_key():
    """Weights sum to one (constant values come back unchanged), and a key
    whose score exceeds the others by 64 takes all the weight for the rows
    that see it."""
    rng = np.random.default_rng(72)
    P, T, D = 2, 12, 2
    q = rng.normal(size=(P, T, D)).astype(np.float32)
    k = rng.normal(size=(P, T, D)).astype(np.float32)
    O, W = oracle.attention(_bf(q), _bf(k), _bf(np.full((P, T, D), 3.0)), causal=True)
    assert np.allclose(O, 3.0, rtol=0, atol=1e-14) and np.allclose(W, 3.0, rtol=0, atol=1e-14)
    q = np.zeros((P, T, D))
    q[..., 0] = 8.0
    k = np.zeros((P, T, D))
    k[:, 5, 0] = 8.0
    v = rng.integers(-4, 5, size=(P, T, D)).astype(np.float64)
    O, _ = oracle.attention(_bf(q), _bf(k), _bf(v), causal=True, scale=1.0)
    for i in range(T):
        want = v[:, 5] if i >= 5 else v[:, :i + 1].mean(axis=1)
        assert np.allclose(O[:, i], want, rtol=0, atol=1e-20 + (1e-25 if i >= 5 else 1e-15)), i


def test_attention_causal_rows_ignore_later_keys_and_values():
    rng = np.random.default_rng(73)
    P, T, D = 2, 16, 8
    q, k, v = (rng.normal(size=(P, T, D)).astype(np.float32) for _ in range(3))
    O1, _ = oracle.attention(_bf(q), _bf(k), _bf(v), causal=True)
    k2, v2 = k.copy(), v.copy()
    k2[:, 10:] = rng.normal(size=(P, T - 10, D))
    v2[:, 10:] = rng.normal(size=(P, T - 10, D))
    O2, _ = oracle.attention(_bf(q), _bf(k2), _bf(v2), causal=True)
    assert np.array_equal(O1[:, :10], O2[:, :10])
    assert not np.allclose(O1[:, 10:], O2[:, 10:])
    O3, _ = oracle.attention(_bf(q), _bf(k2), _bf(v2), causal=False)
    assert not np.allclose(O3[:, :10], O2[:, :10])  # without the mask the early rows see the later keys


def test_attention_score_shift_invariance_and_error_scale_bounds():
    """Adding the same amount to every score of a row changes nothing (an
    extra dimension with q = 1 and the same k for every key); and the error
    scale W satisfies |O| <= W <= max |v|."""
    rng = np.random.default_rng(74)
    P, T, D = 2, 20, 6
    q, k, v = (rng.integers(-3, 4, size=(P, T, D)).astype(np.float32) for _ in range(3))
    O1, W1 = oracle.attention(_bf(q), _bf(k), _bf(v), causal=True, scale=0.25)
    q2 = np.concatenate([q, np.ones((P, T, 1))], axis=2)
    k2 = np.concatenate([k, np.full((P, T, 1), 5.0)], axis=2)
    v2 = np.concatenate([v, np.zeros((P, T, 1))], axis=2)
    O2, _ = oracle.attention(_bf(q2), _bf(k2), _bf(v2), causal=True, scale=0.25)
    assert np.allclose(O2[..., :D], O1, rtol=0, atol=1e-13)
    assert np.all(np.abs(O1) <= W1 * (1 + 1e-15))
    assert np.all(W1 <= float(np.abs(v).max()) * (1 + 1e-14))
