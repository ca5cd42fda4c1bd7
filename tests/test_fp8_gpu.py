"""Parity of the FP8 (E4M3) mode with the CPU oracle, through the C ABI.

The FP8 modes run the tensor-core kernels with kind::f8f6f4 on K-major
operands (A stored M x K, B stored N x K; an MN-major operand is transposed
first): the decode-shaped kernel for M <= 16 and the persistent tile kernel
(every tile width, CTA pairs, K splits) above.
Inputs are quantised per tensor the way FP8 inference stores them (each
tensor divided by max|t| / 440, rounded to E4M3 by torch on the CPU) and the
two scales come back through alpha.  The oracle decodes the same codes
exactly and accumulates in fp64.  Gate: 2e-3 of |alpha| * sum|a||b|
(tests/_gate.py); non-negative operands at decode depth catch a missing or
doubled K block, small integers must come out bit-exact.
"""
import numpy as np
import pytest
import torch

import dense_gemm_transformer_gb300 as dg
import oracle
import seeded_inputs as si
from tests import _gate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    dg.load(build_if_missing=True)
    handle = dg.Gemm()
    yield handle
    handle.close()


def _defaults(h):
    h.set_option("family", "auto")
    h.set_option("split_k", 0)
    h.set_option("tile_n", 0)
    h.set_option("pair", 0)


@pytest.fixture(autouse=True)
def _reset(h):
    _defaults(h)
    yield
    _defaults(h)


def _draw(shape, seed, dist, std=1.0):
    if dist == "int":
        return si.integers(shape, seed)
    if dist == "pos":
        return si.uniform(shape, seed, lo=0.0, hi=1.0)
    return si.normal(shape, seed, std=std)


FORMATS = {"fp8": ("e4m3", "e4m3"), "fp8_e5m2": ("e5m2", "e5m2"), "fp8_e4m3_e5m2": ("e4m3", "e5m2"),
           "fp8_e5m2_e4m3": ("e5m2", "e4m3")}
OTHER_MODES = ["fp8_e5m2", "fp8_e4m3_e5m2", "fp8_e5m2_e4m3"]
_AMAX = {"e4m3": 440.0, "e5m2": 0.98 * si.FP8_E5M2_MAX}
_TORCH = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _operands(M, N, K, seed, dist="normal", mode="fp8"):
    """8-bit codes of the activations (M x K) and weights (N x K), each in
    its mode's format, and the alpha that undoes their per-tensor scales
    (1 for integers)."""
    fa, fb = FORMATS[mode]
    a8, sa = si.to_fp8(_draw((M, K), seed, dist), fa, 0.0 if dist == "int" else _AMAX[fa])
    w8, sw = si.to_fp8(_draw((N, K), seed + 1, dist, std=0.02), fb, 0.0 if dist == "int" else _AMAX[fb])
    return a8, w8, sa * sw


def _device(codes, as_fp8=False, fmt="e4m3"):
    t = torch.from_numpy(codes).cuda()
    return t.view(_TORCH[fmt]) if as_fp8 else t


def _run_and_check(h, M, N, K, seed, dist="normal", beta=0.0, exact=False, as_fp8=False, cols=None, rows=None,
                   family="skinny", mode="fp8"):
    a8, w8, alpha = _operands(M, N, K, seed, dist, mode)
    fa, fb = FORMATS[mode]
    cin = si.normal((M, N), seed + 2).numpy() if beta != 0.0 else None
    C = torch.from_numpy(cin).cuda() if cin is not None else torch.full((M, N), float("nan"), device="cuda")
    h.run(_device(a8, as_fp8, fa), _device(w8, as_fp8, fb), C, mode=mode, transB=True, alpha=alpha, beta=beta)
    assert h.check_device() == 0
    got = C.cpu().numpy()
    assert h.plan()["family"] == family
    for r0, r1 in rows or [(0, M)]:
        for c0, c1 in cols or [(0, N)]:
            cpart = None if cin is None else np.ascontiguousarray(cin[:, c0:c1])
            ref, D = oracle.gemm(mode, a8, w8[c0:c1], transB=True, alpha=alpha, beta=beta, C=cpart,
                                 rows=(r0, r1))
            part = got[r0:r1, c0:c1]
            if exact:
                assert np.array_equal(part.astype(np.float64), ref), (M, N, K, r0, c0)
            else:
                _gate.assert_within("fp8", part, ref, D, alpha=alpha, beta=beta,
                                    Cin=None if cpart is None else cpart[r0:r1],
                                    what=f"{mode} M={M} N={N} K={K} rows {r0}:{r1} cols {c0}:{c1}")
    return got


# ------------------------------------------------------------ ragged shapes
@pytest.mark.parametrize("M,N,K", [(1, 1000, 768), (7, 300, 128), (16, 129, 2048), (3, 65, 40),
                                   (16, 384, 96), (5, 1, 256)])
def test_fp8_ragged(h, M, N, K):
    _run_and_check(h, M, N, K, seed=71)
    _run_and_check(h, M, N, K, seed=72, beta=1.0)


def test_fp8_takes_float8_tensors_and_uint8_codes_alike(h):
    g1 = _run_and_check(h, 4, 300, 512, seed=73)
    g2 = _run_and_check(h, 4, 300, 512, seed=73, as_fp8=True)
    assert np.array_equal(g1, g2)


@pytest.mark.parametrize("K", [1000, 1512])
def test_fp8_row_pitch_not_a_multiple_of_16_bytes(h, K):
    """K = 1000 or 1512 bytes per row: the TMA unit cannot read the rows in
    place, so both operands are re-packed first (and K ends inside a block)."""
    _run_and_check(h, 9, 500, K, seed=74)
    assert h.plan()["packed"] == 3


def test_fp8_unaligned_base_pointer(h):
    M, N, K = 4, 200, 256
    a8, w8, alpha = _operands(M, N, K, 75)
    buf = torch.zeros(M * K + 16, dtype=torch.uint8, device="cuda")
    A = buf[1:1 + M * K].view(M, K)  # base one byte past a 16-byte boundary
    A.copy_(torch.from_numpy(a8).cuda())
    C = torch.full((M, N), float("nan"), device="cuda")
    h.run(A, torch.from_numpy(w8).cuda(), C, mode="fp8", transB=True, alpha=alpha)
    assert h.check_device() == 0
    assert h.plan()["packed"] == 1  # A (the activations) re-packed, the weights read in place
    ref, D = oracle.gemm("fp8", a8, w8, transB=True, alpha=alpha)
    _gate.assert_within("fp8", C.cpu().numpy(), ref, D, alpha=alpha)


# ------------------------------------------------------------ K slices in one cluster
@pytest.mark.parametrize("cs", [1, 2, 3, 8, 12, 16])
def test_fp8_cluster_k_slices(h, cs):
    h.set_option("family", "skinny")
    h.set_option("split_k", cs)
    M, N, K = 5, 300, 46 * 128 + 16  # 47 K blocks, the last one ragged: every cs gives cs slices
    _run_and_check(h, M, N, K, seed=76)
    plan = h.plan()
    assert plan["split_k"] == cs and plan["cluster"] == cs and plan["grid"] == 3 * cs
    _run_and_check(h, M, N, K, seed=77, beta=1.0)


@pytest.mark.parametrize("cs", [1, 5, 16])
def test_fp8_integers_bit_exact(h, cs):
    # integers in [-4, 4] are E4M3 values.  K = 256 keeps every partial sum
    # below 2^12, exact in any accumulator the gate allows; at K = 1792 the
    # sums of these random signs stay far below 2^14 as well
    h.set_option("split_k", cs)
    _run_and_check(h, 16, 260, 256, seed=78, dist="int", exact=True)
    _run_and_check(h, 16, 260, 256 * 7, seed=79, dist="int", exact=True)


# ------------------------------------------------------------ the decode shapes
def _column_ranges(N, tile=128, width=4):
    picks = sorted({0, tile - 2, N // 2 - 1, N - width})
    return [(c, min(c + width, N)) for c in picks if 0 <= c < N]


@pytest.mark.parametrize("M", si.SKINNY_M)
@pytest.mark.parametrize("w", range(len(si.SKINNY_WEIGHTS)))
def test_fp8_decode_shapes_sampled(h, M, w):
    """The decode shapes at full size (the benchmark's launch configuration),
    checked on sampled columns around tile edges."""
    K, N = si.SKINNY_WEIGHTS[w]
    _run_and_check(h, M, N, K, seed=si.seed_for(4, w, 5), cols=_column_ranges(N))
    plan = h.plan()
    tiles = -(-N // 128)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # fewer than two waves of weight tiles: one cluster of K slices per tile;
    # more: the persistent kernel, one CTA per SM, no split
    assert plan["grid"] == (tiles * plan["split_k"] if tiles < 2 * sms else sms)


@pytest.mark.parametrize("w", range(len(si.SKINNY_WEIGHTS)))
def test_fp8_nonnegative_operands_catch_a_missing_k_block(h, w):
    """With non-negative operands D equals |Cref|, and one K block of 128 is
    at least 1/70 of every element at these depths, far above the gate."""
    K, N = si.SKINNY_WEIGHTS[w]
    _run_and_check(h, 16, N, K, seed=si.seed_for(4, w, 7), dist="pos", cols=_column_ranges(N))


# ------------------------------------------------------------ MN-major operands
@pytest.mark.parametrize("mode", ["fp8", "fp8_e4m3_e5m2"])
@pytest.mark.parametrize("tA,tB", [(False, False), (True, False), (True, True), (False, True)])
@pytest.mark.parametrize("M,N,K", [(300, 260, 1024), (4, 1000, 768)])
def test_fp8_any_layout(h, mode, tA, tB, M, N, K):
    """An operand stored MN-major (A as K x M, B as K x N) is transposed into
    the workspace first; the kernels then read K-major operands."""
    a8, w8, alpha = _operands(M, N, K, 107, mode=mode)
    A = np.ascontiguousarray(a8.T) if tA else a8      # op(A) = A^T when stored K x M
    B = w8 if tB else np.ascontiguousarray(w8.T)      # op(B) = B^T when stored N x K
    C = torch.full((M, N), float("nan"), device="cuda")
    h.run(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), C, mode=mode, transA=tA, transB=tB, alpha=alpha)
    assert h.check_device() == 0
    plan = h.plan()
    swapped = plan["family"] == "skinny"
    assert swapped == (M <= 16 and not tA)
    # packed bit 0: A, bit 1: B (re-packed or transposed)
    assert bool(plan["packed"] & 1) == tA
    assert bool(plan["packed"] & 2) == (not tB)
    ref, D = oracle.gemm(mode, A, B, transA=tA, transB=tB, alpha=alpha)
    _gate.assert_within("fp8", C.cpu().numpy(), ref, D, alpha=alpha, what=f"{mode} tA={tA} tB={tB}")


def test_fp8_unsupported_forms(h):
    A = torch.zeros((4, 64), dtype=torch.uint8, device="cuda")
    Wnk = torch.zeros((32, 64), dtype=torch.uint8, device="cuda")
    C = torch.zeros((4, 32), device="cuda")
    h.set_option("family", "simt")
    with pytest.raises(dg.GemmError) as e:
        h.run(A, Wnk, C, mode="fp8", transB=True)
    assert e.value.status == 2
    h.set_option("family", "auto")
    with pytest.raises(dg.GemmError) as e:  # no allocation-free FP8 entry
        dg.run_small_m_noalloc(A, Wnk, C, mode="fp8", transB=True)
    assert e.value.status == 2
    assert h.check_device() == 0


def test_fp8_epilogue_bias_gelu(h):
    """The fused epilogue runs after the FP8 product like after any other."""
    M, N, K = 16, 8960, 1536
    a8, w8, alpha = _operands(M, N, K, 80)
    bias = si.normal((N,), 81).numpy()
    C = torch.full((M, N), float("nan"), device="cuda")
    h.run(torch.from_numpy(a8).cuda(), torch.from_numpy(w8).cuda(), C, mode="fp8", transB=True, alpha=alpha,
          act="gelu", bias=torch.from_numpy(bias).cuda())
    assert h.check_device() == 0
    got = C.cpu().numpy()
    for c0, c1 in _column_ranges(N):
        Y, D = oracle.gemm("fp8", a8, w8[c0:c1], transB=True, alpha=alpha)
        ref = oracle.epilogue("gelu", Y, bias[c0:c1])
        # GELU' is at most 1.13: the product's bound carries through, plus
        # fp32 rounding of the bias sum and of GELU itself
        tol = 1.13 * _gate.TOL["fp8"] * abs(alpha) * D + 1e-6 * (np.abs(ref) + np.abs(bias[c0:c1]) + 1e-3)
        assert np.all(np.abs(got[:, c0:c1] - ref) <= tol), (c0, np.max(np.abs(got[:, c0:c1] - ref) - tol))


# ------------------------------------------------------------ M > 16: the persistent tile kernel
@pytest.mark.parametrize("tile_n,pair", [(128, 1), (128, 0), (192, 1), (192, 0), (224, 1), (224, 0), (256, 1),
                                         (256, 0)])
def test_fp8_tiles_and_pairs(h, tile_n, pair):
    """Every tile width, one CTA per tile (pair option 1) and CTA pairs
    issuing one 256-row MMA (option 0, from 192 columns); ragged M, N and K."""
    h.set_option("tile_n", tile_n)
    h.set_option("pair", pair)
    M, N, K = 700, 650, 1008  # K: 8 blocks of 128 bytes, the last one ragged
    _run_and_check(h, M, N, K, seed=90, family="tc", rows=_cases_rows(M))
    plan = h.plan()
    paired = pair == 0 and tile_n >= 192
    assert plan["tile_n"] == tile_n
    assert plan["cluster"] == (2 if paired else 1)
    assert plan["pair_mma"] == (1 if paired else 0)
    _run_and_check(h, M, N, K, seed=91, beta=1.0, family="tc", rows=_cases_rows(M))


def _cases_rows(M, tile=128, width=2):
    picks = sorted({0, tile - 1, 2 * tile - 1, M // 2, M - (M % tile or tile) - 1, M - width})
    return [(r, min(r + width, M)) for r in picks if 0 <= r < M]


@pytest.mark.parametrize("M,N,K", [(17, 300, 512), (100, 129, 2048), (300, 260, 1000), (1000, 1000, 768),
                                   (2304, 2304, 1024)])
def test_fp8_planner_shapes(h, M, N, K):
    """The planner's own choices (tile width, pairs, cut final wave)."""
    _run_and_check(h, M, N, K, seed=92, family="tc", rows=_cases_rows(M))
    _run_and_check(h, M, N, K, seed=93, beta=1.0, family="tc", rows=_cases_rows(M))


@pytest.mark.parametrize("splits", [2, 3, 7])
def test_fp8_split_k(h, splits):
    h.set_option("split_k", splits)
    M, N, K = 300, 260, 26 * 128 + 64  # 27 K blocks: each count gives that many slices
    _run_and_check(h, M, N, K, seed=94, family="tc", rows=_cases_rows(M))
    assert h.plan()["split_k"] == splits
    _run_and_check(h, M, N, K, seed=95, beta=1.0, family="tc", rows=_cases_rows(M))


@pytest.mark.parametrize("tile_n,pair", [(128, 1), (192, 0), (224, 0), (256, 0)])
def test_fp8_tiles_integers_bit_exact(h, tile_n, pair):
    h.set_option("tile_n", tile_n)
    h.set_option("pair", pair)
    _run_and_check(h, 512, 512, 1024, seed=96, dist="int", exact=True, family="tc")


def test_fp8_nonnegative_deep_k(h):
    """Non-negative operands at K = 8192 (64 K blocks): a missing or doubled
    block would be 1/64 of every element."""
    _run_and_check(h, 512, 768, 8192, seed=97, dist="pos", family="tc", rows=_cases_rows(512))


@pytest.mark.parametrize("M,N,K", [(8192, 8192, 8192), (8192, 28672, 8192)])
def test_fp8_large_sampled(h, M, N, K):
    """The large shapes in FP8 (A stored M x K, B stored N x K), checked on
    rows at tile edges and on columns around tile edges."""
    _run_and_check(h, M, N, K, seed=98, family="tc", rows=[(0, 1), (4095, 4097), (M - 1, M)],
                   cols=_column_ranges(N, tile=256))


# ------------------------------------------------------------ E5M2 and the mixed pairs
@pytest.mark.parametrize("mode", OTHER_MODES)
@pytest.mark.parametrize("M,N,K", [(1, 1000, 768), (16, 129, 2048), (3, 65, 40)])
def test_fp8_formats_small_m(h, mode, M, N, K):
    """The small-M kernel exchanges the operands (C^T = B^T A^T), so the
    formats must follow them: a mixed pair catches a missed exchange."""
    _run_and_check(h, M, N, K, seed=101, mode=mode)
    _run_and_check(h, M, N, K, seed=102, beta=1.0, mode=mode, as_fp8=True)


@pytest.mark.parametrize("mode", OTHER_MODES)
@pytest.mark.parametrize("tile_n,pair", [(128, 1), (224, 0), (256, 0)])
def test_fp8_formats_tiles(h, mode, tile_n, pair):
    h.set_option("tile_n", tile_n)
    h.set_option("pair", pair)
    _run_and_check(h, 700, 650, 1008, seed=103, family="tc", rows=_cases_rows(700), mode=mode)


@pytest.mark.parametrize("mode", OTHER_MODES)
def test_fp8_formats_integers_bit_exact(h, mode):
    h.set_option("split_k", 5)
    _run_and_check(h, 16, 260, 1792, seed=104, dist="int", exact=True, mode=mode)
    h.set_option("split_k", 0)
    _run_and_check(h, 512, 512, 1024, seed=105, dist="int", exact=True, family="tc", mode=mode)


@pytest.mark.parametrize("mode", OTHER_MODES)
@pytest.mark.parametrize("w", [0, 2])
def test_fp8_formats_decode_shapes(h, mode, w):
    """1536 x 8960 (cluster kernel) and 1536 x 151936 (the persistent
    kernel's swapped form), M = 16, sampled columns."""
    K, N = si.SKINNY_WEIGHTS[w]
    _run_and_check(h, 16, N, K, seed=si.seed_for(4, w, 9), cols=_column_ranges(N), mode=mode)


def test_fp8_formats_large_sampled(h):
    _run_and_check(h, 4096, 4096, 4096, seed=106, family="tc", rows=[(0, 2), (2047, 2049), (4094, 4096)],
                   cols=_column_ranges(4096, tile=256), mode="fp8_e5m2_e4m3")
