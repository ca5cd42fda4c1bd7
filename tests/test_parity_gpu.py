"""Parity of the library's kernels with the CPU oracle, through the C ABI.

Every mode and transpose combination, ragged shapes that span several tiles
with a partial last tile, forced split-K and tile widths, unaligned leading
dimensions, alpha/beta, the degenerate sizes, bit-exact small-integer inputs,
and guard bands around C.  Tolerances (tests/_gate.py): 1e-6 FP32, 2e-3 TF32,
8e-3 BF16 of |alpha| * sum|a||b| (+ |beta c|).
"""
import numpy as np
import pytest
import torch

import dense_gemm_transformer_gb300 as dg
import oracle
import seeded_inputs as si
from tests import _cases, _gate

pytestmark = pytest.mark.gpu

MODES = ["fp32", "tf32", "bf16"]
TRANS = [(False, False), (False, True), (True, False), (True, True)]


@pytest.fixture(scope="module")
def h():
    dg.load(build_if_missing=True)
    handle = dg.Gemm()
    yield handle
    handle.close()


@pytest.fixture(autouse=True)
def _reset(h):
    h.set_option("family", "auto")
    h.set_option("split_k", 0)
    h.set_option("tile_n", 0)
    h.set_option("pretranspose", 0)
    h.set_option("pair", 0)
    h.set_option("sk_fixup", 0)
    yield


# ------------------------------------------------------------ the 256^3 case
@pytest.mark.parametrize("mode", MODES)
def test_square256_uniform(h, mode):
    _cases.run_and_check(h, mode, 256, 256, 256, seed=si.seed_for(0, 0, 0))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("tA,tB", TRANS)
def test_square256_integers_bit_exact(h, mode, tA, tB):
    _cases.run_and_check(h, mode, 256, 256, 256, tA, tB, seed=si.seed_for(0, 1, 0), dist="int", exact=True)


@pytest.mark.parametrize("mode", MODES)
def test_integers_bit_exact_deep_k(h, mode):
    # K = 1024 integers in [-4, 4]: every partial sum is an integer below 2^24.
    _cases.run_and_check(h, mode, 300, 200, 1024, seed=7, dist="int", exact=True)
    h.set_option("split_k", 3)
    _cases.run_and_check(h, mode, 300, 200, 1024, seed=8, dist="int", exact=True)


# ------------------------------------------------------------ shapes and layouts
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("tA,tB", TRANS)
def test_ragged_all_layouts(h, mode, tA, tB):
    _cases.run_and_check(h, mode, 300, 264, 200, tA, tB, seed=11, dist="normal")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 9, 5), (65, 65, 65), (127, 129, 33), (129, 127, 130),
                                   (1, 300, 64), (300, 1, 64), (33, 520, 16), (520, 33, 17)])
def test_edge_shapes(h, mode, M, N, K):
    _cases.run_and_check(h, mode, M, N, K, False, False, seed=13, dist="normal")
    _cases.run_and_check(h, mode, M, N, K, True, True, seed=14, dist="normal")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("alpha,beta", [(0.5, 1.0), (-1.5, 0.25), (1.0, -1.0)])
def test_alpha_beta(h, mode, alpha, beta):
    _cases.run_and_check(h, mode, 260, 300, 96, alpha=alpha, beta=beta, seed=17, dist="normal")


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("tile_n", [128, 192, 224, 256])
@pytest.mark.parametrize("tA,tB", TRANS)
def test_tc_tile_widths(h, mode, tile_n, tA, tB):
    """Every tile width in every layout; 224 columns (3.5 chunks of 128
    bytes) cannot take an N-contiguous BF16 B and is refused."""
    h.set_option("tile_n", tile_n)
    if mode == "bf16" and tile_n == 224 and not tB:
        ops, _ = _cases.make(mode, 384, 520, 160, tA, tB)
        C = torch.zeros((384, 520), device="cuda")
        with pytest.raises(dg.GemmError) as e:
            h.run(ops.A, ops.B, C, mode=mode, transA=tA, transB=tB)
        assert e.value.status == 2  # GEMM_ERR_NOT_SUPPORTED
        assert torch.count_nonzero(C).item() == 0
        return
    _cases.run_and_check(h, mode, 384, 520, 160, tA, tB, seed=19, dist="normal")
    assert h.plan()["family"] == "tc" and h.plan()["tile_n"] == tile_n
    _cases.run_and_check(h, mode, 384, 520, 160, tA, tB, alpha=2.0, beta=0.5, seed=20, dist="normal")


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("tA,tB", TRANS)
@pytest.mark.parametrize("M,N,K", [(640, 600, 200), (300, 260, 1000), (1100, 300, 64)])
@pytest.mark.parametrize("tile_n", [192, 224, 256])
def test_tc_paired_ctas(h, mode, pair, tA, tB, M, N, K, tile_n):
    """Tiles of 192-256 columns with and without two-CTA clusters: pairs
    issue one MMA of 256 rows over both CTAs' shared memory and TMEM
    (tcgen05 cta_group::2; option 0, the planner's choice), each CTA
    staging its own 128 rows of A and one half of the B tile (96, 112 or 128
    rows).  Odd tile-row counts leave the second CTA of the last pair with no
    rows of C.  An N-contiguous BF16 B pairs only when its tile is an even
    number of 128-byte chunks (256), and takes no 224-column tile."""
    b_mn = mode == "bf16" and not tB
    if b_mn and tile_n == 224:
        pytest.skip("224-column tiles need a K-major B in BF16 (covered by test_tc_tile_widths)")
    h.set_option("tile_n", tile_n)
    h.set_option("pair", pair)
    _cases.run_and_check(h, mode, M, N, K, tA, tB, alpha=0.5, beta=-1.0, seed=77, dist="normal")
    paired = pair == 0 and not (b_mn and tile_n == 192)
    plan = h.plan()
    assert plan["cluster"] == (2 if paired else 1) and plan["tile_n"] == tile_n
    assert plan["pair_mma"] == (1 if paired else 0)
    _cases.run_and_check(h, mode, M, N, min(K, 1024), tA, tB, seed=78, dist="int", exact=True)
    h.set_option("split_k", 3)
    _cases.run_and_check(h, mode, M, N, K, tA, tB, seed=79, dist="normal")


@pytest.mark.parametrize("mode,M,N,K,tile_n,pair", [("bf16", 4096, 4096, 4096, 256, 0),
                                                      ("tf32", 2304, 2304, 1024, 0, 0),
                                                      ("tf32", 2304, 2304, 1024, 256, 0),
                                                      ("tf32", 2200, 2100, 1000, 0, 0)])
@pytest.mark.parametrize("tB", [False, True])
def test_tc_tail_rows_cut_into_k_slices(h, mode, M, N, K, tile_n, pair, tB):
    """Whole tiles for the leading rows of tile pairs, the last rows cut into
    K slices whose partial sums the reduce kernel adds into C: checked on rows
    of both regions, across their boundary and at the ragged bottom edge."""
    h.set_option("tile_n", tile_n)
    h.set_option("pair", pair)
    probe = torch.zeros((M, N), device="cuda")
    ops, _ = _cases.make(mode, M, N, K, False, tB)
    h.run(ops.A, ops.B, probe, mode=mode, transB=tB)
    plan = h.plan()
    assert plan["schedule"] == "tail_split" and plan["split_k"] > 1 and plan["cluster"] == 2, plan
    rows = [(0, 2), (M // 2, M // 2 + 1), (M - 3, M)]
    # the boundary lies on a pair-row (256 C rows) edge somewhere in the last quarter
    for b in range(256 * ((M // 256) // 2), M, 256):
        rows.append((b - 1, b + 1))
    rows = sorted(set((max(0, r0), min(M, r1)) for r0, r1 in rows))
    _cases.run_and_check(h, mode, M, N, K, False, tB, seed=81, dist="normal", rows=rows)
    if K <= 1024:
        _cases.run_and_check(h, mode, M, N, K, False, tB, seed=83, dist="int", rows=rows, exact=True)
        assert h.plan()["schedule"] == "tail_split"
    # beta != 0 adds a read of C to the reduction, which may tip the planner
    # back to whole tiles; either way the result must hold
    _cases.run_and_check(h, mode, M, N, K, False, tB, alpha=0.5, beta=1.0, seed=82, dist="normal", rows=rows)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("splits", [2, 5])
def test_forced_split_k(h, mode, splits):
    h.set_option("split_k", splits)
    _cases.run_and_check(h, mode, 200, 272, 1000, False, True, alpha=0.75, beta=0.5, seed=23, dist="normal")
    # the planner rounds the slices to whole K blocks, so 5 may become 4
    assert 1 < h.plan()["split_k"] <= splits


@pytest.mark.parametrize("tA,tB", TRANS)
@pytest.mark.parametrize("M,N,K", [(1000, 700, 3000), (130, 390, 20000), (4000, 384, 384)])
def test_fp32_stream_k(h, tA, tB, M, N, K):
    """FP32 shapes whose tiles do not fill whole waves run as stream-K: runs
    of k-tiles that end mid-tile, partial tiles summed by the fixup kernel."""
    rows = _cases.sample_rows(M) if M * N * K > 2e9 else None
    _cases.run_and_check(h, "fp32", M, N, K, tA, tB, alpha=0.5, beta=0.75, seed=61, dist="normal", rows=rows)
    assert h.plan()["schedule"] == "stream_k"
    _cases.run_and_check(h, "fp32", M, N, min(K, 1024), tA, tB, seed=62, dist="int", exact=True)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("M,N,K,tA,tB,auto", [(5000, 1000, 520, True, False, "inline"),
                                              (4000, 384, 384, False, False, "kernel"),
                                              (1000, 700, 3000, False, True, "kernel"),
                                              (130, 390, 20000, True, True, "kernel")])
def test_fp32_stream_k_fixup_forms(h, tile_n, M, N, K, tA, tB, auto):
    """Stream-K partial tiles summed by the fixup kernel or by the last CTA
    to finish a part of each tile: both sum the parts in ascending k order,
    so the results are bit-identical, and the per-tile arrival counters the
    second form uses are back at zero after every call (it runs twice)."""
    ops, c0 = _cases.make("fp32", M, N, K, tA, tB, seed=63, dist="normal", with_c=True)
    out = {}
    for fix in (0, 1, 2, 2):
        h.set_option("tile_n", tile_n)
        h.set_option("sk_fixup", fix)
        C = c0.clone().cuda()
        h.run(ops.A, ops.B, C, mode="fp32", transA=tA, transB=tB, alpha=0.5, beta=0.75)
        assert h.check_device() == 0
        plan = h.plan()
        if plan["schedule"] != "stream_k":
            pytest.skip(f"tile_n {tile_n}: the planner chose {plan['schedule']}")
        want = {0: None, 1: "kernel", 2: "inline"}[fix]
        assert plan["sk_fixup"] == (want or plan["sk_fixup"]), plan
        if fix == 0 and tile_n == 128:
            assert plan["sk_fixup"] == auto, plan
        out.setdefault(fix, []).append(C.cpu().numpy())
    h.set_option("sk_fixup", 0)
    with pytest.raises(dg.GemmError) as e:
        h.set_option("sk_fixup", 3)
    assert e.value.status == 1  # GEMM_ERR_INVALID_VALUE
    assert np.array_equal(out[1][0], out[2][0]) and np.array_equal(out[2][0], out[2][1])
    assert np.array_equal(out[0][0], out[1][0])
    rows = _cases.sample_rows(M)
    _cases.run_and_check(h, "fp32", M, N, K, tA, tB, alpha=0.5, beta=0.75, seed=63, dist="normal", rows=rows)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("tA,tB", TRANS)
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (1000, 700, 3000), (129, 257, 1025)])
def test_fp32_tile_widths(h, tile_n, tA, tB, M, N, K):
    """Both SIMT tile widths, whatever schedule the planner gives them."""
    h.set_option("tile_n", tile_n)
    rows = _cases.sample_rows(M) if M * N * K > 2e9 else None
    _cases.run_and_check(h, "fp32", M, N, K, tA, tB, alpha=-0.5, beta=0.5, seed=67, dist="normal", rows=rows)
    assert h.plan()["tile_n"] == tile_n
    _cases.run_and_check(h, "fp32", M, N, min(K, 1024), tA, tB, seed=68, dist="int", exact=True)


@pytest.mark.parametrize("pre", [1, 2])
@pytest.mark.parametrize("tA,tB", TRANS)
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (129, 257, 1025), (1000, 700, 3000)])
def test_fp32_pretranspose(h, pre, tA, tB, M, N, K):
    """FP32 with K-contiguous operands read in place (1) or transposed into
    the workspace first (2), on ragged shapes and both schedules."""
    h.set_option("pretranspose", pre)
    rows = _cases.sample_rows(M) if M * N * K > 2e9 else None
    _cases.run_and_check(h, "fp32", M, N, K, tA, tB, alpha=1.25, beta=-0.5, seed=71, dist="normal", rows=rows)
    # pre = 2 transposes the K-contiguous operands; an M/N-contiguous one
    # whose rows are not 16-byte aligned is re-packed (neither with pre = 1)
    a_copy = (not tA) or M % 4 != 0
    b_copy = tB or N % 4 != 0
    want = 0 if pre == 1 else ((1 if a_copy else 0) | (2 if b_copy else 0))
    assert h.plan()["packed"] == want
    _cases.run_and_check(h, "fp32", M, N, min(K, 1024), tA, tB, seed=72, dist="int", exact=True)


@pytest.mark.parametrize("tile_n", [128, 256])
@pytest.mark.parametrize("pre", [0, 1])
@pytest.mark.parametrize("M,N,K", [(200, 300, 1), (129, 130, 3), (300, 260, 17), (1000, 384, 383),
                                   (257, 520, 1537)])
def test_fp32_k_contiguous_a_transposed_in_kernel(h, tile_n, pre, M, N, K):
    """A stored M x K (K contiguous, rows 16-byte aligned) goes to shared
    memory row by row and is transposed there.  Its rows sit in a wider
    buffer whose padding columns hold NaN: a K quad that runs past K must be
    zero-filled, not read, or the NaN would reach C."""
    h.set_option("tile_n", tile_n)
    h.set_option("pretranspose", pre)
    lda = (K + 3) // 4 * 4 + 4
    a = si.normal((M, K), 81)
    b = si.normal((K, N), 82)
    c0 = si.normal((M, N), 83)
    buf = torch.full((M, lda), float("nan"), device="cuda")
    buf[:, :K] = a.cuda()
    A = buf[:, :K]
    C = c0.clone().cuda()
    h.run(A, b.cuda(), C, mode="fp32", alpha=0.75, beta=-0.5)
    assert h.check_device() == 0
    assert h.plan()["packed"] & 1 == 0  # read in place, not copied into the workspace
    ref, D = oracle.gemm("fp32", a.numpy(), b.numpy(), alpha=0.75, beta=-0.5, C=c0.numpy())
    _gate.assert_within("fp32", C.cpu().numpy(), ref, D, 0.75, -0.5, c0.numpy(), what=f"{M}x{N}x{K}")
    ai = si.integers((M, K), 84)
    bi = si.integers((K, N), 85)
    buf[:, :K] = ai.cuda()
    C = torch.full((M, N), float("nan"), device="cuda")
    h.run(A, bi.cuda(), C, mode="fp32")
    ref, _ = oracle.gemm("fp32", ai.numpy(), bi.numpy())
    assert np.array_equal(C.cpu().numpy().astype(np.float64), ref), "not bit-exact"


@pytest.mark.parametrize("pre", [0, 2])
@pytest.mark.parametrize("M,N,K,splits", [(384, 1152, 4096, 0), (300, 260, 1000, 0), (129, 130, 70, 0),
                                          (1000, 384, 2048, 3), (256, 300, 16384, 0)])
def test_tf32_mn_major_a_through_tmem(h, pre, M, N, K, splits):
    """TF32 with A stored K x M (MN-major) on 128-column tiles: the kernel
    moves each stage of A into TMEM and the MMA reads it there (pre = 0), or
    the planner transposes A into the workspace first (pre = 2).  Ragged
    M, N and K, split-K and deep K."""
    h.set_option("tile_n", 128)
    h.set_option("pretranspose", pre)
    if splits:
        h.set_option("split_k", splits)
    rows = _cases.sample_rows(M) if M * N * K > 2e9 else None
    _cases.run_and_check(h, "tf32", M, N, K, True, False, alpha=0.75, beta=0.5, seed=91, dist="normal", rows=rows)
    plan = h.plan()
    assert plan["family"] == "tc" and plan["tile_n"] == 128 and plan["cluster"] == 1
    if M % 4 == 0:  # A rows 16-byte aligned: read in place (N < 1536) unless asked to transpose
        assert plan["packed"] & 1 == (0 if pre == 0 and N < 1536 else 1)
    _cases.run_and_check(h, "tf32", M, N, min(K, 1024), True, False, seed=92, dist="int", exact=True)


@pytest.mark.parametrize("M,N,K", [(384, 1152, 4096), (200, 610, 4100), (129, 1000, 8192)])
def test_tf32_weight_gradient_form(h, M, N, K):
    """TF32 C = A^T B with A stored K x M, B stored K x N, N >= 2 M and
    K >= 4096 (a weight gradient): computed as C^T = B^T A into the
    handle's second buffer (B through TMEM, only A transposed) and
    transposed into place.  Ragged M, N and K; alpha scales the product;
    integer inputs bit-exact."""
    rows = _cases.sample_rows(M) if M * N * K > 2e9 else None
    _cases.run_and_check(h, "tf32", M, N, K, True, False, alpha=0.75, seed=95, dist="normal", rows=rows)
    plan = h.plan()
    assert plan["family"] == "tc" and plan["tile_n"] == 128 and plan["pair_mma"] == 0, plan
    _cases.run_and_check(h, "tf32", M, N, K, True, False, seed=96, dist="int", exact=True)


@pytest.mark.parametrize("mode", MODES)
def test_many_tiles_persistent_loop(h, mode):
    # More tiles than SMs: every CTA of the persistent grid loops over several
    # tiles and both TMEM accumulators are reused.
    _cases.run_and_check(h, mode, 2048 + 64, 2048 + 40, 256, seed=29, dist="normal", rows=_cases.sample_rows(2112))


@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"])
@pytest.mark.parametrize("tA,tB", TRANS)
def test_unaligned_leading_dimension(h, mode, tA, tB):
    # N = K = 65: a row of 65 elements breaks the 16-byte rule of the TMA unit,
    # so TF32/BF16 operands go through the re-pack into the workspace.
    _cases.run_and_check(h, mode, 190, 65, 65, tA, tB, seed=31, dist="normal")


@pytest.mark.parametrize("pre", [0, 1])
@pytest.mark.parametrize("tA,tB", TRANS)
@pytest.mark.parametrize("M,N,K", [(700, 65, 384), (700, 384, 65), (65, 300, 1000)])
def test_fp32_misaligned_operands(h, pre, tA, tB, M, N, K):
    """FP32 operands whose rows are not 16-byte aligned (a dimension of 65):
    the planner re-packs them into an aligned workspace copy (or transposes
    a K-contiguous one); with pretranspose = 1 the kernel reads them in place
    with 4-byte copies and scalar FMAs."""
    h.set_option("pretranspose", pre)
    _cases.run_and_check(h, "fp32", M, N, K, tA, tB, seed=39, dist="normal")
    lda = M if tA else K
    ldb = K if tB else N
    plan = h.plan()
    if pre == 1:
        assert plan["packed"] == 0
    elif lda % 4 or ldb % 4:
        assert plan["packed"] != 0
    _cases.run_and_check(h, "fp32", M, N, K, tA, tB, seed=40, dist="int", exact=True)


@pytest.mark.parametrize("mode", MODES)
def test_padded_leading_dimensions_and_offsets(h, mode):
    M, N, K = 150, 90, 70
    ops, _ = _cases.make(mode, M, N, K, seed=37, dist="normal")
    dt = ops.A.dtype
    # operands inside larger buffers, starting one element in
    Abig = torch.zeros((M, K + 9), dtype=dt, device="cuda")
    Bbig = torch.zeros((K, N + 5), dtype=dt, device="cuda")
    Abig[:, 1:K + 1] = ops.A
    Bbig[:, 3:N + 3] = ops.B
    Cbig = torch.full((M + 2, N + 11), 7.0, device="cuda")
    A, B, C = Abig[:, 1:K + 1], Bbig[:, 3:N + 3], Cbig[1:M + 1, 2:N + 2]
    h.run(A, B, C, mode=mode)
    assert h.check_device() == 0
    ref, D = oracle.gemm(mode, ops.a_host, ops.b_host)
    _gate.assert_within(mode, C.cpu().numpy(), ref, D)
    host = Cbig.cpu().numpy()
    mask = np.ones_like(host, dtype=bool)
    mask[1:M + 1, 2:N + 2] = False
    assert np.all(host[mask] == 7.0), "wrote outside C"


@pytest.mark.parametrize("mode", MODES)
def test_guard_bands_untouched(h, mode):
    """C sits inside a buffer whose every other element is a NaN canary."""
    M, N, K = 257, 130, 48
    ops, _ = _cases.make(mode, M, N, K, seed=41, dist="normal")
    canary = float("nan")
    buf = torch.full(((M + 4) * (N + 8) + 64,), canary, device="cuda")
    C = buf[32:32 + (M + 4) * (N + 8)].view(M + 4, N + 8)[2:M + 2, 4:N + 4]
    h.run(ops.A, ops.B, C, mode=mode)
    assert h.check_device() == 0
    ref, D = oracle.gemm(mode, ops.a_host, ops.b_host)
    _gate.assert_within(mode, C.cpu().numpy(), ref, D)
    host = buf.cpu().numpy()
    inside = np.zeros(host.shape, dtype=bool)
    idx = 32 + (np.arange(2, M + 2)[:, None] * (N + 8) + np.arange(4, N + 4)[None, :])
    inside[idx.ravel()] = True
    assert np.all(np.isnan(host[~inside])), "a canary was overwritten"


# ------------------------------------------------------------ degenerate calls
@pytest.mark.parametrize("mode", MODES)
def test_k_zero_and_alpha_zero(h, mode):
    M, N = 70, 50
    c0 = si.normal((M, N), 43)
    dt = torch.bfloat16 if mode == "bf16" else torch.float32
    C = c0.clone().cuda()
    h.run(torch.empty((M, 0), dtype=dt, device="cuda"), torch.empty((0, N), dtype=dt, device="cuda"), C,
          mode=mode, beta=-2.0)
    assert torch.equal(C.cpu(), -2.0 * c0)
    C = torch.full((M, N), float("nan"), device="cuda")
    A = torch.full((M, 8), float("nan"), device="cuda").to(dt)
    B = torch.ones((8, N), device="cuda").to(dt)
    h.run(A, B, C, mode=mode, alpha=0.0, beta=0.0)
    assert torch.equal(C.cpu(), torch.zeros(M, N))


def test_empty_output_is_a_no_op(h):
    C = torch.empty((0, 5), device="cuda")
    h.run(torch.empty((0, 3), device="cuda"), torch.empty((3, 5), device="cuda"), C)
    assert h.plan()["kernels"] == 0


def test_beta_zero_ignores_nan_in_c(h):
    for mode in MODES:
        _cases.run_and_check(h, mode, 140, 150, 40, beta=0.0, seed=47)  # C starts as NaN


def test_bad_arguments_launch_nothing(h):
    C = torch.full((4, 4), 3.0, device="cuda")
    A = torch.ones((4, 4), device="cuda")
    with pytest.raises(dg.GemmError) as e:
        h.run_ptr("fp32", 0, 0, 4, 4, 4, 1.0, A.data_ptr(), 3, A.data_ptr(), 4, 0.0, C.data_ptr(), 4)
    assert e.value.status == 1
    assert torch.equal(C.cpu(), torch.full((4, 4), 3.0))
    with pytest.raises(dg.GemmError):
        h.set_option("family", "tc")
        h.run(A, A, C, mode="fp32")  # the FP32 mode has no tensor-core family
    assert torch.equal(C.cpu(), torch.full((4, 4), 3.0))


# ------------------------------------------------------------ TF32 operand rule
def test_tf32_operand_reduction_matches_oracle_reading():
    """A one-column probe: C[i] = a_i * 1 for a_i = 1 + i * 2^-12 .. shows
    whether the tensor cores drop or round the 13 low mantissa bits."""
    dg.load(build_if_missing=True)
    h = dg.Gemm()
    M = 64
    a = torch.tensor([1.0 + i * 2.0 ** -12 for i in range(M)], dtype=torch.float32).reshape(M, 1)
    a = torch.cat([a, -a[: M // 2]], 0)
    b = torch.ones((1, 16), dtype=torch.float32)
    C = torch.zeros((a.shape[0], 16), device="cuda")
    h.run(a.cuda(), b.cuda(), C, mode="tf32")
    got = C.cpu().numpy()[:, 0]
    want = oracle.tf32(a.numpy()[:, 0])          # the oracle's reading (truncation)
    other = oracle.tf32(a.numpy()[:, 0], "nearest_away")
    h.close()
    assert np.array_equal(got, want), (got[:8], want[:8], other[:8])


# ------------------------------------------------------------ the GPT shapes, full size
@pytest.mark.parametrize("mode", ["fp32", "tf32"])
@pytest.mark.parametrize("proj", range(len(si.GPT_PROJECTIONS)))
def test_gpt_projection_shapes_sampled(h, mode, proj):
    """Full-size forward, dX and dW of one projection in the launch
    configuration the benchmark uses; sampled rows against the oracle."""
    name, kin, nout = si.GPT_PROJECTIONS[proj]
    X, W, dY = si.gpt_tensors(proj, kin, nout)
    Xd, Wd, dYd = X.cuda(), W.cuda(), dY.cuda()
    T = si.GPT_TOKENS
    cases = [("fwd", Xd, Wd, X, W, False, False, T, nout, kin),
             ("dX", dYd, Wd, dY, W, False, True, T, kin, nout),
             ("dW", Xd, dYd, X, dY, True, False, kin, nout, T)]
    for tag, Ad, Bd, Ah, Bh, tA, tB, M, N, K in cases:
        C = torch.full((M, N), float("nan"), device="cuda")
        h.run(Ad, Bd, C, mode=mode, transA=tA, transB=tB)
        assert h.check_device() == 0
        got = C.cpu().numpy()
        width = 1 if K > 4096 else 2
        for r0, r1 in _cases.sample_rows(M, width=width):
            ref, D = oracle.gemm(mode, Ah.numpy(), Bh.numpy(), transA=tA, transB=tB, rows=(r0, r1))
            _gate.assert_within(mode, got[r0:r1], ref, D, what=f"{name}.{tag} rows {r0}:{r1}")


# ------------------------------------------------------------ small M (swapped form)
@pytest.mark.parametrize("mode", ["bf16", "tf32"])
@pytest.mark.parametrize("tB", [False, True])
@pytest.mark.parametrize("M,N,K", [(1, 1000, 700), (7, 300, 64), (16, 129, 2000), (3, 65, 40)])
def test_skinny_ragged(h, mode, tB, M, N, K):
    _cases.run_and_check(h, mode, M, N, K, False, tB, seed=53, dist="normal")
    assert h.plan()["family"] == "skinny"
    _cases.run_and_check(h, mode, M, N, K, False, tB, alpha=0.5, beta=1.0, seed=54, dist="normal")


@pytest.mark.parametrize("mode", ["bf16", "tf32"])
@pytest.mark.parametrize("tB", [False, True])
@pytest.mark.parametrize("cs", [1, 2, 3, 8, 12, 16])
def test_skinny_cluster_k_slices(h, mode, tB, cs):
    """The small-M kernel with K cut into `cs` slices across one cluster
    (above 8: non-portable cluster sizes), slices summed in distributed
    shared memory; ragged N (3 tiles, the last partial) and ragged K."""
    h.set_option("family", "skinny")
    h.set_option("split_k", cs)
    M, N, K = 5, 300, 3000 if mode == "bf16" else 1500
    _cases.run_and_check(h, mode, M, N, K, False, tB, seed=61, dist="normal")
    plan = h.plan()
    assert plan["family"] == "skinny" and plan["split_k"] == cs and plan["cluster"] == cs
    assert plan["grid"] == 3 * cs
    _cases.run_and_check(h, mode, M, N, K, False, tB, alpha=0.5, beta=1.0, seed=62, dist="normal")


@pytest.mark.parametrize("mode", ["bf16", "tf32"])
@pytest.mark.parametrize("cs", [1, 8, 13])
def test_skinny_cluster_integers_bit_exact(h, mode, cs):
    h.set_option("split_k", cs)
    K = 1024
    _cases.run_and_check(h, mode, 16, 260, K, False, True, seed=63, dist="int", exact=True)
    kb = -(-K // (64 if mode == "bf16" else 32))
    per = -(-kb // cs)
    assert h.plan()["cluster"] == -(-kb // per)  # slices actually used: none of them empty


@pytest.mark.parametrize("M", [1, 16])
def test_skinny_one_slice_many_tiles(h, M):
    """Between one and two waves of weight tiles: one CTA per tile, no
    split, C written straight from TMEM."""
    N, K = 128 * 160 - 37, 200
    rows = [(0, M)]
    _cases.run_and_check(h, "bf16", M, N, K, False, False, seed=64, dist="normal", rows=rows)
    plan = h.plan()
    assert plan["family"] == "skinny" and plan["split_k"] == 1 and plan["grid"] == 160


def _column_ranges(N, tile=128, width=3):
    picks = sorted({0, tile - 1, N // 2, N - width})
    return [(c, min(c + width, N)) for c in picks if 0 <= c < N]


@pytest.mark.parametrize("M", si.SKINNY_M)
@pytest.mark.parametrize("w", range(len(si.SKINNY_WEIGHTS)))
@pytest.mark.parametrize("tB", [False, True])
def test_skinny_decode_shapes_sampled(h, M, w, tB):
    """The decode shapes at full size in bf16 (the benchmark's launch
    configuration), checked on sampled columns against the oracle."""
    K, N = si.SKINNY_WEIGHTS[w]
    a32 = si.normal((M, K), si.seed_for(4, w, 0))
    b32 = si.normal((N, K) if tB else (K, N), si.seed_for(4, w, 1), std=0.02)
    a16, b16 = si.to_bf16(a32), si.to_bf16(b32)
    C = torch.full((M, N), float("nan"), device="cuda")
    h.run(a16.cuda(), b16.cuda(), C, mode="bf16", transB=tB)
    assert h.check_device() == 0
    assert h.plan()["family"] == "skinny"
    got = C.cpu().numpy()
    abits, bbits = si.bf16_bits(a16), si.bf16_bits(b16)
    for c0, c1 in _column_ranges(N):
        bcols = bbits[c0:c1, :] if tB else bbits[:, c0:c1]
        ref, D = oracle.gemm("bf16", abits, bcols, transB=tB)
        _gate.assert_within("bf16", got[:, c0:c1], ref, D, what=f"skinny M={M} {K}x{N} cols {c0}:{c1}")
