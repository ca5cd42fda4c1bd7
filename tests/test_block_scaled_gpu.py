"""Block-scaled products (gemm_run_block_scaled) against the oracle's
block-scaled definition: MXFP8 (E4M3 / E5M2 elements, one E8M0 scale per 32
K) and NVFP4 (E2M1 elements two per byte, one UE4M3 scale per 16 K): the
decode shape M <= 16 (the small-M kernels) and M > 16 (128 x 128 tiles).

Products of the decoded elements and scales are exact in fp32 and the tensor
cores accumulate in fp32, so the FP8 gate (2e-3 of |alpha| D) applies.
Small integers with scales of 1/2, 1 and 2 are bit-exact in every order of
summation; they catch a scale read for the wrong block or row, a wrong
nibble order, or a partial last block handled wrongly.
"""
import numpy as np
import pytest
import torch

import dense_gemm_transformer_gb300 as dg
import oracle
import seeded_inputs as si
from tests import _gate

pytestmark = pytest.mark.gpu

MODES = {m: v[1:] for m, v in dg.BLOCK_SCALED_MODES.items()}  # mode -> (element, block, scale format)


@pytest.fixture(scope="module")
def h():
    dg.load(build_if_missing=True)
    handle = dg.Gemm()
    yield handle
    handle.close()


@pytest.fixture(autouse=True)
def _reset(h):
    h.set_option("split_k", 0)
    yield


def _padded(codes):
    """The codes on the device with each row padded to a multiple of 16
    bytes (the row pitch the TMA unit reads), as a view of the first
    `cols` bytes of each row: lda > K when K's bytes are not whole 16s."""
    rows, cols = codes.shape
    pitch = -(-max(cols, 1) // 16) * 16
    buf = torch.zeros((rows, pitch), dtype=torch.uint8, device="cuda")
    buf[:, :cols] = torch.from_numpy(codes).cuda()
    return buf[:, :cols]


def _run(h, mode, ac, sa, bc, sb, M, N, alpha=1.0, beta=0.0, c0=None):
    A, B = _padded(ac), _padded(bc)
    SA = dg.tile_block_scales(torch.from_numpy(sa).cuda())
    SB = dg.tile_block_scales(torch.from_numpy(sb).cuda())
    C = c0.clone().cuda() if c0 is not None else torch.full((M, N), float("nan"), device="cuda")
    h.run_block_scaled(A, SA, B, SB, C, mode=mode, alpha=alpha, beta=beta)
    assert h.check_device() == 0
    return C.cpu().numpy()


def _oracle(mode, ac, sa, bc, sb, alpha=1.0, beta=0.0, c0=None):
    elem, bs, sf = MODES[mode]
    return oracle.gemm_block_scaled(elem, elem, ac, sa, bc, sb, block=bs, scale_fmt=sf, alpha=alpha, beta=beta,
                                    C=None if c0 is None else c0.numpy())


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("M,N,K", [(1, 300, 512), (4, 1000, 2048), (16, 129, 1056), (7, 260, 3008), (16, 384, 200)])
def test_block_scaled_matches_oracle(h, mode, M, N, K):
    """Normal inputs quantised with per-block scales; ragged N, a partial last
    stage (K = 1056, 3008) and a partial last block (K = 200: 6.25 blocks of
    32, 12.5 of 16, rows padded to 16 bytes so lda > K), alpha / beta."""
    elem, bs, sf = MODES[mode]
    ac, sa = si.to_block_scaled(si.normal((M, K), 611), elem, bs, sf)
    bc, sb = si.to_block_scaled(si.normal((N, K), 612, std=0.02), elem, bs, sf)
    got = _run(h, mode, ac, sa, bc, sb, M, N)
    ref, D = _oracle(mode, ac, sa, bc, sb)
    _gate.assert_within("fp8", got, ref, D, what=f"{mode} {M}x{N}x{K}")
    plan = h.plan()
    assert plan["family"] == "skinny" and plan["tile_k"] == (256 if mode == "nvfp4" else 128), plan
    c0 = si.normal((M, N), 613)
    got = _run(h, mode, ac, sa, bc, sb, M, N, alpha=0.75, beta=-0.5, c0=c0)
    ref, D = _oracle(mode, ac, sa, bc, sb, alpha=0.75, beta=-0.5, c0=c0)
    _gate.assert_within("fp8", got, ref, D, 0.75, -0.5, c0.numpy(), what=f"{mode} {M}x{N}x{K} alpha/beta")


def _integer_codes(mode, shape, rng):
    """Codes of small integers exact in the element format."""
    elem = MODES[mode][0]
    if elem == "e2m1":
        vals = rng.choice(np.array([0.0, 1.0, 2.0, 3.0, 4.0, 6.0, -1.0, -2.0, -3.0, -4.0, -6.0]), size=shape)
        c = si._e2m1_codes(vals)
        return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    vals = rng.integers(-4, 5, size=shape).astype(np.float32)
    dt = torch.float8_e4m3fn if elem == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(vals).to(dt).view(torch.uint8).numpy().copy()


def _pow2_scales(mode, rows, blocks, rng):
    """Scales of 1/2, 1 and 2, drawn per (row, block)."""
    sf = MODES[mode][2]
    codes = np.array([126, 127, 128] if sf == "e8m0" else [0x30, 0x38, 0x40], dtype=np.uint8)
    return codes[rng.integers(0, 3, size=(rows, blocks))]


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("M,N,K,splits", [(16, 260, 1088, 0), (5, 130, 4096, 3), (16, 300, 4096, 16), (1, 128, 96, 1)])
def test_block_scaled_integers_bit_exact(h, mode, M, N, K, splits):
    """Integers times power-of-two scales: bit-exact, for the planner's K
    split and forced ones (1, 3 and 16 slices per cluster); K = 96 ends in a
    partial stage, and for MXFP8 in a whole block."""
    elem, bs, sf = MODES[mode]
    rng = np.random.default_rng(614 + K + splits)
    nb = -(-K // bs)
    ac, bc = _integer_codes(mode, (M, K), rng), _integer_codes(mode, (N, K), rng)
    sa, sb = _pow2_scales(mode, M, nb, rng), _pow2_scales(mode, N, nb, rng)
    if splits:
        h.set_option("split_k", splits)
    got = _run(h, mode, ac, sa, bc, sb, M, N)
    ref, _ = _oracle(mode, ac, sa, bc, sb)
    assert np.array_equal(got.astype(np.float64), ref), f"{mode} {M}x{N}x{K} splits {splits}"
    if splits:
        kb = -(-K // (256 if elem == "e2m1" else 128))  # 128-byte stages of K
        per = -(-kb // min(splits, kb))
        assert h.plan()["split_k"] == -(-kb // per), h.plan()


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("deep", [False, True])
def test_block_scaled_persistent_form(h, mode, deep):
    """Two or more waves of 128-row weight tiles go to the persistent kernel
    (each CTA streams tile after tile, no K split): ragged N, a partial last
    stage; normal inputs within the gate and integers bit-exact.  K = 1056
    keeps the activations' scale atoms in TMEM for the whole call; the deep
    K (more than 32 atoms) copies them with every stage."""
    elem, bs, sf = MODES[mode]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    K = (2400 if elem == "e2m1" else 4200) if deep else 1056
    M, N = 5, 128 * (2 * sms + 9) - 37
    ac, sa = si.to_block_scaled(si.normal((M, K), 617), elem, bs, sf)
    bc, sb = si.to_block_scaled(si.normal((N, K), 618, std=0.02), elem, bs, sf)
    got = _run(h, mode, ac, sa, bc, sb, M, N)
    plan = h.plan()
    assert plan["family"] == "skinny" and plan["cluster"] == 1 and plan["split_k"] == 1 and plan["grid"] == sms, plan
    ref, D = _oracle(mode, ac, sa, bc, sb)
    _gate.assert_within("fp8", got, ref, D, what=f"{mode} persistent {M}x{N}x{K}")
    rng = np.random.default_rng(619)
    nb = -(-K // bs)
    ac, bc = _integer_codes(mode, (M, K), rng), _integer_codes(mode, (N, K), rng)
    sa, sb = _pow2_scales(mode, M, nb, rng), _pow2_scales(mode, N, nb, rng)
    c0 = si.normal((M, N), 620)
    got = _run(h, mode, ac, sa, bc, sb, M, N, alpha=2.0, beta=1.0, c0=c0)
    ref, _ = _oracle(mode, ac, sa, bc, sb, alpha=2.0, beta=1.0, c0=c0)
    # integers and power-of-two scales: exact products and sums; adding
    # beta * C rounds the result once
    assert np.all(np.abs(got.astype(np.float64) - ref) <= 2.0 ** -24 * np.abs(ref)), mode


def _random_codes(mode, shape, rng):
    """Random finite codes of moderate magnitude (no scaling needed)."""
    elem = MODES[mode][0]
    if elem == "e2m1":
        return rng.integers(0, 256, size=(shape[0], shape[1] // 2), dtype=np.uint8)
    lo, hi = (0x20, 0x50) if elem == "e4m3" else (0x20, 0x48)
    mag = rng.integers(lo, hi, size=shape, dtype=np.uint8)
    return mag | (rng.integers(0, 2, size=shape, dtype=np.uint8) << 7)


def _random_scales(mode, rows, blocks, rng):
    sf = MODES[mode][2]
    lo, hi = (120, 131) if sf == "e8m0" else (0x28, 0x48)
    return rng.integers(lo, hi, size=(rows, blocks), dtype=np.uint8)


@pytest.mark.parametrize("mode", ["nvfp4", "mxfp8_e4m3"])
@pytest.mark.parametrize("M", [1, 16])
@pytest.mark.parametrize("w", range(len(si.SKINNY_WEIGHTS)))
def test_block_scaled_decode_shapes_sampled(h, mode, M, w):
    """The decode shapes at full size (weights N x K), in the launch
    configuration the benchmark times, on sampled columns."""
    K, N = si.SKINNY_WEIGHTS[w]
    elem, bs, sf = MODES[mode]
    rng = np.random.default_rng(615 + w)
    nb = -(-K // bs)
    ac, bc = _random_codes(mode, (M, K), rng), _random_codes(mode, (N, K), rng)
    sa, sb = _random_scales(mode, M, nb, rng), _random_scales(mode, N, nb, rng)
    got = _run(h, mode, ac, sa, bc, sb, M, N)
    for c0 in sorted({0, 127, 128, N // 2, N - 130, N - 3}):
        c1 = min(c0 + 3, N)
        ref, D = _oracle(mode, ac, sa, np.ascontiguousarray(bc[c0:c1]), np.ascontiguousarray(sb[c0:c1]))
        _gate.assert_within("fp8", got[:, c0:c1], ref, D, what=f"{mode} M={M} {K}x{N} cols {c0}:{c1}")


def test_scale_tiling_layout(h):
    """The tiled layout written by gemm_block_scales_tile, against a direct
    restatement of its definition (row r of a 128-row tile and block j of a
    group of four at byte 16 (r % 32) + 4 (r / 32) + j of the group's atom)."""
    rng = np.random.default_rng(616)
    rows, blocks = 300, 70
    S = rng.integers(1, 256, size=(rows, blocks), dtype=np.uint8)
    T = dg.tile_block_scales(torch.from_numpy(S).cuda()).cpu().numpy()
    groups = 4 * -(-blocks // 16)
    assert T.size == -(-rows // 128) * groups * 512
    want = np.zeros_like(T)
    for r in range(-(-rows // 128) * 128):
        for b in range(groups * 4):
            rt, rr, g, j = r // 128, r % 128, b // 4, b % 4
            off = (rt * groups + g) * 512 + 16 * (rr % 32) + 4 * (rr // 32) + j
            want[off] = S[r, b] if (r < rows and b < blocks) else 0
    assert np.array_equal(T, want)


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("M,N,K", [(200, 300, 1056), (256, 256, 4096), (1000, 130, 520), (17, 129, 96)])
def test_block_scaled_large_m(h, mode, M, N, K):
    """M > 16: the persistent kernel on 128 x 128 tiles, both operands'
    scale atoms brought with every stage.  Ragged M and N, a partial last
    stage (K = 1056, 520, 96) and a partial last block (K = 520 in MXFP8:
    16.25 blocks of 32), alpha / beta, then integers with power-of-two
    scales bit-exact."""
    elem, bs, sf = MODES[mode]
    ac, sa = si.to_block_scaled(si.normal((M, K), 621), elem, bs, sf)
    bc, sb = si.to_block_scaled(si.normal((N, K), 622, std=0.02), elem, bs, sf)
    got = _run(h, mode, ac, sa, bc, sb, M, N)
    ref, D = _oracle(mode, ac, sa, bc, sb)
    _gate.assert_within("fp8", got, ref, D, what=f"{mode} {M}x{N}x{K}")
    plan = h.plan()
    assert plan["family"] == "tc" and plan["tile_n"] == 128, plan
    c0 = si.normal((M, N), 623)
    got = _run(h, mode, ac, sa, bc, sb, M, N, alpha=0.75, beta=-0.5, c0=c0)
    ref, D = _oracle(mode, ac, sa, bc, sb, alpha=0.75, beta=-0.5, c0=c0)
    _gate.assert_within("fp8", got, ref, D, 0.75, -0.5, c0.numpy(), what=f"{mode} {M}x{N}x{K} alpha/beta")
    rng = np.random.default_rng(624 + M + K)
    nb = -(-K // bs)
    ac, bc = _integer_codes(mode, (M, K), rng), _integer_codes(mode, (N, K), rng)
    sa, sb = _pow2_scales(mode, M, nb, rng), _pow2_scales(mode, N, nb, rng)
    got = _run(h, mode, ac, sa, bc, sb, M, N)
    ref, _ = _oracle(mode, ac, sa, bc, sb)
    assert np.array_equal(got.astype(np.float64), ref), f"{mode} {M}x{N}x{K} integers"


def test_block_scaled_argument_checks(h):
    C = torch.full((4, 256), 5.0, device="cuda")
    A = torch.zeros((4, 64), dtype=torch.uint8, device="cuda")
    B = torch.zeros((256, 64), dtype=torch.uint8, device="cuda")
    S = dg.tile_block_scales(torch.zeros((256, 4), dtype=torch.uint8, device="cuda"))
    with pytest.raises(dg.GemmError) as e:  # scales not 16-byte aligned
        h.run_block_scaled(A, S[1:], B, S, C, mode="mxfp8_e4m3")
    assert e.value.status == 3
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), torch.full((4, 256), 5.0))
    # K == 0: C = beta * C, nothing read
    h.run_block_scaled(torch.zeros((4, 0), dtype=torch.uint8, device="cuda"), S,
                       torch.zeros((256, 0), dtype=torch.uint8, device="cuda"), S, C, mode="nvfp4", beta=2.0)
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), torch.full((4, 256), 10.0))
