"""Parity at the benchmark configurations' own sizes, in the launch
configuration the planner picks for them (the one the benchmark times).

* The square sweep: M = N = K in {1024, 2048, 4096}, every mode, inputs
  N(0, 1), alpha = 1, beta = 0 and alpha = 0.5, beta = 1 with C N(0, 1):
  every element against the oracle.
* The large BF16 shapes, 8192^3 and 8192 x 28672 x 8192, N(0, 1) rounded to
  bf16: whole rows at the edges of tiles, CTA pairs, the start of any K-sliced
  last rows and the bottom edge, every column; and the same rows bit-exact on
  small-integer inputs (K = 8192: every partial sum is an integer below
  2^17, exact in fp32 in any order).

The tolerance is the stated one (tests/_gate.py): |C - Cref| <= tol * |alpha|
* D after the one fp32 rounding of beta * C.
"""
import numpy as np
import pytest
import torch

import dense_gemm_transformer_gb300 as dg
import oracle
import seeded_inputs as si
from tests import _cases, _gate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    dg.load(build_if_missing=True)
    handle = dg.Gemm()
    yield handle
    handle.close()


def _host_and_device(mode, t):
    if mode == "bf16":
        t16 = si.to_bf16(t)
        return si.bf16_bits(t16), t16.cuda()
    return t.numpy(), t.cuda()


@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"])
@pytest.mark.parametrize("n_index", range(len(si.SQUARE_SWEEP)))
def test_square_sweep_full_size(h, mode, n_index):
    n = si.SQUARE_SWEEP[n_index]
    a_host, A = _host_and_device(mode, si.normal((n, n), si.seed_for(2, n_index, 0)))
    b_host, B = _host_and_device(mode, si.normal((n, n), si.seed_for(2, n_index, 1)))
    c0 = si.normal((n, n), si.seed_for(2, n_index, 2))
    for alpha, beta in ((1.0, 0.0), (0.5, 1.0)):
        C = c0.clone().cuda() if beta != 0.0 else torch.full((n, n), float("nan"), device="cuda")
        h.run(A, B, C, mode=mode, alpha=alpha, beta=beta)
        assert h.check_device() == 0
        plan = h.plan()
        assert plan["family"] == ("simt" if mode == "fp32" else "tc"), plan
        got = C.cpu().numpy()
        cin = c0.numpy() if beta != 0.0 else None
        ref, D = oracle.gemm(mode, a_host, b_host, alpha=alpha, beta=beta, C=cin)
        _gate.assert_within(mode, got, ref, D, alpha, beta, cin, what=f"square {n} a={alpha} b={beta} plan {plan}")


def _large_rows(M, plan):
    """Rows at tile (128) and pair (256) edges near the top, the middle and
    the bottom, at every 1024-row boundary, and the bottom rows."""
    picks = {0, 127, 128, 255, 256, M // 2 - 1, M // 2, M - 257, M - 256, M - 129, M - 128, M - 1}
    picks |= {r for b in range(1024, M, 1024) for r in (b - 1, b)}
    return [(r, r + 1) for r in sorted(p for p in picks if 0 <= p < M)]


@pytest.mark.parametrize("shape_index", range(len(si.LARGE_BF16)))
def test_large_bf16_sampled_rows(h, shape_index):
    M, N, K = si.LARGE_BF16[shape_index]
    a_host, A = _host_and_device("bf16", si.normal((M, K), si.seed_for(3, shape_index, 0)))
    b_host, B = _host_and_device("bf16", si.normal((K, N), si.seed_for(3, shape_index, 1)))
    C = torch.full((M, N), float("nan"), device="cuda")
    h.run(A, B, C, mode="bf16")
    assert h.check_device() == 0
    plan = h.plan()
    assert plan["family"] == "tc" and plan["pair_mma"] == 1, plan
    got = C.cpu().numpy()
    del C
    rows = _large_rows(M, plan)
    for r0, r1 in rows:
        ref, D = oracle.gemm("bf16", a_host, b_host, rows=(r0, r1))
        _gate.assert_within("bf16", got[r0:r1], ref, D, what=f"{M}x{N}x{K} row {r0} plan {plan}")
    del A, B, got
    torch.cuda.empty_cache()
    # small integers in [-4, 4]: bit-exact on the same rows
    ai, A = _host_and_device("bf16", si.integers((M, K), si.seed_for(3, shape_index, 3)))
    bi, B = _host_and_device("bf16", si.integers((K, N), si.seed_for(3, shape_index, 4)))
    C = torch.full((M, N), float("nan"), device="cuda")
    h.run(A, B, C, mode="bf16")
    assert h.check_device() == 0
    got = C.cpu().numpy()
    for r0, r1 in rows:
        ref, _ = oracle.gemm("bf16", ai, bi, rows=(r0, r1))
        assert np.array_equal(got[r0:r1].astype(np.float64), ref), f"{M}x{N}x{K} integers row {r0} not bit-exact"
