"""The epilogue (gemm_run_epilogue) against the oracle: a per-column bias,
GELU after it, and the product with GELU'(Z) of a kept pre-activation, in
every kernel family and schedule -- applied in the split-K reduction where a
call ends with one that writes all of C, in the pass over C after the GEMM
otherwise (whole tiles, stream-K, tail slices, the small-M kernel), and in
the beta-only path for K = 0."""
import numpy as np
import pytest
import torch

import dense_gemm_transformer_gb300 as dg
import oracle
import seeded_inputs as si
from tests import _cases, _gate

pytestmark = pytest.mark.gpu

GELU_SLOPE = 1.13  # max |GELU'| and max |GELU''|-free bound on how GELU scales an input error


@pytest.fixture(scope="module")
def h():
    dg.load(build_if_missing=True)
    handle = dg.Gemm()
    yield handle
    handle.close()


@pytest.fixture(autouse=True)
def _reset(h):
    for name in ("split_k", "tile_n", "pretranspose", "pair"):
        h.set_option(name, 0)
    h.set_option("family", "auto")
    yield


def _check(mode, got, Y, D, act, bias, Z, alpha, beta, cin, what):
    ref = oracle.epilogue(act, Y, bias, Z)
    beta_c = np.abs(beta * cin.astype(np.float64)) if cin is not None else 0.0
    # the product's error (the mode's gate on |alpha| D, plus the one fp32
    # rounding of the beta * C term), scaled by at most |GELU'| <= 1.13, plus
    # the fp32 roundings of the bias add and of the activation itself
    extra = np.abs(Y) + (np.abs(bias.astype(np.float64))[None, :] if bias is not None else 0.0)
    bound = (GELU_SLOPE * (_gate.TOL[mode] * np.abs(alpha) * D + _gate.U32 * beta_c) + 4e-6 * (np.abs(ref) + extra)
             + 1e-30)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(err <= bound), (what, float(np.max(err / bound)))


CASES = [
    # mode, M, N, K, transA, transB, options  (what each exercises)
    ("fp32", 300, 260, 200, False, False, {}),                     # SIMT whole tiles
    ("fp32", 1000, 700, 3000, False, True, {}),                    # SIMT stream-K + fixup
    ("fp32", 200, 272, 1000, True, False, {"split_k": 3}),         # SIMT split-K + reduce
    ("tf32", 512, 512, 256, False, False, {}),                     # TC tiles, TMA-staged stores
    ("tf32", 384, 1152, 4096, True, False, {"tile_n": 128}),       # TC split-K, A through TMEM
    ("bf16", 2048, 2048, 256, False, False, {}),                   # TC pairs, one 256-row MMA
    ("bf16", 2304, 1000, 1024, False, True, {}),                   # ragged N
    ("bf16", 4096, 4096, 1024, False, True, {}),                   # tail slices + reduce
    ("bf16", 4, 1536, 8960, False, True, {}),                      # small M: cluster reduction
    ("bf16", 16, 8960, 1536, False, False, {}),                    # small M: clusters of 4
    ("tf32", 8, 1536, 896, False, True, {"split_k": 1}),           # small M: no split
]


@pytest.mark.parametrize("mode,M,N,K,tA,tB,opts", CASES)
@pytest.mark.parametrize("act,use_bias,beta", [("none", True, 0.0), ("gelu", True, 0.0), ("gelu", False, 0.5),
                                               ("dgelu", False, 0.0), ("dgelu", False, 1.0)])
def test_epilogue_matches_oracle(h, mode, M, N, K, tA, tB, opts, act, use_bias, beta):
    for k, v in opts.items():
        h.set_option(k, v)
    ops, c0 = _cases.make(mode, M, N, K, tA, tB, seed=101, dist="normal", with_c=True)
    alpha = 0.75
    bias = si.normal((N,), 102).numpy() if use_bias else None
    Z = si.normal((M, N), 103).numpy() if act == "dgelu" else None
    C = c0.clone().cuda() if beta != 0.0 else torch.full((M, N), float("nan"), device="cuda")
    h.run(ops.A, ops.B, C, mode=mode, transA=tA, transB=tB, alpha=alpha, beta=beta, act=act,
          bias=torch.from_numpy(bias).cuda() if bias is not None else None,
          aux=torch.from_numpy(Z).cuda() if Z is not None else None)
    assert h.check_device() == 0
    got = C.cpu().numpy()
    cin = c0.numpy() if beta != 0.0 else None
    rows = _cases.sample_rows(M) if M * N * K > 2e9 else [(0, M)]
    for r0, r1 in rows:
        Y, D = oracle.gemm(mode, ops.a_host, ops.b_host, transA=tA, transB=tB, alpha=alpha, beta=beta, C=cin,
                           rows=(r0, r1))
        _check(mode, got[r0:r1], Y, D, act, bias, Z[r0:r1] if Z is not None else None, alpha, beta,
               cin[r0:r1] if cin is not None else None, f"{mode} {M}x{N}x{K} rows {r0}:{r1}")


@pytest.mark.parametrize("mode", ["fp32", "tf32", "bf16"])
def test_bias_is_exact_on_integers(h, mode):
    """Integer operands and an integer bias: product and bias add are exact."""
    M, N, K = 300, 260, 512
    ops, _ = _cases.make(mode, M, N, K, seed=104, dist="int")
    bias = si.integers((N,), 105).numpy()
    C = torch.full((M, N), float("nan"), device="cuda")
    h.run(ops.A, ops.B, C, mode=mode, bias=torch.from_numpy(bias).cuda())
    Y, _ = oracle.gemm(mode, ops.a_host, ops.b_host)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), Y + bias.astype(np.float64)[None, :])


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_k_zero_applies_the_epilogue_to_beta_c(h, mode):
    M, N = 70, 50
    c0 = si.normal((M, N), 106)
    bias = si.normal((N,), 107)
    dt = torch.bfloat16 if mode == "bf16" else torch.float32
    C = c0.clone().cuda()
    h.run(torch.empty((M, 0), dtype=dt, device="cuda"), torch.empty((0, N), dtype=dt, device="cuda"), C, mode=mode,
          beta=-2.0, act="gelu", bias=bias.cuda())
    ref = oracle.epilogue("gelu", -2.0 * c0.numpy().astype(np.float64), bias.numpy())
    assert np.max(np.abs(C.cpu().numpy() - ref)) <= 4e-6 * (np.max(np.abs(ref)) + 1)


def test_epilogue_argument_checks(h):
    A = torch.randn(8, 8, device="cuda")
    C = torch.empty(8, 8, device="cuda")
    Z = torch.randn(8, 8, device="cuda")
    with pytest.raises(dg.GemmError):  # a bias with dgelu
        h.run(A, A, C, act="dgelu", aux=Z, bias=torch.zeros(8, device="cuda"))
    with pytest.raises(dg.GemmError):  # dgelu without Z
        h.run(A, A, C, act="dgelu")
    h.run(A, A, C, act="gelu")  # no bias is fine
    assert h.check_device() == 0
