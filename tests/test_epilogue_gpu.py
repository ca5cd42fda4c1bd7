"""The epilogue (gemm_run_epilogue) against the oracle: a per-column bias,
GELU after it, and the product with GELU'(Z) of a kept pre-activation, in
every kernel family and schedule -- fused into the tensor-core kernel's
epilogue warps where A is read K-major (whole tiles, TMA-staged and direct
stores, pairs, tail slices with their reduction), applied in the split-K
reduction where a call ends with one that writes all of C, in the pass over
C after the GEMM otherwise (SIMT tiles and stream-K, A through TMEM, the
small-M kernels), and in the beta-only path for K = 0.  GELU itself (an
Abramowitz-Stegun erfc) is swept densely against the oracle and against
CUDA's erf."""
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
    # mode, M, N, K, transA, transB, options, fused in the GEMM kernel  (what each exercises)
    ("fp32", 300, 260, 200, False, False, {}, False),                  # SIMT whole tiles
    ("fp32", 1000, 700, 3000, False, True, {}, False),                 # SIMT stream-K + fixup
    ("fp32", 200, 272, 1000, True, False, {"split_k": 3}, False),      # SIMT split-K + reduce
    ("tf32", 512, 512, 256, False, False, {}, True),                   # TC tiles, TMA-staged stores
    ("tf32", 384, 1152, 4096, True, False, {"tile_n": 128}, False),    # TC split-K, A through TMEM
    ("tf32", 384, 1152, 4096, True, False, {"tile_n": 256}, True),     # TC split-K, A transposed first
    ("tf32", 700, 650, 300, False, True, {"tile_n": 192}, True),       # TC 192-column pairs
    ("bf16", 2048, 2048, 256, False, False, {}, True),                 # TC pairs, one 256-row MMA
    ("bf16", 2304, 1000, 1024, False, True, {}, True),                 # ragged N
    ("bf16", 4096, 4096, 1024, False, True, {}, True),                 # tail slices + reduce
    ("bf16", 600, 520, 96, True, False, {}, False),                    # MN-major A read in place
    ("bf16", 4, 1536, 8960, False, True, {}, False),                   # small M: cluster reduction
    ("bf16", 16, 8960, 1536, False, False, {}, False),                 # small M: clusters of 4
    ("tf32", 8, 1536, 896, False, True, {"split_k": 1}, False),        # small M: no split
]


@pytest.mark.parametrize("mode,M,N,K,tA,tB,opts,fused", CASES)
@pytest.mark.parametrize("act,use_bias,beta", [("none", True, 0.0), ("gelu", True, 0.0), ("gelu", False, 0.5),
                                               ("dgelu", False, 0.0), ("dgelu", False, 1.0)])
def test_epilogue_matches_oracle(h, mode, M, N, K, tA, tB, opts, fused, act, use_bias, beta):
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
    assert h.plan()["epilogue_fused"] == (1 if fused else 0), h.plan()
    got = C.cpu().numpy()
    cin = c0.numpy() if beta != 0.0 else None
    rows = _cases.sample_rows(M) if M * N * K > 2e9 else [(0, M)]
    for r0, r1 in rows:
        Y, D = oracle.gemm(mode, ops.a_host, ops.b_host, transA=tA, transB=tB, alpha=alpha, beta=beta, C=cin,
                           rows=(r0, r1))
        _check(mode, got[r0:r1], Y, D, act, bias, Z[r0:r1] if Z is not None else None, alpha, beta,
               cin[r0:r1] if cin is not None else None, f"{mode} {M}x{N}x{K} rows {r0}:{r1}")


@pytest.mark.parametrize("mode,opts", [("tf32", {"tile_n": 192}), ("bf16", {})])
@pytest.mark.parametrize("pad,offset", [(0, 0), (4, 0), (3, 0), (4, 1)])
def test_dgelu_z_layouts(h, mode, opts, pad, offset):
    """GELU' with Z a view into a wider buffer: rows padded by 4 (Z still
    read in 32 x 32 blocks by the epilogue's TMA loads, through a map whose
    row pitch is not N), by 3 (rows no longer 16-byte aligned: per-row loads
    instead) and shifted by one element (a misaligned start: per-row loads),
    on ragged M and N."""
    for k, v in opts.items():
        h.set_option(k, v)
    M, N, K = 700, 650, 300
    ops, _ = _cases.make(mode, M, N, K, False, True, seed=111, dist="normal")
    Zw = si.normal((M, N + pad + offset), 112).numpy()
    Z = Zw[:, offset:offset + N]
    Zd = torch.from_numpy(Zw).cuda()[:, offset:offset + N]
    assert Zd.stride(0) == N + pad + offset
    C = torch.full((M, N), float("nan"), device="cuda")
    h.run(ops.A, ops.B, C, mode=mode, transB=True, act="dgelu", aux=Zd)
    assert h.check_device() == 0
    assert h.plan()["epilogue_fused"] == 1
    Y, D = oracle.gemm(mode, ops.a_host, ops.b_host, transB=True)
    _check(mode, C.cpu().numpy(), Y, D, "dgelu", None, np.ascontiguousarray(Z), 1.0, 0.0, None,
           f"{mode} pad {pad} offset {offset}")


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


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
@pytest.mark.parametrize("act", ["gelu", "dgelu"])
def test_gelu_dense_sweep_against_oracle_and_cuda_erf(h, mode, act):
    """GELU and GELU' on 8192 x 64 exact inputs spanning [-8, 8] (a K = 1
    product a_i * b_j of values the mode holds exactly, so the GEMM adds no
    error), fused into the tensor-core kernel: against the oracle's fp64
    definition within the approximation's bound (|Phi error| <= 1.5e-7 plus
    fp32 rounding), and against CUDA's erf through torch's exact GELU within
    the same bound."""
    M, N = 8192, 64
    # a grid rounded to bf16 values (exact in both modes), b with 7 significant bits
    a = np.empty((M, 1), dtype=np.float32)  # fresh arrays: unit stride along the length-1 axis too
    a[:, 0] = si.to_bf16(torch.from_numpy((-8.0 + np.arange(M) / 512.0).astype(np.float32))).float().numpy()
    b = np.empty((1, N), dtype=np.float32)
    b[0, :] = 1.0 + np.arange(N) / 64.0
    A = torch.from_numpy(a)
    B = torch.from_numpy(b)
    if mode == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
        a_host, b_host = si.bf16_bits(A), si.bf16_bits(B)
    else:
        a_host, b_host = a, b
    Y, D = oracle.gemm(mode, a_host, b_host)
    assert np.array_equal(Y, np.float64(a) * np.float64(b))  # the inputs are exact in the mode
    C = torch.full((M, N), float("nan"), device="cuda")
    if act == "gelu":
        h.run(A.cuda(), B.cuda(), C, mode=mode, act="gelu")
        ref = oracle.epilogue("gelu", Y)
        cuda_ref = torch.nn.functional.gelu(torch.from_numpy(Y.astype(np.float32)).cuda(), approximate="none")
        scale = np.abs(Y)
    else:
        Z = torch.from_numpy(Y.astype(np.float32)).cuda()
        ones_a = torch.ones((M, 1), dtype=A.dtype)
        ones_b = torch.ones((1, N), dtype=B.dtype)
        h.run(ones_a.cuda(), ones_b.cuda(), C, mode=mode, act="dgelu", aux=Z)
        ref = oracle.epilogue("dgelu", np.ones((M, N)), None, Y.astype(np.float32))
        x = Z.double()
        cuda_ref = (0.5 * (1.0 + torch.erf(x / np.sqrt(2.0))) + x * torch.exp(-0.5 * x * x) / np.sqrt(2 * np.pi))
        scale = 1.0 + np.abs(Y)
    assert h.check_device() == 0
    assert h.plan()["epilogue_fused"] == 1
    got = C.cpu().numpy().astype(np.float64)
    bound = 4e-7 * scale + 1e-6 * np.abs(ref) + 1e-30
    assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) / bound))
    assert np.all(np.abs(got - cuda_ref.cpu().numpy()) <= bound + 1e-6 * np.abs(ref) + 2e-7 * scale)
