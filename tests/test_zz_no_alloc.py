"""gemm_run_small_m_noalloc: the small-M product for callers that cannot
allocate device memory (a runtime that hands out all memory from its own
pool, a plug-in living inside someone else's CUDA context).  It must give
the same C as gemm_run, within the parity tolerance, on consecutive calls
that share the library's fixed scratch array, in both of its modes, and
refuse what it cannot serve without touching C.  Its companion
gemm_noalloc_check_device reads the array's status word.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_gemm_transformer_gb300 as dg
import oracle
import seeded_inputs as si
from tests import _gate

pytestmark = pytest.mark.gpu

NOT_SUPPORTED, MISALIGNED, TOO_LARGE = 2, 3, 7


def _noalloc_fn():
    lib = dg.load(build_if_missing=True)
    fn = lib.gemm_run_small_m_noalloc
    i64, vp, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
    fn.argtypes = [i32, i32, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
    fn.restype = i32
    return fn


def _check_fn():
    fn = dg.load(build_if_missing=True).gemm_noalloc_check_device
    fn.argtypes = [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _case(mode, M, N, K, transB, seed, dist="normal"):
    if dist == "int":
        a = si.integers((M, K), seed)
        b = si.integers((N, K) if transB else (K, N), seed + 1)
    else:
        a = si.normal((M, K), seed)
        b = si.normal((N, K) if transB else (K, N), seed + 1, std=0.02)
    c0 = si.normal((M, N), seed + 2)
    if mode == "bf16":
        a16, b16 = si.to_bf16(a), si.to_bf16(b)
        return a16.cuda(), b16.cuda(), si.bf16_bits(a16), si.bf16_bits(b16), c0
    return a.cuda(), b.cuda(), a.numpy(), b.numpy(), c0


def _call(fn, mode, tB, M, N, K, alpha, A, B, beta, C, stream):
    return fn(dg.MODES[mode], int(tB), M, N, K, alpha, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), beta,
              C.data_ptr(), C.stride(0), stream.cuda_stream)


# Every case splits K, so consecutive calls keep partial sums in the shared
# array: BF16 with weights K x N and N x K, and TF32 (weights N x K, the
# layout kind::tf32 reads in place).
CASES = [("bf16", 4, 1536, 8960, False, 0.5, 1.0, 501), ("bf16", 16, 8960, 1536, True, 1.0, 0.0, 511),
         ("tf32", 16, 1536, 8960, True, 1.0, 0.0, 521), ("tf32", 3, 1000, 4000, True, 0.5, 1.0, 531)]


def test_noalloc_matches_gemm_run_on_consecutive_calls():
    fn, check = _noalloc_fn(), _check_fn()
    h = dg.Gemm()
    stream = torch.cuda.current_stream()
    for mode, M, N, K, tB, alpha, beta, seed in CASES:
        A, B, a_h, b_h, c0 = _case(mode, M, N, K, tB, seed)
        C_ref = c0.clone().cuda()
        h.run(A, B, C_ref, mode=mode, transB=tB, alpha=alpha, beta=beta)
        C = c0.clone().cuda()
        st = _call(fn, mode, tB, M, N, K, alpha, A, B, beta, C, stream)
        assert st == 0, dg.status_string(st)
        assert check(stream.cuda_stream) == 0
        got, want = C.cpu().numpy(), C_ref.cpu().numpy()
        cin = c0.numpy() if beta else None
        ref, D = oracle.gemm(mode, a_h, b_h, transB=tB, alpha=alpha, beta=beta, C=cin)
        _gate.assert_within(mode, got, want, D, alpha, beta, cin, what=f"noalloc vs gemm_run {mode} M={M} N={N} K={K}")
        _gate.assert_within(mode, got, ref, D, alpha, beta, cin, what=f"noalloc vs oracle {mode} M={M} N={N} K={K}")
    h.close()


@pytest.mark.parametrize("mode,K", [("bf16", 8960), ("tf32", 8960)])
def test_noalloc_integers_bit_exact(mode, K):
    """Small integers with K split across slices: every partial sum is an
    integer below 2^24, so the result is exact whatever the slice count."""
    fn, check = _noalloc_fn(), _check_fn()
    stream = torch.cuda.current_stream()
    M, N = 16, 1536
    A, B, a_h, b_h, _ = _case(mode, M, N, K, True, 541, dist="int")
    C = torch.full((M, N), float("nan"), device="cuda")
    assert _call(fn, mode, True, M, N, K, 1.0, A, B, 0.0, C, stream) == 0
    assert check(stream.cuda_stream) == 0
    ref, _ = oracle.gemm(mode, a_h, b_h, transB=True)
    assert np.array_equal(C.cpu().numpy().astype(np.float64), ref)


def test_noalloc_rejects_what_it_cannot_serve():
    fn = _noalloc_fn()
    stream = torch.cuda.current_stream()
    # M > 16
    C = torch.full((17, 64), 5.0, device="cuda")
    A = torch.zeros((17, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    st = _call(fn, "bf16", False, 17, 64, 64, 1.0, A, B, 0.0, C, stream)
    assert st == TOO_LARGE and dg.status_string(st) == "GEMM_ERR_TOO_LARGE"
    # a weight row pitch the TMA unit cannot read in place (65 bf16 = 130 bytes)
    C = torch.full((4, 64), 5.0, device="cuda")
    A = torch.ones((4, 64), dtype=torch.bfloat16, device="cuda")
    Bwide = torch.ones((64, 65), dtype=torch.bfloat16, device="cuda")
    B = Bwide[:, :64]
    st = fn(dg.MODES["bf16"], 0, 4, 64, 64, 1.0, A.data_ptr(), 64, B.data_ptr(), 65, 0.0, C.data_ptr(), 64,
            stream.cuda_stream)
    assert st == MISALIGNED, dg.status_string(st)
    # TF32 weights stored K x N: kind::tf32 reads K-major operands only
    A32 = torch.ones((4, 64), device="cuda")
    B32 = torch.ones((64, 64), device="cuda")
    st = _call(fn, "tf32", False, 4, 64, 64, 1.0, A32, B32, 0.0, C, stream)
    assert st == NOT_SUPPORTED, dg.status_string(st)
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), torch.full((4, 64), 5.0))
