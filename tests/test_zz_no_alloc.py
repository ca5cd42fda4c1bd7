"""gemm_run_small_m_noalloc: the small-M product for callers that cannot
allocate device memory (a runtime that hands out all memory from its own
pool, a plug-in living inside someone else's CUDA context).  It must give
the same C as gemm_run, within the parity tolerance, on consecutive calls
that share the library's fixed scratch array.

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

TOO_LARGE = 7


def _noalloc_fn():
    fn = dg.load(build_if_missing=True).gemm_run_small_m_noalloc
    i64, vp, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
    fn.argtypes = [i32, i32, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
    fn.restype = i32
    return fn


def _case(M, N, K, transB, seed):
    a = si.normal((M, K), seed)
    b = si.normal((N, K) if transB else (K, N), seed + 1, std=0.02)
    c0 = si.normal((M, N), seed + 2)
    return si.to_bf16(a), si.to_bf16(b), c0


def test_noalloc_matches_gemm_run_on_consecutive_calls():
    fn = _noalloc_fn()
    h = dg.Gemm()
    stream = torch.cuda.current_stream()
    # Both shapes split K, so both calls keep partial sums in the shared array.
    cases = [(4, 1536, 8960, False, 0.5, 1.0, 501), (16, 8960, 1536, True, 1.0, 0.0, 511)]
    for M, N, K, tB, alpha, beta, seed in cases:
        a16, b16, c0 = _case(M, N, K, tB, seed)
        A, B = a16.cuda(), b16.cuda()
        C_ref = c0.clone().cuda()
        h.run(A, B, C_ref, mode="bf16", transB=tB, alpha=alpha, beta=beta)
        assert h.plan()["split_k"] > 1
        C = c0.clone().cuda()
        st = fn(2, int(tB), M, N, K, alpha, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), beta,
                C.data_ptr(), C.stride(0), stream.cuda_stream)
        assert st == 0, dg.status_string(st)
        torch.cuda.synchronize()
        got, want = C.cpu().numpy(), C_ref.cpu().numpy()
        _, D = oracle.gemm("bf16", si.bf16_bits(a16), si.bf16_bits(b16), transB=tB)
        _gate.assert_within("bf16", got, want, D, alpha, beta, c0.numpy() if beta else None,
                            what=f"noalloc vs gemm_run M={M} N={N} K={K}")
        ref, _ = oracle.gemm("bf16", si.bf16_bits(a16), si.bf16_bits(b16), transB=tB, alpha=alpha, beta=beta,
                             C=c0.numpy() if beta else None)
        _gate.assert_within("bf16", got, ref, D, alpha, beta, c0.numpy() if beta else None,
                            what=f"noalloc vs oracle M={M} N={N} K={K}")
    h.close()


def test_noalloc_rejects_what_exceeds_its_limits():
    fn = _noalloc_fn()
    C = torch.full((17, 64), 5.0, device="cuda")
    A = torch.zeros((17, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    st = fn(2, 0, 17, 64, 64, 1.0, A.data_ptr(), 64, B.data_ptr(), 64, 0.0, C.data_ptr(), 64, None)
    assert st == TOO_LARGE and dg.status_string(st) == "GEMM_ERR_TOO_LARGE"
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), torch.full((17, 64), 5.0))
