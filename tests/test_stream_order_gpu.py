"""Stream order across back-to-back calls.

Every kernel of the library is launched with programmatic dependent launch
and may start before the previous kernel in the stream has finished; each
must still read only what earlier kernels completed.  These tests chain
calls on one stream with no synchronisation between them, where each call
reads what the previous one wrote (its C as the next call's A, or through
beta), in every kernel family and with the extra kernels some plans launch
(operand transposes and re-packs, split-K reductions, stream-K fixups).
Every intermediate buffer starts as NaN, so a read that runs ahead of its
producer shows up as NaN or as a missing term.  Each stage is checked
against the oracle applied to the previous stage's device result.
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


def _rows(M):
    picks = sorted({0, 1, M // 3, M // 2, M - 130, M - 2})
    return [(r, min(r + 2, M)) for r in picks if 0 <= r < M]


def _operand(mode, shape, seed, std=1.0):
    x = si.normal(shape, seed, std=std)
    if mode == "bf16":
        x16 = si.to_bf16(x)
        return x16.cuda(), si.bf16_bits(x16)
    return x.cuda(), x.numpy()


@pytest.mark.parametrize("mode,M,dims,transB", [
    # FP32 SIMT: K-contiguous A transposed first, stream-K with fixups
    ("fp32", 1000, [300, 520, 260, 400], False),
    ("fp32", 1000, [300, 520, 260, 400], True),
    # TF32 tensor cores: MN-major W transposed first; pairs, tiles cut into K slices
    ("tf32", 2304, [1024, 2304, 1024, 2304], False),
    ("tf32", 700, [200, 600, 300], True),
    # TF32 small M: the cluster kernel, W re-packed K-major each call
    ("tf32", 8, [1536, 8960, 1536], False),
])
def test_chained_outputs_feed_the_next_call(h, mode, M, dims, transB):
    """X_{i+1} = X_i op(W_i), all calls enqueued back to back."""
    stream = torch.cuda.Stream()
    X0, x0 = _operand(mode, (M, dims[0]), si.seed_for(9, 0, 0))
    Ws, ws = [], []
    for i in range(len(dims) - 1):
        shape = (dims[i + 1], dims[i]) if transB else (dims[i], dims[i + 1])
        W, w = _operand(mode, shape, si.seed_for(9, 1, i), std=1.0 / np.sqrt(dims[i]))
        Ws.append(W)
        ws.append(w)
    Xs = [X0] + [torch.full((M, d), float("nan"), device="cuda") for d in dims[1:]]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i, W in enumerate(Ws):
            h.run(Xs[i], W, Xs[i + 1], mode=mode, transB=transB, stream=stream)
    assert h.check_device(stream) == 0
    prev = x0
    for i in range(len(Ws)):
        got = Xs[i + 1].cpu().numpy()
        assert not np.isnan(got).any(), f"stage {i}: NaN read ahead of its producer"
        for r0, r1 in _rows(M):
            ref, D = oracle.gemm(mode, prev, ws[i], transB=transB, rows=(r0, r1))
            _gate.assert_within(mode, got[r0:r1], ref, D, what=f"stage {i} rows {r0}:{r1}")
        prev = got


@pytest.mark.parametrize("mode,M,N,K,transB", [
    ("bf16", 2304, 2304, 1024, False),   # two-CTA MMA pairs
    ("bf16", 4096, 4096, 1024, True),    # tiles cut into K slices, slice reduction
    ("bf16", 16, 8960, 1536, False),     # small M: clusters of 4 K slices
    ("bf16", 4, 1536, 8960, True),       # small M: clusters of 16 K slices
    ("tf32", 300, 260, 1000, True),      # forced split-K below
    ("fp32", 130, 390, 20000, False),    # stream-K over deep K
])
def test_accumulation_through_beta(h, mode, M, N, K, transB):
    """C = A_i op(B_i) + 1 * C for several i, all enqueued back to back: each
    call reads the C the previous call wrote."""
    if mode == "tf32":
        h.set_option("split_k", 3)
    try:
        stream = torch.cuda.Stream()
        calls = 3
        As, Bs, a_h, b_h = [], [], [], []
        for i in range(calls):
            A, a = _operand(mode, (M, K), si.seed_for(10, 0, i))
            B, b = _operand(mode, (N, K) if transB else (K, N), si.seed_for(10, 1, i), std=0.05)
            As.append(A)
            Bs.append(B)
            a_h.append(a)
            b_h.append(b)
        c0 = si.normal((M, N), si.seed_for(10, 2, 0))
        C = c0.clone().cuda()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for A, B in zip(As, Bs):
                h.run(A, B, C, mode=mode, transB=transB, alpha=1.0, beta=1.0, stream=stream)
        assert h.check_device(stream) == 0
        got = C.cpu().numpy()
        for r0, r1 in _rows(M):
            ref = c0.numpy()[r0:r1].astype(np.float64)
            D = np.zeros_like(ref)
            for a, b in zip(a_h, b_h):
                r, d = oracle.gemm(mode, a, b, transB=transB, rows=(r0, r1))
                ref = ref + r
                D = D + d
            # each call's products within the gate, and each call's stored
            # result rounded once to fp32 (at most |c0| + D in magnitude);
            # a call that read C before the previous call wrote it would
            # drop a whole product
            rounding = calls * _gate.U32 * (np.abs(c0.numpy()[r0:r1]) + D)
            err = np.maximum(np.abs(got[r0:r1].astype(np.float64) - ref) - rounding, 0.0) / np.maximum(D, 1e-30)
            assert err.max() <= _gate.TOL[mode], (mode, r0, err.max())
    finally:
        h.set_option("split_k", 0)
