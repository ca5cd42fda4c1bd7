"""The GPT projection step captured as one CUDA graph and replayed: one
layer's QKV, attention-out, MLP-up and MLP-down projections plus the LM head
at 16384 token rows, each forward, dX and dW (15 GEMMs, the step's every
shape), in TF32 and BF16.  The graph must recompute every output on each
replay (outputs are poisoned with NaN between replays) and match the oracle
on sampled rows, and its replay must equal the same calls issued eagerly.
"""
import pytest
import torch

import dense_gemm_transformer_gb300 as dg
import oracle
import seeded_inputs as si
from tests import _cases, _gate

pytestmark = pytest.mark.gpu


def _step(mode):
    calls = []
    for p, (name, kin, nout) in enumerate(si.GPT_PROJECTIONS):
        X, W, dY = si.gpt_tensors(p, kin, nout)
        if mode == "bf16":
            X, W, dY = si.to_bf16(X), si.to_bf16(W), si.to_bf16(dY)
        Xd, Wd, dYd = X.cuda(), W.cuda(), dY.cuda()
        T = si.GPT_TOKENS
        for tag, Ad, Bd, Ah, Bh, tA, tB, M, N in (("fwd", Xd, Wd, X, W, False, False, T, nout),
                                                  ("dX", dYd, Wd, dY, W, False, True, T, kin),
                                                  ("dW", Xd, dYd, X, dY, True, False, kin, nout)):
            calls.append((f"{name}.{tag}", Ad, Bd, Ah, Bh, tA, tB, torch.empty((M, N), device="cuda")))
    return calls


def _host(mode, t):
    return si.bf16_bits(t) if mode == "bf16" else t.numpy()


@pytest.mark.parametrize("mode", ["tf32", "bf16"])
def test_step_as_one_graph(mode):
    dg.load(build_if_missing=True)
    h = dg.Gemm()
    stream = torch.cuda.Stream()
    calls = _step(mode)

    def step():
        for _, A, B, _, _, tA, tB, C in calls:
            h.run(A, B, C, mode=mode, transA=tA, transB=tB, stream=stream)

    with torch.cuda.stream(stream):
        step()  # eager: grows the workspace to its final size before capture
    stream.synchronize()
    assert h.check_device(stream) == 0
    eager = [C.clone() for *_, C in calls]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for _ in range(2):
        for *_, C in calls:
            C.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        for (name, *_), C, E in zip(calls, (c[-1] for c in calls), eager):
            assert torch.equal(C, E), f"{name}: graph replay differs from the eager call"
    assert h.check_device(stream) == 0
    for name, _, _, Ah, Bh, tA, tB, C in calls:
        got = C.cpu().numpy()
        M = got.shape[0]
        for r0, r1 in _cases.sample_rows(M, width=1):
            ref, D = oracle.gemm(mode, _host(mode, Ah), _host(mode, Bh), transA=tA, transB=tB, rows=(r0, r1))
            _gate.assert_within(mode, got[r0:r1], ref, D, what=f"graph {mode} {name} rows {r0}:{r1}")
    del graph
    h.close()
