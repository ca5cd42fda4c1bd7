"""Helpers for the GPU parity tests: seeded operands for a mode, one call of
the library on the device, and the oracle's answer for the same inputs."""
import numpy as np
import torch

import dense_gemm_transformer_gb300 as dg
import oracle
import seeded_inputs as si
from tests import _gate


class Operands:
    """Host copies (for the oracle) and device copies (for the library)."""

    def __init__(self, mode, a32, b32):
        self.mode = mode
        if mode == "bf16":
            a16, b16 = si.to_bf16(a32), si.to_bf16(b32)
            self.a_host, self.b_host = si.bf16_bits(a16), si.bf16_bits(b16)
            self.A, self.B = a16.cuda(), b16.cuda()
        else:
            self.a_host, self.b_host = a32.numpy(), b32.numpy()
            self.A, self.B = a32.cuda(), b32.cuda()


def make(mode, M, N, K, transA=False, transB=False, seed=100, dist="uniform", with_c=False):
    a_shape = (K, M) if transA else (M, K)
    b_shape = (N, K) if transB else (K, N)
    if dist == "uniform":
        a32, b32 = si.uniform(a_shape, seed), si.uniform(b_shape, seed + 1)
    elif dist == "normal":
        a32, b32 = si.normal(a_shape, seed), si.normal(b_shape, seed + 1)
    elif dist == "int":
        a32, b32 = si.integers(a_shape, seed), si.integers(b_shape, seed + 1)
    else:
        raise ValueError(dist)
    ops = Operands(mode, a32, b32)
    c0 = si.normal((M, N), seed + 2) if with_c else None
    return ops, c0


def run_and_check(h, mode, M, N, K, transA=False, transB=False, alpha=1.0, beta=0.0, seed=100,
                  dist="uniform", rows=None, exact=False):
    """Run the library once and compare with the oracle; returns max err."""
    ops, c0 = make(mode, M, N, K, transA, transB, seed, dist, with_c=beta != 0.0)
    C = c0.clone().cuda() if c0 is not None else torch.full((M, N), float("nan"), device="cuda")
    h.run(ops.A, ops.B, C, mode=mode, transA=transA, transB=transB, alpha=alpha, beta=beta)
    assert h.check_device() == 0
    got = C.cpu().numpy()
    cin = c0.numpy() if c0 is not None else None
    if rows is None:
        ref, D = oracle.gemm(mode, ops.a_host, ops.b_host, transA=transA, transB=transB, alpha=alpha, beta=beta,
                             C=cin)
        g, ci = got, cin
    else:
        refs, Ds, gs, cs = [], [], [], []
        for r0, r1 in rows:
            r, d = oracle.gemm(mode, ops.a_host, ops.b_host, transA=transA, transB=transB, alpha=alpha, beta=beta,
                               C=cin, rows=(r0, r1))
            refs.append(r)
            Ds.append(d)
            gs.append(got[r0:r1])
            if cin is not None:
                cs.append(cin[r0:r1])
        ref, D, g = np.concatenate(refs), np.concatenate(Ds), np.concatenate(gs)
        ci = np.concatenate(cs) if cs else None
    if exact:
        assert np.array_equal(g.astype(np.float64), ref), f"{mode} not bit-exact"
        return 0.0
    return _gate.assert_within(mode, g, ref, D, alpha, beta, ci, what=f"{M}x{N}x{K} tA={transA} tB={transB}")


def sample_rows(M, tile=128, width=2):
    """Row ranges at the start, the end, and around tile boundaries."""
    picks = {0, M - width, M // 2}
    for t in (tile, 2 * tile, M - (M % tile or tile)):
        picks.add(t - 1)
    out = []
    for r in sorted(p for p in picks if 0 <= p < M):
        out.append((r, min(r + width, M)))
    merged = []
    for r0, r1 in out:
        if merged and r0 <= merged[-1][1]:
            merged[-1] = (merged[-1][0], max(merged[-1][1], r1))
        else:
            merged.append((r0, r1))
    return merged
