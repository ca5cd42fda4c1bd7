"""The fused attention forward (gemm_attention_forward) against the oracle:
causal and full attention over one or many 128-query tiles and 128-key
blocks, ragged tails of both, a single token, peaked softmaxes whose running
maximum moves from block to block, other scales, the GPT's own size (batch 64
x 6 heads at context 256) and the long contexts (1024 and 2048 tokens) on
sampled problems, and the argument checks.

Gate, per element: |O - Oref| <= TOL * W + 4e-6 * |Oref|, W = sum_j p_j |v_j|
/ l the oracle's error scale.  The kernel rounds each probability to bf16
for the P V product (relative error at most 2^-8 per weight, so at most
2^-8 W on O); TOL = 8e-3 leaves twice that.  The scores themselves (exact
bf16 products summed in fp32) and the base-2 exponential add far less."""
import numpy as np
import pytest
import torch

import dense_gemm_transformer_gb300 as dg
import oracle
import seeded_inputs as si

pytestmark = pytest.mark.gpu

TOL = 8e-3
D = si.ATTN_HEAD_DIM


@pytest.fixture(scope="module")
def h():
    dg.load(build_if_missing=True)
    handle = dg.Gemm()
    yield handle
    handle.close()


def _run(h, Q, K, V, causal, scale=None, guard=0):
    """O from the library, in a buffer with `guard` sentinel floats after it."""
    dev = torch.device("cuda", 0)
    Qd, Kd, Vd = (t.to(dev).contiguous() for t in (Q, K, V))
    n = Q.numel()
    buf = torch.full((n + guard,), 12345.0, dtype=torch.float32, device=dev)
    O = buf[:n].view(Q.shape)
    h.attention(Qd, Kd, Vd, O, causal=causal, scale=scale)
    torch.cuda.synchronize()
    tail = buf[n:].cpu()
    assert torch.all(tail == 12345.0), "the kernel wrote past O"
    return O.cpu().numpy().astype(np.float64)


def _check(got, Q, K, V, causal, scale=None, problems=None, what=""):
    ref, W = oracle.attention(si.bf16_bits(Q), si.bf16_bits(K), si.bf16_bits(V), causal=causal, scale=scale,
                              problems=problems)
    p0, p1 = problems if problems is not None else (0, Q.shape[0])
    g = got[p0:p1]
    assert np.all(np.isfinite(g)), what
    err = np.abs(g - ref)
    bound = TOL * W + 4e-6 * np.abs(ref) + 1e-30
    assert np.all(err <= bound), (what, float(np.max(err / bound)))


CASES = [
    # problems, T, causal, std_q  (what each exercises)
    (3, 200, True, 1.0),    # two query tiles, ragged tail of rows and keys
    (2, 128, True, 1.0),    # exactly one tile and one key block
    (2, 1, True, 1.0),      # a single token
    (2, 1, False, 1.0),
    (2, 129, True, 1.0),    # one row past a tile
    (2, 129, False, 1.0),
    (2, 300, False, 1.0),   # full attention, three key blocks with a ragged last one
    (2, 384, True, 4.0),    # peaked: the running maximum moves between blocks
    (2, 640, False, 6.0),   # peaked, full, five key blocks
    (5, 1000, True, 1.0),   # eight query tiles, ragged
]


@pytest.mark.parametrize("P,T,causal,std_q", CASES)
def test_attention_matches_oracle(h, P, T, causal, std_q):
    Q, K, V = si.attention_qkv(P, T, shape=T % 97, std_q=std_q)
    got = _run(h, Q, K, V, causal, guard=4096)
    _check(got, Q, K, V, causal, what=f"P={P} T={T} causal={causal}")
    assert h.plan()["family"] == "attention"
    assert h.check_device() == 0


@pytest.mark.parametrize("scale", [0.0, 0.3, -0.125, 2.0])
def test_attention_other_scales(h, scale):
    Q, K, V = si.attention_qkv(2, 260, shape=3)
    got = _run(h, Q, K, V, True, scale=scale)
    _check(got, Q, K, V, True, scale=scale, what=f"scale={scale}")


def test_attention_gpt_size_sampled(h):
    """The GPT's attention at full size in the launch the bench times:
    64 sequences x 6 heads at context 256; the first and last 16 problems
    against the oracle, every output finite."""
    name, P, T = si.ATTN_WORKLOADS[0]
    Q, K, V = si.attention_qkv(P, T, shape=0)
    got = _run(h, Q, K, V, True)
    assert np.all(np.isfinite(got))
    _check(got, Q, K, V, True, problems=(0, 16), what=name)
    _check(got, Q, K, V, True, problems=(P - 16, P), what=name)


@pytest.mark.parametrize("causal", [True, False])
def test_attention_many_items_per_cta(h, causal):
    """Far more (problem, query tile) items than CTAs, so that every CTA of
    the persistent grid runs several in turn (Q buffers and the output
    accumulator handed from one item to the next); ragged T; sampled."""
    P, T = 700, 200
    Q, K, V = si.attention_qkv(P, T, shape=7, std_q=2.0)
    got = _run(h, Q, K, V, causal, guard=1024)
    assert h.plan()["grid"] < P * 2
    assert np.all(np.isfinite(got))
    _check(got, Q, K, V, causal, problems=(0, 12), what="first")
    _check(got, Q, K, V, causal, problems=(343, 351), what="middle")
    _check(got, Q, K, V, causal, problems=(P - 12, P), what="last")


@pytest.mark.parametrize("idx", [1, 2])
def test_attention_long_context_sampled(h, idx):
    """Context 1024 and 2048 at full size; the first and last problems against the oracle."""
    name, P, T = si.ATTN_WORKLOADS[idx]
    Q, K, V = si.attention_qkv(P, T, shape=idx)
    got = _run(h, Q, K, V, True)
    assert np.all(np.isfinite(got))
    _check(got, Q, K, V, True, problems=(0, 1), what=name)
    _check(got, Q, K, V, True, problems=(P - 1, P), what=name)


@pytest.mark.parametrize("offset", [4, 8])
def test_attention_output_only_16_byte_aligned(h, offset):
    """O at 16 (not 32) bytes past an allocation: the kernel stores 16 bytes
    at a time there; the floats around O stay untouched."""
    P, T = 3, 300
    Q, K, V = si.attention_qkv(P, T, shape=11)
    dev = torch.device("cuda", 0)
    n = Q.numel()
    buf = torch.full((n + 2 * offset + 64,), 12345.0, dtype=torch.float32, device=dev)
    O = buf[offset:offset + n].view(Q.shape)
    assert O.data_ptr() % 32 == 16 if offset == 4 else O.data_ptr() % 32 == 0
    h.attention(Q.to(dev), K.to(dev), V.to(dev), O, causal=True)
    torch.cuda.synchronize()
    out = buf.cpu()
    assert torch.all(out[:offset] == 12345.0) and torch.all(out[offset + n:] == 12345.0)
    _check(O.cpu().numpy().astype(np.float64), Q, K, V, True, what=f"offset {offset}")


def test_attention_row_sums_of_constant_values(h):
    """V constant c: every output is c whatever the weights (the weights sum to one)."""
    Q, K, _ = si.attention_qkv(2, 333, shape=5, std_q=3.0)
    V = torch.full_like(Q, 0.75)
    got = _run(h, Q, K, V, True)
    assert np.max(np.abs(got - 0.75)) <= TOL * 0.75


def test_attention_argument_checks(h):
    dev = torch.device("cuda", 0)
    Q = torch.zeros((2, 64, 64), dtype=torch.bfloat16, device=dev)
    O = torch.zeros((2, 64, 64), dtype=torch.float32, device=dev)
    p = Q.data_ptr()
    with pytest.raises(dg.GemmError, match="NOT_SUPPORTED"):
        h.attention_ptr(2, 64, 32, 1, 0.125, p, p, p, O.data_ptr())
    with pytest.raises(dg.GemmError, match="INVALID_VALUE"):
        h.attention_ptr(2, 64, 64, 2, 0.125, p, p, p, O.data_ptr())
    with pytest.raises(dg.GemmError, match="INVALID_VALUE"):
        h.attention_ptr(2, 64, 64, 1, float("nan"), p, p, p, O.data_ptr())
    with pytest.raises(dg.GemmError, match="INVALID_VALUE"):
        h.attention_ptr(-1, 64, 64, 1, 0.125, p, p, p, O.data_ptr())
    with pytest.raises(dg.GemmError, match="INVALID_VALUE"):
        h.attention_ptr(2, 64, 64, 1, 0.125, p, 0, p, O.data_ptr())
    with pytest.raises(dg.GemmError, match="MISALIGNED"):
        h.attention_ptr(1, 64, 64, 1, 0.125, p + 8, p, p, O.data_ptr())
    with pytest.raises(dg.GemmError, match="MISALIGNED"):
        h.attention_ptr(1, 64, 64, 1, 0.125, p, p, p, O.data_ptr() + 4)
    # empty problems are no-ops that touch nothing
    O.fill_(7.0)
    h.attention_ptr(0, 64, 64, 1, 0.125, p, p, p, O.data_ptr())
    h.attention_ptr(2, 0, 64, 1, 0.125, p, p, p, O.data_ptr())
    torch.cuda.synchronize()
    assert torch.all(O == 7.0)
    assert h.check_device() == 0
