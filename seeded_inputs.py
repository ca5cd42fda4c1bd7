"""Seeded synthetic inputs and the workload shapes, shared by both sides.

This module only draws random numbers and names shapes.  It holds none of the
GEMM arithmetic: the library (``dense_gemm_transformer_gb300``) and the oracle
(``oracle``) both take their inputs from here and share nothing else.

Inputs are drawn on the CPU with ``torch.Generator`` so that every machine
produces the same tensors for the same seed.  The seed scheme is
``1234 + 1000 * config + 10 * shape + tensor_id`` (seed 1234 is the one the
"gpu kernels" write-up on devpost uses for its synthetic tensors, section
"Tools").

Workloads (every one stands in for data that is not available here):

* ``square256``: C = A B with M = N = K = 256, A and B uniform on [-1, 1];
  the same shape with integers in [-4, 4] for the exact check.
* GPT projections: the matmuls of a 6-layer, d_model = 384, 6-head character
  GPT at batch 64 x context 256 (16384 token rows), which "bare-metal-bard"
  (second paragraph) trains with its own kernels.  Weights W are stored
  K_in x N_out (so forward is NN, dX = dY W^T is NT and dW = X^T dY is TN),
  activations X and upstream gradients dY are N(0, 1), weights N(0, 0.02^2).
* the square sweep 1024 / 2048 / 4096, the large bf16 shapes, and the skinny
  decode shapes (1, 4 or 16 token rows against 1536 x 8960, 8960 x 1536 and
  1536 x 151936 weights: the hidden, MLP and vocabulary widths of the decode
  step on vidyal.ai's "One Token, Kernel by Kernel").
* attention: the GPT's causal self-attention, which "bare-metal-bard"
  (third paragraph) runs as one fused kernel -- 64 sequences x 6 heads of 64
  at context 256 -- and the same 16384 tokens per step at the longer
  contexts the page trains at (16 x 1024 and 8 x 2048 tokens, 6 heads); Q,
  K and V are N(0, 1) rounded to bf16, so that with the usual 1 / sqrt(64)
  scale the scores are N(0, 1).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

BASE_SEED = 1234
GPT_TOKENS = 64 * 256
# (name, K_in, N_out) of each projection of the d_model = 384 GPT; the
# vocabulary of the character model has 65 symbols.
GPT_PROJECTIONS = (
    ("qkv", 384, 1152),
    ("attn_out", 384, 384),
    ("mlp_up", 384, 1536),
    ("mlp_down", 1536, 384),
    ("lm_head", 384, 65),
)
SQUARE_SWEEP = (1024, 2048, 4096)
LARGE_BF16 = ((8192, 8192, 8192), (8192, 28672, 8192))
SKINNY_M = (1, 4, 16)
SKINNY_WEIGHTS = ((1536, 8960), (8960, 1536), (1536, 151936))  # K x N


ATTN_HEAD_DIM = 64
# (name, problems = sequences x heads, context T)
ATTN_WORKLOADS = (
    ("gpt_ctx256", 64 * 6, 256),
    ("ctx1024", 16 * 6, 1024),
    ("ctx2048", 8 * 6, 2048),
)


def seed_for(config: int, shape: int, tensor_id: int) -> int:
    return BASE_SEED + 1000 * config + 10 * shape + tensor_id


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def uniform(shape, seed, lo=-1.0, hi=1.0) -> torch.Tensor:
    """fp32 i.i.d. uniform on [lo, hi)."""
    u = torch.rand(tuple(shape), generator=_gen(seed), dtype=torch.float32)
    return u * (hi - lo) + lo


def normal(shape, seed, std=1.0) -> torch.Tensor:
    """fp32 i.i.d. N(0, std^2)."""
    return torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32) * std


def integers(shape, seed, lo=-4, hi=4) -> torch.Tensor:
    """fp32 holding i.i.d. integers drawn uniformly from [lo, hi]."""
    return torch.randint(lo, hi + 1, tuple(shape), generator=_gen(seed)).to(torch.float32)


def to_bf16(t: torch.Tensor) -> torch.Tensor:
    """Round fp32 to bfloat16 (torch's round-to-nearest-even) on the CPU."""
    return t.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """The uint16 bit patterns of a bfloat16 tensor, as a numpy array."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view("uint16")


FP8_E4M3_MAX = 448.0    # largest finite E4M3 magnitude
FP8_E5M2_MAX = 57344.0  # largest finite E5M2 magnitude


def to_fp8(t: torch.Tensor, fmt: str = "e4m3", amax_to: float = 0.0):
    """to_fp8_e4m3, or with fmt == "e5m2" the same into E5M2 codes."""
    if fmt == "e4m3":
        return to_fp8_e4m3(t, amax_to)
    s = 1.0
    if amax_to > 0.0:
        amax = float(t.abs().max())
        s = amax / amax_to if amax > 0.0 else 1.0
    q = (t / s).to(torch.float8_e5m2)
    return q.contiguous().view(torch.uint8).numpy(), s


def to_fp8_e4m3(t: torch.Tensor, amax_to: float = 0.0):
    """Quantise fp32 to 8-bit E4M3 codes (torch's round-to-nearest-even
    conversion on the CPU) with one scale for the whole tensor.

    amax_to == 0: no scaling, the values must already lie within +-448.
    amax_to > 0: the tensor is divided by s = max|t| / amax_to first, the way
    per-tensor FP8 recipes map a tensor's range onto the format's.
    Returns (codes as a uint8 numpy array, s); the product of two operands'
    s is the alpha that restores the unscaled product."""
    s = 1.0
    if amax_to > 0.0:
        amax = float(t.abs().max())
        s = amax / amax_to if amax > 0.0 else 1.0
    q = (t / s).to(torch.float8_e4m3fn)
    return q.contiguous().view(torch.uint8).numpy(), s


# Largest magnitudes of the block-scaled element formats and the exponent of
# each one's largest power of two (448 = 1.75 * 2^8, 57344 = 1.75 * 2^15,
# 6 = 1.5 * 2^2).
_ELEM_MAX = {"e4m3": (448.0, 8), "e5m2": (57344.0, 15), "e2m1": (6.0, 2)}
E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _e2m1_codes(x):
    """Round to the nearest E2M1 value (ties to the even code), saturating
    at +-6; returns 4-bit codes as uint8."""
    import numpy as np
    mags = np.array(E2M1_MAGNITUDES)
    a = np.minimum(np.abs(x), 6.0)
    d = np.abs(a[..., None] - mags)
    best = d.min(axis=-1, keepdims=True)
    tie = (d == best)
    # among equally near values take the even code (mantissa bit 0)
    even = tie & ((np.arange(8) % 2) == 0)
    idx = np.where(even.any(axis=-1), even.argmax(axis=-1), tie.argmax(axis=-1)).astype(np.uint8)
    return np.where(np.signbit(x) & (idx > 0), idx | 8, idx).astype(np.uint8)


def to_block_scaled(t: torch.Tensor, elem: str = "e4m3", block: int = 32, scale: str = "e8m0"):
    """Quantise a rows x K fp32 tensor to a block-scaled format: every run of
    `block` elements of a row gets one scale, chosen from the run's largest
    magnitude, and the elements are rounded to `elem` after division by it.

    E8M0 scales (MX): 2^(floor(log2 amax) - e), e the exponent of the
    element format's largest power of two, so the run's largest element lands
    in the format's top binade.  UE4M3 scales (NVFP4): amax / 6 rounded to
    E4M3, kept within [2^-9, 448].  An all-zero run takes the scale 1.  Returns (element codes as
    uint8 -- two E2M1 codes per byte, the even element in the low nibble --,
    scale codes as uint8 rows x ceil(K / block))."""
    import numpy as np
    x = t.to(torch.float64).numpy()
    rows, K = x.shape
    nb = -(-K // block)
    pad = np.zeros((rows, nb * block))
    pad[:, :K] = x
    amax = np.abs(pad.reshape(rows, nb, block)).max(axis=-1)
    emax_val, emax_exp = _ELEM_MAX[elem]
    if scale == "e8m0":
        e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - emax_exp, 0.0)
        e = np.clip(e, -127, 127)
        scodes = (e + 127).astype(np.uint8)
        sval = np.ldexp(1.0, e.astype(np.int64))
    else:
        # amax / 6 kept inside the positive E4M3 range, [2^-9, 448], before
        # the cast (which does not saturate): a run beyond 6 * 448 takes the
        # largest scale and its elements clip to +-6; a run so small that
        # amax / 6 is below the smallest subnormal takes the smallest scale.
        want = np.where(amax > 0, np.clip(amax / 6.0, 2.0 ** -9, 448.0), 1.0)
        want = torch.from_numpy(want).to(torch.float8_e4m3fn)
        scodes = want.view(torch.uint8).numpy().copy()
        sval = want.to(torch.float64).numpy()
    y = pad / np.repeat(sval, block, axis=1)
    y = np.clip(y, -emax_val, emax_val)[:, :K]
    if elem == "e2m1":
        if K % 2:
            raise ValueError("E2M1 rows need an even K (two codes per byte)")
        c = _e2m1_codes(y)
        codes = (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    else:
        dt = torch.float8_e4m3fn if elem == "e4m3" else torch.float8_e5m2
        codes = torch.from_numpy(y).to(dt).view(torch.uint8).numpy().copy()
    return codes, scodes.astype(np.uint8)


@dataclass(frozen=True)
class GemmCase:
    """One GEMM of a workload: C (M x N) = alpha op(A) op(B) + beta C."""
    name: str
    transA: bool
    transB: bool
    M: int
    N: int
    K: int

    @property
    def a_shape(self):
        return (self.K, self.M) if self.transA else (self.M, self.K)

    @property
    def b_shape(self):
        return (self.N, self.K) if self.transB else (self.K, self.N)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def gpt_cases():
    """The 15 GEMMs of one GPT training step's projections (forward, dX, dW)."""
    out = []
    T = GPT_TOKENS
    for name, kin, nout in GPT_PROJECTIONS:
        out.append(GemmCase(f"{name}.fwd", False, False, T, nout, kin))   # Y  = X W
        out.append(GemmCase(f"{name}.dX", False, True, T, kin, nout))     # dX = dY W^T
        out.append(GemmCase(f"{name}.dW", True, False, kin, nout, T))     # dW = X^T dY
    return out


def gpt_tensors(shape_index: int, kin: int, nout: int, config: int = 1):
    """X (T x K_in), W (K_in x N_out), dY (T x N_out) for one projection."""
    T = GPT_TOKENS
    X = normal((T, kin), seed_for(config, shape_index, 0))
    W = normal((kin, nout), seed_for(config, shape_index, 1), std=0.02)
    dY = normal((T, nout), seed_for(config, shape_index, 2))
    return X, W, dY


def square_case(n: int) -> GemmCase:
    return GemmCase(f"square{n}", False, False, n, n, n)


def skinny_cases():
    out = []
    for m in SKINNY_M:
        for k, n in SKINNY_WEIGHTS:
            out.append(GemmCase(f"skinny_m{m}_{k}x{n}", False, False, m, n, k))
    return out


def attention_qkv(problems: int, T: int, shape: int = 0, config: int = 1, std_q: float = 1.0):
    """Q, K, V: bf16 CPU tensors of [problems, T, 64], N(0, 1) (Q: N(0, std_q^2),
    a larger std_q makes the softmax peaked)."""
    D = ATTN_HEAD_DIM
    Q = to_bf16(normal((problems, T, D), seed_for(config, shape, 0), std=std_q))
    K = to_bf16(normal((problems, T, D), seed_for(config, shape, 1)))
    V = to_bf16(normal((problems, T, D), seed_for(config, shape, 2)))
    return Q, K, V
