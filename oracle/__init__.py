"""CPU oracle for dense GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library
(``dense_gemm_transformer_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle_gemm.c`` (plain C, fp64, a triple loop with k
ascending); this module only marshals numpy arrays into it.  It computes the
textbook matmul of "bare-metal-bard", first paragraph (the one-thread-per-output
kernel), with BLAS scaling:

    Cref = alpha * op(A) @ op(B) + beta * Cin,   D = |op(A)| @ |op(B)|

with the operands first reduced to the mode's precision (FP32: unchanged,
TF32: reduced to 10 mantissa bits, BF16: bfloat16 inputs widened exactly,
FP8: E4M3 / E5M2 codes decoded exactly, each operand in its mode's format).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

MODES = {"fp32": 0, "tf32": 1, "bf16": 2, "fp8": 3, "fp8_e4m3": 3, "fp8_e5m2": 4, "fp8_e4m3_e5m2": 5,
         "fp8_e5m2_e4m3": 6}
_OPERAND_DTYPE = {"fp32": np.float32, "tf32": np.float32, "bf16": np.uint16}
TF32_RULES = {"truncate": 0, "nearest_away": 1}
# The reading taken for how the tensor cores treat raw fp32 operands in
# kind::tf32: the 13 low mantissa bits are dropped.  A GPU test checks this
# reading against the hardware on a one-column probe.
DEFAULT_TF32_RULE = "truncate"

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, p, d = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    i64, i64, i64, d, p, i64, p, i64, d, p, i64,
                                    i64, i64, p, p, i64]
        lib.oracle_tf32_array.restype = None
        lib.oracle_tf32_array.argtypes = [ctypes.c_int, p, p, i64]
        lib.oracle_bf16_array.restype = None
        lib.oracle_bf16_array.argtypes = [p, p, i64]
        lib.oracle_e4m3_array.restype = None
        lib.oracle_e4m3_array.argtypes = [p, p, i64]
        lib.oracle_e5m2_array.restype = None
        lib.oracle_e5m2_array.argtypes = [p, p, i64]
        for name in ("oracle_e2m1_array", "oracle_e8m0_array", "oracle_ue4m3_array"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = [p, p, i64]
        lib.oracle_gemm_block_scaled.restype = ctypes.c_int
        lib.oracle_gemm_block_scaled.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, i64, i64, i64, i64, d,
                                                 p, i64, p, i64, p, i64, p, i64, d, p, i64, i64, i64, p, p, i64]
        lib.oracle_gelu.restype = d
        lib.oracle_gelu.argtypes = [d]
        lib.oracle_dgelu.restype = d
        lib.oracle_dgelu.argtypes = [d]
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_attention.argtypes = [i64, i64, i64, ctypes.c_int, d, p, p, p, i64, i64, p, p]
        lib.oracle_epilogue.restype = ctypes.c_int
        lib.oracle_epilogue.argtypes = [ctypes.c_int, i64, i64, p, i64, p, p, i64, p, i64]
        _lib = lib
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _operand(x, mode):
    want = _OPERAND_DTYPE.get(mode, np.uint8)  # the FP8 modes take 8-bit codes
    x = np.asarray(x)
    if x.dtype != want:
        raise TypeError(f"mode {mode} takes {want.__name__} operands, got {x.dtype}")
    if x.ndim != 2:
        raise ValueError("operands must be 2-D")
    if x.size == 0:
        return np.ascontiguousarray(x)
    if x.strides[1] != x.itemsize:
        raise ValueError("operands need unit stride in the last dimension")
    return x


def gemm(mode, A, B, *, transA=False, transB=False, alpha=1.0, beta=0.0, C=None,
         rows=None, tf32_rule=DEFAULT_TF32_RULE):
    """Return (Cref, D) as float64 arrays of shape (rows, N).

    A, B: 2-D numpy arrays, float32 for fp32/tf32, uint16 bfloat16 bit patterns
    for bf16, uint8 codes for the fp8 modes ("fp8" = "fp8_e4m3", "fp8_e5m2",
    "fp8_e4m3_e5m2": A E4M3 and B E5M2, "fp8_e5m2_e4m3"), stored as described for gemm_run
    (row-major, op() by trans flag).
    C: float32 M x N input, read only when beta != 0.
    rows: (row0, row1) to compute only part of the output.
    """
    lib = _load()
    A = _operand(A, mode)
    B = _operand(B, mode)
    M, K = (A.shape[1], A.shape[0]) if transA else A.shape
    Kb, N = (B.shape[1], B.shape[0]) if transB else B.shape
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    row0, row1 = rows if rows is not None else (0, M)
    if beta != 0.0:
        if C is None:
            raise ValueError("beta != 0 needs C")
        C = np.asarray(C)
        if C.dtype != np.float32 or C.shape != (M, N) or C.strides[1] != 4:
            raise ValueError("C must be float32 M x N with unit column stride")
        ldc = C.strides[0] // 4
    else:
        C, ldc = None, max(N, 1)
    out = np.zeros((row1 - row0, N), dtype=np.float64)
    D = np.zeros((row1 - row0, N), dtype=np.float64)
    rc = lib.oracle_gemm(MODES[mode], TF32_RULES[tf32_rule], int(bool(transA)), int(bool(transB)),
                         M, N, K, float(alpha), _ptr(A), A.strides[0] // A.itemsize,
                         _ptr(B), B.strides[0] // B.itemsize, float(beta), _ptr(C), ldc,
                         row0, row1, _ptr(out), _ptr(D), max(N, 1))
    if rc != 0:
        raise ValueError(f"oracle_gemm rejected its arguments ({rc})")
    return out, D


def tf32(x, rule=DEFAULT_TF32_RULE):
    """Reduce float32 values to TF32 by the given rule (elementwise)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    lib.oracle_tf32_array(TF32_RULES[rule], _ptr(x), _ptr(out), x.size)
    return out


def bf16_to_f64(bits):
    """Widen bfloat16 bit patterns (uint16) to float64 exactly."""
    lib = _load()
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib.oracle_bf16_array(_ptr(bits), _ptr(out), bits.size)
    return out


def e5m2_to_f64(codes):
    """Decode 8-bit E5M2 codes (uint8) to float64 exactly (+-Inf, NaN as in IEEE 754)."""
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    lib.oracle_e5m2_array(_ptr(codes), _ptr(out), codes.size)
    return out


def e4m3_to_f64(codes):
    """Decode 8-bit E4M3 codes (uint8) to float64 exactly (NaN for S.1111.111)."""
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    lib.oracle_e4m3_array(_ptr(codes), _ptr(out), codes.size)
    return out


def _decode(fn_name, codes):
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    getattr(lib, fn_name)(_ptr(codes), _ptr(out), codes.size)
    return out


def e2m1_to_f64(codes):
    """Decode 4-bit E2M1 codes (uint8 values 0..15, one per byte) exactly."""
    return _decode("oracle_e2m1_array", codes)


def e8m0_to_f64(codes):
    """Decode E8M0 scale codes: 2^(e - 127), NaN for 0xFF."""
    return _decode("oracle_e8m0_array", codes)


def ue4m3_to_f64(codes):
    """Decode UE4M3 scale codes: the E4M3 magnitude, sign bit ignored."""
    return _decode("oracle_ue4m3_array", codes)


ELEMENT_FORMATS = {"e4m3": 0, "e5m2": 1, "e2m1": 2}
SCALE_FORMATS = {"e8m0": 0, "ue4m3": 1}
# The block-scaled formats: (element format, block size, scale format).
BLOCK_SCALED = {"mxfp8_e4m3": ("e4m3", 32, "e8m0"), "mxfp8_e5m2": ("e5m2", 32, "e8m0"),
                "mxfp4": ("e2m1", 32, "e8m0"), "nvfp4": ("e2m1", 16, "ue4m3")}


def gemm_block_scaled(fmt_a, fmt_b, A, SA, B, SB, *, block, scale_fmt, alpha=1.0, beta=0.0, C=None, rows=None):
    """Return (Cref, D) of the block-scaled product, float64 (rows, N).

    A: uint8 M x K codes (M x K/2 bytes for e2m1, two per byte, the even
    element in the low nibble); SA: uint8 M x ceil(K / block) scale codes.
    B and SB likewise for B stored N x K (K-major).  fmt_a / fmt_b: "e4m3",
    "e5m2" or "e2m1"; scale_fmt: "e8m0" or "ue4m3".  K is A's width in
    elements (twice its bytes for e2m1, so K is even there)."""
    lib = _load()
    A, SA, B, SB = (np.ascontiguousarray(x, dtype=np.uint8) for x in (A, SA, B, SB))
    M, N = A.shape[0], B.shape[0]
    K = A.shape[1] * (2 if fmt_a == "e2m1" else 1)
    Kb = B.shape[1] * (2 if fmt_b == "e2m1" else 1)
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    nb = -(-K // block)
    if SA.shape != (M, nb) or SB.shape != (N, nb):
        raise ValueError(f"scales must be {M} x {nb} and {N} x {nb}")
    row0, row1 = rows if rows is not None else (0, M)
    if beta != 0.0:
        C = np.asarray(C)
        if C is None or C.dtype != np.float32 or C.shape != (M, N) or C.strides[1] != 4:
            raise ValueError("beta != 0 needs C, float32 M x N with unit column stride")
        ldc = C.strides[0] // 4
    else:
        C, ldc = None, max(N, 1)
    out = np.zeros((row1 - row0, N), dtype=np.float64)
    D = np.zeros((row1 - row0, N), dtype=np.float64)
    rc = lib.oracle_gemm_block_scaled(ELEMENT_FORMATS[fmt_a], ELEMENT_FORMATS[fmt_b], SCALE_FORMATS[scale_fmt],
                                      int(block), M, N, K, float(alpha), _ptr(A), max(A.shape[1], 1), _ptr(SA),
                                      max(nb, 1), _ptr(B), max(B.shape[1], 1), _ptr(SB), max(nb, 1), float(beta),
                                      _ptr(C), ldc, row0, row1, _ptr(out), _ptr(D), max(N, 1))
    if rc != 0:
        raise ValueError(f"oracle_gemm_block_scaled rejected its arguments ({rc})")
    return out, D


ACTIVATIONS = {"none": 0, "gelu": 1, "dgelu": 2}


def gelu(x: float) -> float:
    """GELU(x) = x * Phi(x), Phi the standard normal distribution function."""
    return _load().oracle_gelu(float(x))


def dgelu(x: float) -> float:
    """GELU'(x) = Phi(x) + x * phi(x)."""
    return _load().oracle_dgelu(float(x))


def attention(Q, K, V, *, causal=True, scale=None, problems=None):
    """Scaled dot-product attention, forward: (O, W) as float64 arrays of
    shape [p1 - p0, T, Dh] for problems p0 .. p1-1 (all by default).

    Q, K, V: uint16 bfloat16 bit patterns of shape [problems, T, Dh].
    O[i] = sum_j softmax_j(scale * q_i . k_j) v_j over the keys query i sees
    (j <= i when causal); W[i] = sum_j softmax_j |v_j|, the error scale.
    scale defaults to 1 / sqrt(Dh)."""
    lib = _load()
    Q, K, V = (np.ascontiguousarray(x, dtype=np.uint16) for x in (Q, K, V))
    if Q.ndim != 3 or K.shape != Q.shape or V.shape != Q.shape:
        raise ValueError("Q, K and V must share one [problems, T, Dh] shape")
    P, T, Dh = Q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(Dh)
    p0, p1 = problems if problems is not None else (0, P)
    O = np.zeros((p1 - p0, T, Dh), dtype=np.float64)
    W = np.zeros((p1 - p0, T, Dh), dtype=np.float64)
    rc = lib.oracle_attention(P, T, Dh, int(bool(causal)), float(scale), _ptr(Q), _ptr(K), _ptr(V), p0, p1,
                              _ptr(O), _ptr(W))
    if rc != 0:
        raise ValueError(f"oracle_attention rejected its arguments ({rc})")
    return O, W


def epilogue(act, Y, bias=None, Z=None):
    """The fused epilogue of gemm_run_epilogue applied to the exact
    pre-activation Y (float64 rows x N, e.g. from gemm()):
    none: Y + bias; gelu: GELU(Y + bias); dgelu: Y * GELU'(Z).
    bias: float32 vector of N (or None); Z: float32 rows x N."""
    lib = _load()
    Y = np.ascontiguousarray(Y, dtype=np.float64)
    rows, N = Y.shape
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        if bias.shape != (N,):
            raise ValueError("bias must have N elements")
    if Z is not None:
        Z = np.ascontiguousarray(Z, dtype=np.float32)
        if Z.shape != (rows, N):
            raise ValueError("Z must be rows x N")
    out = np.empty_like(Y)
    rc = lib.oracle_epilogue(ACTIVATIONS[act], rows, N, _ptr(Y), max(N, 1), _ptr(bias), _ptr(Z), max(N, 1),
                             _ptr(out), max(N, 1))
    if rc != 0:
        raise ValueError(f"oracle_epilogue rejected its arguments ({rc})")
    return out
