"""Python binding of libgemm.so, the GB300 dense GEMM library.

Argument marshalling only: torch tensors are turned into device pointers,
sizes, leading dimensions and the current CUDA stream, and every call goes
through the C ABI declared in include/gemm.h.  All arithmetic happens in the
library's kernels; there is no CPU or PyTorch fallback, and using the library
without the built extension raises.

    import torch, dense_gemm_transformer_gb300 as dg
    C = torch.empty(M, N, device="cuda")
    dg.gemm(A, B, C, mode="tf32")                # C = A @ B
    dg.gemm(A, W, C, mode="bf16", transB=True)   # C = A @ W^T, W stored N x K
    dg.gemm(X8, W8, C, mode="fp8", transB=True, alpha=sx * sw)  # E4M3 codes, W stored N x K
"""
from __future__ import annotations

import ctypes
import math
import os
import re
import threading

from . import _build

MODES = {"fp32": 0, "tf32": 1, "bf16": 2, "fp8": 3, "fp8_e4m3": 3, "fp8_e5m2": 4, "fp8_e4m3_e5m2": 5,
         "fp8_e5m2_e4m3": 6}
# The 8-bit format of (A, B) in each FP8 mode.
FP8_FORMATS = {"fp8": ("e4m3", "e4m3"), "fp8_e4m3": ("e4m3", "e4m3"), "fp8_e5m2": ("e5m2", "e5m2"),
               "fp8_e4m3_e5m2": ("e4m3", "e5m2"), "fp8_e5m2_e4m3": ("e5m2", "e4m3")}
# Block-scaled modes (gemm_run_block_scaled): element format, K elements per
# scale, scale format.
BLOCK_SCALED_MODES = {"mxfp8_e4m3": (7, "e4m3", 32, "e8m0"), "mxfp8_e5m2": (8, "e5m2", 32, "e8m0"),
                      "nvfp4": (9, "e2m1", 16, "ue4m3")}
FAMILIES = {"auto": 0, "simt": 1, "tc": 2, "skinny": 3}
OPTIONS = {"family": 1, "split_k": 2, "tile_n": 3, "pretranspose": 4, "pair": 5, "wait_limit_us": 6,
           "fault_skip_stage": 7, "sk_fixup": 8}
STATUS = {0: "GEMM_OK", 1: "GEMM_ERR_INVALID_VALUE", 2: "GEMM_ERR_NOT_SUPPORTED", 3: "GEMM_ERR_MISALIGNED",
          4: "GEMM_ERR_CUDA", 5: "GEMM_ERR_ALLOC", 6: "GEMM_ERR_DEVICE_TIMEOUT", 7: "GEMM_ERR_TOO_LARGE"}
HEADER = os.path.join(_build.ROOT, "include", "gemm.h")


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


ACTIVATIONS = {"none": 0, "gelu": 1, "dgelu": 2}


class Epilogue(ctypes.Structure):
    """gemm_epilogue_t."""
    _fields_ = [("activation", ctypes.c_int32), ("reserved", ctypes.c_int32), ("bias", ctypes.c_void_p),
                ("aux", ctypes.c_void_p), ("ld_aux", ctypes.c_int64)]


class Plan(ctypes.Structure):
    _fields_ = [("family", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("tile_k", ctypes.c_int32), ("split_k", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("grid", ctypes.c_int32), ("kernels", ctypes.c_int32), ("packed", ctypes.c_int32),
                ("schedule", ctypes.c_int32), ("cluster", ctypes.c_int32), ("pair_mma", ctypes.c_int32),
                ("epilogue_fused", ctypes.c_int32), ("sk_fixup", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 2)]


_lib = None
_lib_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Load libgemm.so (building it first only if asked) and declare its ABI."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                               "(the library has no fallback path)")
        lib = ctypes.CDLL(path)
        i64, vp, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        lib.gemm_create.argtypes = [ctypes.POINTER(vp)]
        lib.gemm_destroy.argtypes = [vp]
        lib.gemm_run.argtypes = [vp, i32, i32, i32, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
        lib.gemm_validate.argtypes = [i32, i32, i32, i64, i64, i64, f32, vp, i64, vp, i64, vp, i64]
        lib.gemm_set_option.argtypes = [vp, i32, i64]
        lib.gemm_get_plan.argtypes = [vp, ctypes.POINTER(Plan)]
        lib.gemm_check_device.argtypes = [vp, vp]
        lib.gemm_launch_null.argtypes = [vp, vp]
        lib.gemm_run_epilogue.argtypes = [vp, i32, i32, i32, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64,
                                          ctypes.POINTER(Epilogue), vp]
        lib.gemm_status_string.argtypes = [i32]
        lib.gemm_status_string.restype = ctypes.c_char_p
        for name in ("gemm_create", "gemm_destroy", "gemm_run", "gemm_validate", "gemm_set_option",
                     "gemm_get_plan", "gemm_check_device", "gemm_launch_null", "gemm_run_epilogue"):
            getattr(lib, name).restype = i32
        _lib = lib
        return lib


def header_functions() -> list[str]:
    """Names of the functions include/gemm.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:gemm_status_t|const char\*|int64_t)\s+(gemm_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


def validate(mode, transA, transB, M, N, K, alpha, A, lda, B, ldb, C, ldc) -> int:
    """Run the library's argument checks on raw pointers (no device needed)."""
    return load().gemm_validate(MODES[mode] if isinstance(mode, str) else int(mode), int(transA), int(transB),
                                M, N, K, float(alpha), A, lda, B, ldb, C, ldc)


def _check(status: int, what: str):
    if status != 0:
        raise GemmError(status, what)


def _matrix(t, name):
    """(device pointer, leading dimension) of a row-major 2-D tensor."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    rows, cols = t.shape
    if rows > 0 and cols > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} needs unit stride along its last dimension (row-major storage)")
    ld = t.stride(0) if rows > 1 else max(cols, 1)
    if rows > 1 and ld < cols:
        raise ValueError(f"{name} has overlapping rows")
    return t.data_ptr(), ld


def _operand_dtypes(torch, mode, which):
    """Tensor types operand `which` (0 = A, 1 = B) may have in `mode`: FP8
    codes as torch's float8 type of the operand's format or as raw uint8."""
    if mode == "bf16":
        return (torch.bfloat16,)
    if mode in FP8_FORMATS:
        fmt = FP8_FORMATS[mode][which]
        return (torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2, torch.uint8)
    return (torch.float32,)


class Gemm:
    """A library handle bound to the current CUDA device."""

    def __init__(self):
        self._lib = load()
        h = ctypes.c_void_p()
        _check(self._lib.gemm_create(ctypes.byref(h)), "gemm_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            st = self._lib.gemm_destroy(self._h)
            self._h = None
            _check(st, "gemm_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_option(self, name: str, value):
        if name == "family" and isinstance(value, str):
            value = FAMILIES[value]
        _check(self._lib.gemm_set_option(self._h, OPTIONS[name], int(value)), f"gemm_set_option({name})")

    def plan(self) -> dict:
        p = Plan()
        _check(self._lib.gemm_get_plan(self._h, ctypes.byref(p)), "gemm_get_plan")
        fam = {**{v: k for k, v in FAMILIES.items()}, 4: "attention"}.get(p.family, "none")
        return {"family": fam if p.kernels else "none", "tile_m": p.tile_m, "tile_n": p.tile_n,
                "tile_k": p.tile_k, "split_k": p.split_k, "stages": p.stages, "grid": p.grid,
                "kernels": p.kernels, "packed": p.packed,
                "schedule": {0: "tiles", 1: "split_k", 2: "stream_k", 3: "tail_split"}.get(p.schedule, "tiles"),
                "cluster": p.cluster, "pair_mma": p.pair_mma, "epilogue_fused": p.epilogue_fused,
                "sk_fixup": {1: "kernel", 2: "inline"}.get(p.sk_fixup, "none")}

    def check_device(self, stream=None) -> int:
        """Synchronize the stream and return the device status (0 = ok)."""
        return self._lib.gemm_check_device(self._h, _stream_ptr(stream))

    def launch_null(self, stream=None):
        """gemm_launch_null: an empty kernel with the launch configuration of
        the last call's main kernel, on `stream`."""
        _check(self._lib.gemm_launch_null(self._h, _stream_ptr(stream)), "gemm_launch_null")

    def run_ptr(self, mode, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None):
        """gemm_run on raw device pointers; `stream` is a torch stream, a raw handle or None."""
        st = self._lib.gemm_run(self._h, MODES[mode] if isinstance(mode, str) else int(mode), int(transA),
                                int(transB), int(M), int(N), int(K), float(alpha), A, int(lda), B, int(ldb),
                                float(beta), C, int(ldc), _stream_ptr(stream))
        _check(st, "gemm_run")

    def run_block_scaled(self, A, SA, B, SB, C, mode="nvfp4", alpha=1.0, beta=0.0, stream=None):
        """C = alpha * (A . SA) (B . SB)^T + beta * C through gemm_run_block_scaled.

        A: M x K codes (uint8; NVFP4: M x K/2 bytes, two E2M1 codes a byte),
        B: N x K codes (N x K/2 for NVFP4), both K contiguous; SA, SB: their
        scales in the tiled layout (tile_block_scales); C: M x N float32."""
        import torch
        code, _, _, _ = BLOCK_SCALED_MODES[mode]
        for t, name in ((A, "A"), (B, "B"), (SA, "SA"), (SB, "SB")):
            if t.dtype != torch.uint8 or not t.is_cuda:
                raise TypeError(f"{name} must be a uint8 CUDA tensor")
        per = 2 if mode == "nvfp4" else 1
        M, K = A.shape[0], A.shape[1] * per
        N = B.shape[0]
        if B.shape[1] * per != K or tuple(C.shape) != (M, N) or C.dtype != torch.float32:
            raise ValueError("shapes do not agree")
        pa, lda = _matrix(A, "A")
        pb, ldb = _matrix(B, "B")
        pc, ldc = _matrix(C, "C")
        if stream is None:
            stream = torch.cuda.current_stream(C.device)
        fn = self._lib.gemm_run_block_scaled
        i64, vp, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        fn.argtypes = [vp, i32, i64, i64, i64, f32, vp, i64, vp, vp, i64, vp, f32, vp, i64, vp]
        fn.restype = i32
        st = fn(self._h, code, M, N, K, float(alpha), pa, lda * per, SA.data_ptr(), pb, ldb * per, SB.data_ptr(),
                float(beta), pc, ldc, _stream_ptr(stream))
        _check(st, "gemm_run_block_scaled")
        return C

    def attention_ptr(self, problems, T, Dh, causal, scale, Q, K, V, O, stream=None):
        """gemm_attention_forward on raw device pointers."""
        fn = self._lib.gemm_attention_forward
        i64, vp, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        fn.argtypes = [vp, i64, i64, i64, i32, f32, vp, vp, vp, vp, vp]
        fn.restype = i32
        st = fn(self._h, int(problems), int(T), int(Dh), int(causal), float(scale), Q, K, V, O, _stream_ptr(stream))
        _check(st, "gemm_attention_forward")

    def attention(self, Q, K, V, O=None, causal=True, scale=None, stream=None):
        """O = softmax(scale Q K^T [causal mask]) V through gemm_attention_forward.

        Q, K, V: contiguous bfloat16 CUDA tensors of one shape [..., T, 64]
        (the leading dimensions, e.g. batch and head, are the independent
        problems); O: float32 of the same shape (allocated when None).
        scale defaults to 1 / sqrt(64)."""
        import torch
        if Q.dim() < 2 or K.shape != Q.shape or V.shape != Q.shape:
            raise ValueError("Q, K and V must share one [..., T, Dh] shape")
        for t, name in ((Q, "Q"), (K, "K"), (V, "V")):
            if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
                raise TypeError(f"{name} must be a contiguous bfloat16 CUDA tensor")
        T, Dh = Q.shape[-2], Q.shape[-1]
        problems = Q.numel() // max(T * Dh, 1)
        if O is None:
            O = torch.empty(Q.shape, dtype=torch.float32, device=Q.device)
        elif O.shape != Q.shape or O.dtype != torch.float32 or not O.is_contiguous():
            raise ValueError("O must be a contiguous float32 tensor of Q's shape")
        if scale is None:
            scale = 1.0 / math.sqrt(Dh)
        if stream is None:
            stream = torch.cuda.current_stream(Q.device)
        self.attention_ptr(problems, T, Dh, causal, scale, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                           stream)
        return O

    def run(self, A, B, C, mode="fp32", transA=False, transB=False, alpha=1.0, beta=0.0, stream=None,
            act="none", bias=None, aux=None):
        """C = alpha * op(A) op(B) + beta * C on torch CUDA tensors (row-major).

        mode: "fp32", "tf32", "bf16", or an FP8 mode ("fp8" = "fp8_e4m3",
        "fp8_e5m2", "fp8_e4m3_e5m2", "fp8_e5m2_e4m3": the formats of A and B),
        whose operands are torch.float8_e4m3fn / torch.float8_e5m2 tensors or
        raw uint8 codes; FP8 is fastest with A stored M x K and B stored N x K
        (transB=True), which the kernels read in place.

        With act / bias / aux, the fused epilogue of gemm_run_epilogue:
        act "none" or "gelu": C = act(alpha op(A) op(B) + beta C + bias) with
        bias a float32 vector of N (or None); act "dgelu": C = (alpha op(A)
        op(B) + beta C) * GELU'(aux), aux the float32 M x N pre-activation.
        """
        import torch
        for which, t in enumerate((A, B)):
            want = _operand_dtypes(torch, mode, which)
            if t.dtype not in want:
                raise TypeError(f"mode {mode} takes {want} for {'AB'[which]}, got {t.dtype}")
        if C.dtype != torch.float32:
            raise TypeError("C must be float32")
        M, K = (A.shape[1], A.shape[0]) if transA else (A.shape[0], A.shape[1])
        Kb, N = (B.shape[1], B.shape[0]) if transB else (B.shape[0], B.shape[1])
        if K != Kb or tuple(C.shape) != (M, N):
            raise ValueError(f"shapes do not agree: op(A) {M}x{K}, op(B) {Kb}x{N}, C {tuple(C.shape)}")
        pa, lda = _matrix(A, "A")
        pb, ldb = _matrix(B, "B")
        pc, ldc = _matrix(C, "C")
        if stream is None:
            stream = torch.cuda.current_stream(C.device)
        if act == "none" and bias is None and aux is None:
            self.run_ptr(mode, transA, transB, M, N, K, alpha, pa, lda, pb, ldb, beta, pc, ldc, stream)
            return C
        ep = Epilogue(ACTIVATIONS[act], 0, None, None, 0)
        if bias is not None:
            if bias.dtype != torch.float32 or bias.dim() != 1 or bias.numel() != N or bias.stride(0) != 1:
                raise ValueError("bias must be a contiguous float32 vector of N elements")
            ep.bias = bias.data_ptr()
        if aux is not None:
            if aux.dtype != torch.float32 or tuple(aux.shape) != (M, N):
                raise ValueError("aux must be float32 M x N")
            ep.aux, ep.ld_aux = _matrix(aux, "aux")
        st = self._lib.gemm_run_epilogue(self._h, MODES[mode], int(transA), int(transB), int(M), int(N), int(K),
                                         float(alpha), pa, int(lda), pb, int(ldb), float(beta), pc, int(ldc),
                                         ctypes.byref(ep), _stream_ptr(stream))
        _check(st, "gemm_run_epilogue")
        return C


def tile_block_scales(S, stream=None):
    """The tiled layout of block scales that gemm_run_block_scaled reads:
    S is a rows x blocks uint8 tensor on the device (row-major); returns a
    new uint8 device tensor written by gemm_block_scales_tile."""
    import torch
    lib = load()
    fn_bytes, fn = lib.gemm_block_scales_tiled_bytes, lib.gemm_block_scales_tile
    fn_bytes.argtypes, fn_bytes.restype = [ctypes.c_int64, ctypes.c_int64], ctypes.c_int64
    fn.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    if S.dtype != torch.uint8 or S.dim() != 2 or not S.is_cuda:
        raise ValueError("scales must be a 2-D uint8 CUDA tensor")
    rows, blocks = S.shape
    T = torch.empty((max(int(fn_bytes(rows, blocks)), 16),), dtype=torch.uint8, device=S.device)
    ps, lds = _matrix(S, "S")
    if stream is None:
        stream = torch.cuda.current_stream(S.device)
    _check(fn(rows, blocks, ps, lds, T.data_ptr(), _stream_ptr(stream)), "gemm_block_scales_tile")
    return T


def _stream_ptr(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return getattr(stream, "cuda_stream", stream)


_default = {}


def default_handle() -> Gemm:
    import torch
    dev = torch.cuda.current_device()
    if dev not in _default:
        _default[dev] = Gemm()
    return _default[dev]


def gemm(A, B, C, mode="fp32", transA=False, transB=False, alpha=1.0, beta=0.0, stream=None, act="none",
         bias=None, aux=None):
    """C = alpha * op(A) op(B) + beta * C with the current device's default handle
    (and the fused epilogue of Gemm.run when act / bias / aux are given)."""
    return default_handle().run(A, B, C, mode, transA, transB, alpha, beta, stream, act, bias, aux)


def attention(Q, K, V, O=None, causal=True, scale=None, stream=None):
    """Fused attention forward with the current device's default handle (Gemm.attention)."""
    return default_handle().attention(Q, K, V, O, causal=causal, scale=scale, stream=stream)


def run_small_m_noalloc(A, B, C, mode="bf16", transB=False, alpha=1.0, beta=0.0, stream=None):
    """C = alpha * A op(B) + beta * C for M <= 16 through gemm_run_small_m_noalloc.

    For callers that may not allocate device memory (a runtime that owns all
    allocations, a plug-in in another program's CUDA context): the library
    uses only its fixed internal scratch array and no handle.  A is M x K,
    B is K x N (or N x K with transB), C is M x N float32, all on the device.
    """
    import torch
    lib = load()
    fn = lib.gemm_run_small_m_noalloc
    if fn.argtypes is None:
        i64, vp, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
        fn.argtypes = [i32, i32, i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
        fn.restype = i32
    M, K = A.shape
    N = B.shape[0] if transB else B.shape[1]
    pa, lda = _matrix(A, "A")
    pb, ldb = _matrix(B, "B")
    pc, ldc = _matrix(C, "C")
    if stream is None:
        stream = torch.cuda.current_stream(C.device)
    _check(fn(MODES[mode], int(bool(transB)), M, N, K, float(alpha), pa, lda, pb, ldb, float(beta), pc, ldc,
              _stream_ptr(stream)), "gemm_run_small_m_noalloc")
    return C
