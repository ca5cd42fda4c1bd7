"""The C ABI on the host: symbols, argument checks, status strings, and the
register/spill guard of the built kernels.  No GPU and no kernel launch."""
import ctypes
import re

import pytest

import dense_gemm_transformer_gb300 as dg
from dense_gemm_transformer_gb300 import _build

OK, INVALID, NOT_SUPPORTED, MISALIGNED = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    return dg.load(build_if_missing=True)


def test_library_exports_every_declared_function(lib):
    names = dg.header_functions()
    assert {"gemm_create", "gemm_run", "gemm_destroy", "gemm_status_string"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in dg.STATUS.items():
        assert dg.status_string(code) == name
    assert dg.status_string(99) == "GEMM_ERR_UNKNOWN"


P = 0x10000  # a 64 KiB-aligned fake device address: never dereferenced by the checks


def v(mode="fp32", tA=0, tB=0, M=8, N=8, K=8, alpha=1.0, A=P, lda=None, B=P, ldb=None, C=P, ldc=None):
    lda = lda if lda is not None else (M if tA else K)
    ldb = ldb if ldb is not None else (K if tB else N)
    ldc = ldc if ldc is not None else N
    return dg.validate(mode, tA, tB, M, N, K, alpha, A, lda, B, ldb, C, ldc)


def test_validate_accepts_good_arguments(lib):
    for mode in ("fp32", "tf32", "bf16"):
        for tA in (0, 1):
            for tB in (0, 1):
                assert v(mode, tA, tB, M=33, N=17, K=5) == OK
    assert v(M=4, N=3, K=2, lda=100, ldb=100, ldc=100) == OK


def test_validate_rejects_bad_flags_and_sizes(lib):
    assert dg.validate(7, 0, 0, 8, 8, 8, 1.0, P, 8, P, 8, P, 8) == INVALID
    for fp8_mode in (4, 5, 6):  # E5M2 and the mixed pairs
        assert dg.validate(fp8_mode, 0, 1, 8, 8, 8, 1.0, P + 1, 8, P + 3, 8, P, 8) == OK
    # FP8 (mode 3): one-byte operands, so any operand address is aligned
    assert dg.validate(3, 0, 1, 8, 8, 8, 1.0, P + 1, 8, P + 3, 8, P, 8) == OK
    assert dg.validate(-1, 0, 0, 8, 8, 8, 1.0, P, 8, P, 8, P, 8) == INVALID
    assert v(tA=2) == INVALID and v(tB=-1) == INVALID
    assert v(M=-1) == INVALID and v(N=-5) == INVALID and v(K=-1) == INVALID
    assert v(M=2**31) == INVALID


def test_validate_leading_dimensions(lib):
    assert v(M=8, K=16, lda=15) == INVALID            # A stored M x K needs lda >= K
    assert v(tA=1, M=8, K=16, lda=7) == INVALID       # A stored K x M needs lda >= M
    assert v(tA=1, M=8, K=16, lda=8) == OK
    assert v(N=9, K=4, ldb=8) == INVALID              # B stored K x N needs ldb >= N
    assert v(tB=1, N=9, K=4, ldb=3) == INVALID        # B stored N x K needs ldb >= K
    assert v(N=9, ldc=8) == INVALID


def test_validate_null_and_misaligned_pointers(lib):
    assert v(A=None) == INVALID and v(B=None) == INVALID and v(C=None) == INVALID
    assert v(mode="fp32", A=P + 2) == MISALIGNED
    assert v(mode="bf16", A=P + 2) == OK              # bf16 needs 2-byte alignment only
    assert v(mode="bf16", B=P + 1) == MISALIGNED
    assert v(C=P + 2) == MISALIGNED


def test_validate_degenerate_sizes(lib):
    # M == 0 or N == 0: nothing is touched, nothing else is checked.
    assert v(M=0, A=None, B=None, C=None) == OK
    assert v(N=0, A=None, B=None, C=None) == OK
    # K == 0 or alpha == 0: C = beta * C, A and B are never read.
    assert v(K=0, A=None, B=None) == OK
    assert v(alpha=0.0, A=None, B=None, lda=0, ldb=0) == OK
    assert v(K=0, C=None) == INVALID


def test_null_handle_is_rejected_everywhere(lib):
    assert lib.gemm_run(None, 0, 0, 0, 8, 8, 8, 1.0, P, 8, P, 8, 0.0, P, 8, None) == INVALID
    assert lib.gemm_destroy(None) == INVALID
    assert lib.gemm_set_option(None, 1, 0) == INVALID
    assert lib.gemm_get_plan(None, ctypes.byref(dg.Plan())) == INVALID
    assert lib.gemm_check_device(None, None) == INVALID
    assert lib.gemm_create(None) == INVALID


def test_every_kernel_is_free_of_spills(lib):
    """Spilling to local memory (or trading it for registers past an occupancy
    step) is the silent regression "bare-metal-bard" describes in its fourth
    paragraph; the build's ptxas report must show zero spill bytes."""
    with open(_build.PTXAS_REPORT) as f:
        text = f.read()
    spills = re.findall(r"(\d+) bytes spill stores, (\d+) bytes spill loads", text)
    assert spills, "ptxas report has no kernels"
    assert all(s == "0" and l == "0" for s, l in spills), spills
    # Registers per kernel: the 128-column SIMT kernel keeps two 256-thread
    # CTAs per SM only at <= 128 registers; one 256-thread CTA of the
    # 256-column kernel fits the 64K register file at <= 255.
    per_kernel = re.findall(r"Compiling entry function '(\w+)'.*?Used (\d+) registers", text, re.S)
    assert per_kernel
    for name, regs in per_kernel:
        limit = 128 if "simt_gemm_kernelILi128" in name else 255
        assert int(regs) <= limit, (name, regs)


def _header_enum(prefix):
    """NAME -> value of the enumerators of include/gemm.h that start with prefix."""
    import os
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gemm.h")
    text = re.sub(r"/\*.*?\*/", " ", open(path).read(), flags=re.S)
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(" + prefix + r"\w*)\s*=\s*(\d+)", text)}


def test_binding_constants_match_the_header():
    """The ctypes binding's option, mode, family, activation and status
    codes are the header's enumerators, so no call passes a stale code."""
    opts = _header_enum("GEMM_OPT_")
    assert sorted(dg.OPTIONS.values()) == sorted(opts.values())
    for name, code in dg.OPTIONS.items():
        assert opts["GEMM_OPT_" + name.upper()] == code, name
    modes = _header_enum("GEMM_MODE_")
    for name, code in dg.MODES.items():
        key = "GEMM_MODE_" + ("FP8_E4M3" if name == "fp8" else name.upper())
        assert modes[key] == code, name
    for name, (code, _, _, _) in dg.BLOCK_SCALED_MODES.items():
        assert modes["GEMM_MODE_" + name.upper()] == code, name
    assert set(modes.values()) == set(dg.MODES.values()) | {v[0] for v in dg.BLOCK_SCALED_MODES.values()}
    fams = _header_enum("GEMM_FAMILY_")
    for name, code in dg.FAMILIES.items():
        assert fams["GEMM_FAMILY_" + name.upper()] == code, name
    acts = _header_enum("GEMM_ACT_")
    for name, code in dg.ACTIVATIONS.items():
        assert acts["GEMM_ACT_" + name.upper()] == code, name
    status = {**_header_enum("GEMM_OK"), **_header_enum("GEMM_ERR_")}
    assert {v: k for k, v in status.items()} == dg.STATUS


def test_plan_struct_matches_the_header():
    """gemm_plan_t field by field: every int32 member of the header's struct,
    in order, is a field of the ctypes Plan at the same offset."""
    import os
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gemm.h")
    text = re.sub(r"/\*.*?\*/", " ", open(path).read(), flags=re.S)
    body = re.search(r"typedef struct \{([^}]*)\} gemm_plan_t;", text).group(1)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if not decl:
            continue
        assert decl.startswith("int32_t "), decl
        for name in decl[len("int32_t "):].split(","):
            name = name.strip()
            m = re.fullmatch(r"(\w+)\[(\d+)\]", name)
            fields.append((m.group(1), int(m.group(2))) if m else (name, 1))
    offset = 0
    for name, count in fields:
        f = getattr(dg.Plan, name)
        assert f.offset == offset and f.size == 4 * count, name
        offset += 4 * count
    assert ctypes.sizeof(dg.Plan) == offset
