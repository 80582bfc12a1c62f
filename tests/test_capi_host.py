"""Host-side checks of the C ABI that launch nothing (run without a GPU).

The library must load, export every function the header declares, and
reject bad arguments on the host with the documented status codes before any
CUDA call.
"""

from __future__ import annotations

import os
import re

import pytest
import torch

from int8_quantized_linear_gb300 import build as lib_build
from int8_quantized_linear_gb300 import capi

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "i8ql.h")


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return capi.lib()


def _declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = "\n".join(line for line in text.splitlines() if not line.lstrip().startswith("#"))
    names = re.findall(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", text)
    return sorted({n for n in names if n not in {"if", "defined"}})


def test_header_declares_the_five_operations():
    names = _declared_functions()
    for op in ("quantize_weight_per_channel_int8", "quantize_act_per_token_int8", "w8a8_gemm",
               "w8a16_gemm", "grouped_w8a16_gemm"):
        assert op in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert names, "no declarations parsed"
    for name in names:
        assert hasattr(lib, name), f"libi8ql.so does not export {name}"
        assert name in capi.SIGNATURES, f"binding has no signature for {name}"


def test_status_strings_and_version(lib):
    for s in range(0, 8):
        assert capi.status_string(s) != "unknown status"
    assert capi.status_string(99) == "unknown status"
    assert capi.i8ql_version() >= 10000


A = 0x10000  # a fake, 16-byte-aligned "device" address: never dereferenced here
B = 0x20000
C = 0x30000
D = 0x40000


@pytest.mark.parametrize("fn", ["quantize_weight_per_channel_int8", "quantize_act_per_token_int8"])
def test_quant_argument_errors(lib, fn):
    f = getattr(lib, fn)
    assert f(A, 4, 0, B, C, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(A, 4, 24, B, C, None) == capi.I8QL_ERR_UNSUPPORTED
    assert f(A, 4, capi.I8QL_MAX_K + 16, B, C, None) == capi.I8QL_ERR_UNSUPPORTED
    assert f(A, -1, 16, B, C, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(None, 4, 16, B, C, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(A + 8, 4, 16, B, C, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(A, 4, 16, B + 4, C, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(A, 4, 16, B, C + 2, None) == capi.I8QL_ERR_INVALID_ARG
    # an empty problem launches nothing and succeeds, whatever the pointers
    assert f(None, 0, 16, None, None, None) == capi.I8QL_OK


def test_w8a8_argument_errors(lib):
    f = lib.w8a8_gemm
    ok = (A, B, C, D, None, A, None, 8, 16, 64, None)
    args = list(ok)
    args[9] = 40  # K not a multiple of 16
    assert f(*args) == capi.I8QL_ERR_UNSUPPORTED
    args = list(ok); args[8] = 0  # N = 0
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG
    args = list(ok); args[0] = None
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG
    args = list(ok); args[2] = B + 1
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG
    args = list(ok); args[4] = A + 1  # bias must be 2-byte aligned
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG
    args = list(ok); args[6] = A + 4  # acc_debug must be 16-byte aligned
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG
    args = list(ok); args[7] = 0
    assert f(*args) == capi.I8QL_OK


def test_w8a16_argument_errors(lib):
    f = lib.w8a16_gemm
    assert f(A, B, C, D, 4, 16, 8, None) == capi.I8QL_ERR_UNSUPPORTED
    assert f(A, B, C, D, 4, -2, 64, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(A, None, C, D, 4, 16, 64, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(A, B, C + 2, D, 4, 16, 64, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(None, B, C, None, 0, 16, 64, None) == capi.I8QL_OK


def test_grouped_argument_errors(lib):
    f = lib.grouped_w8a16_gemm
    ok = [A, B, 4, C, D, A, 8, 16, 64, None]
    a = list(ok); a[1] = None
    assert f(*a) == capi.I8QL_ERR_INVALID_ARG
    a = list(ok); a[2] = 0
    assert f(*a) == capi.I8QL_ERR_INVALID_ARG
    a = list(ok); a[2] = 70000
    assert f(*a) == capi.I8QL_ERR_UNSUPPORTED
    a = list(ok); a[8] = 20
    assert f(*a) == capi.I8QL_ERR_UNSUPPORTED
    a = list(ok); a[6] = 0
    assert f(*a) == capi.I8QL_OK


def test_w8a8_noalloc_argument_errors(lib):
    f = lib.w8a8_gemm_noalloc
    ok = (A, B, C, D, None, A, None, 8, 16, 64, None)
    args = list(ok); args[9] = 40
    assert f(*args) == capi.I8QL_ERR_UNSUPPORTED
    args = list(ok); args[2] = None
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG
    args = list(ok); args[7] = 0
    assert f(*args) == capi.I8QL_OK
    # beyond the fixed array on the large-M path: refused before any CUDA call
    big = list(ok); big[7] = capi.I8QL_NOALLOC_MAX_ELEMENTS // 4096 + 1; big[8] = 48; big[9] = 4096
    assert f(*big) == capi.I8QL_ERR_WORKSPACE_LIMIT


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_reports_no_device(lib):
    assert lib.w8a16_gemm(A, B, C, D, 4, 16, 64, None) == capi.I8QL_ERR_NO_DEVICE


@pytest.mark.parametrize("fn", ["i8ql_w8a8_plan", "i8ql_w8a8_noalloc_plan", "i8ql_fp8_plan"])
def test_w8a8_plan_argument_errors(lib, fn):
    import ctypes
    a, b, c = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    ra, rb, rc = ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)
    f = getattr(lib, fn)
    assert f(256, 512, 40, ra, rb, rc) == capi.I8QL_ERR_UNSUPPORTED
    assert f(256, 0, 64, ra, rb, rc) == capi.I8QL_ERR_INVALID_ARG
    assert f(-1, 16, 64, ra, rb, rc) == capi.I8QL_ERR_INVALID_ARG
    assert f(256, 16, 64, None, rb, rc) == capi.I8QL_ERR_INVALID_ARG
    assert f(256, 16, 64, ra, rb, None) == capi.I8QL_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert f(256, 16, 64, ra, rb, rc) == capi.I8QL_ERR_NO_DEVICE


def test_w8a8_linear_argument_errors(lib):
    f = lib.w8a8_linear
    ok = (A, B, C, None, D, None, None, None, 8, 16, 64, None)
    args = list(ok); args[10] = 40
    assert f(*args) == capi.I8QL_ERR_UNSUPPORTED          # K % 16
    args = list(ok); args[0] = None
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG          # x
    args = list(ok); args[5] = A + 8
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG          # qx misaligned
    args = list(ok); args[6] = A + 2
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG          # sx misaligned
    args = list(ok); args[8] = 0
    assert f(*args) == capi.I8QL_OK                        # M = 0: nothing to do
    if not torch.cuda.is_available():
        assert f(*ok) == capi.I8QL_ERR_NO_DEVICE


@pytest.mark.parametrize("fn", ["quantize_weight_per_channel_fp8", "quantize_act_per_token_fp8"])
def test_fp8_quant_argument_errors(lib, fn):
    f = getattr(lib, fn)
    assert f(A, 4, 0, B, C, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(A, 4, 24, B, C, None) == capi.I8QL_ERR_UNSUPPORTED
    assert f(None, 4, 16, B, C, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(A, 4, 16, B + 4, C, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(A, 4, 16, B, C + 2, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(None, 0, 16, None, None, None) == capi.I8QL_OK


def test_fp8_gemm_and_linear_argument_errors(lib):
    f = lib.w8a8_fp8_gemm
    ok = (A, B, C, D, None, A, 8, 16, 64, None)
    args = list(ok); args[8] = 40
    assert f(*args) == capi.I8QL_ERR_UNSUPPORTED          # K % 16
    args = list(ok); args[7] = 0
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG          # N = 0
    args = list(ok); args[2] = None
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG          # qw
    args = list(ok); args[4] = A + 1
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG          # bias misaligned
    args = list(ok); args[6] = 0
    assert f(*args) == capi.I8QL_OK
    g = lib.w8a8_fp8_linear
    ok = (A, B, C, None, D, None, None, 8, 16, 64, None)
    args = list(ok); args[9] = 40
    assert g(*args) == capi.I8QL_ERR_UNSUPPORTED
    args = list(ok); args[5] = A + 8
    assert g(*args) == capi.I8QL_ERR_INVALID_ARG          # qx misaligned
    args = list(ok); args[7] = 0
    assert g(*args) == capi.I8QL_OK
    if not torch.cuda.is_available():
        assert f(*(A, B, C, D, None, A, 8, 16, 64, None)) == capi.I8QL_ERR_NO_DEVICE


def test_w4_argument_errors(lib):
    f = lib.quantize_weight_w4_g128
    assert f(A, 4, 64, B, C, None) == capi.I8QL_ERR_UNSUPPORTED        # K % 128
    assert f(A, 4, 128, B, C + 1, None) == capi.I8QL_ERR_INVALID_ARG   # scale misaligned
    assert f(None, 0, 128, None, None, None) == capi.I8QL_OK
    g = lib.w4a16_gemm
    assert g(A, B, C, D, 4, 16, 192, None) == capi.I8QL_ERR_UNSUPPORTED
    assert g(A, None, C, D, 4, 16, 256, None) == capi.I8QL_ERR_INVALID_ARG
    assert g(A, B, C, D, 4, 0, 256, None) == capi.I8QL_ERR_INVALID_ARG
    assert g(None, B, C, None, 0, 16, 256, None) == capi.I8QL_OK
    if not torch.cuda.is_available():
        assert g(A, B, C, D, 4, 16, 256, None) == capi.I8QL_ERR_NO_DEVICE


def test_moe_argument_errors(lib):
    r = lib.moe_route_topk
    assert r(A, 8, 64, 0, 2, B, C, D, A, None) == capi.I8QL_ERR_INVALID_ARG      # top_k = 0
    assert r(A, 8, 64, 65, 2, B, C, D, A, None) == capi.I8QL_ERR_INVALID_ARG     # top_k > E
    assert r(A, 8, 300, 6, 2, B, C, D, A, None) == capi.I8QL_ERR_UNSUPPORTED     # E > 256
    assert r(A, 8, 64, 6, 2, None, C, D, A, None) == capi.I8QL_ERR_INVALID_ARG   # offsets
    g = lib.grouped_w8a16_silu_mul
    ok = [A, None, B, 66, C, D, A, 8, 16, 64, None]
    a = list(ok); a[9] = 40
    assert g(*a) == capi.I8QL_ERR_UNSUPPORTED                                    # K % 16
    a = list(ok); a[2] = None
    assert g(*a) == capi.I8QL_ERR_INVALID_ARG                                    # offsets
    a = list(ok); a[7] = 0
    assert g(*a) == capi.I8QL_OK                                                 # no rows
    c = lib.moe_combine
    assert c(A, B, C, D, 4, 8, 12, None) == capi.I8QL_ERR_UNSUPPORTED            # H % 8
    assert c(A, B, C, D, 0, 8, 16, None) == capi.I8QL_OK
    m = lib.moe_expert_mlp_w8a16
    ok = [A, B, 64, 6, 2, C, D, A, B, C, 8, 2048, 1408, None]
    a = list(ok); a[11] = 2050
    assert m(*a) == capi.I8QL_ERR_UNSUPPORTED                                    # H % 16
    a = list(ok); a[10] = 0
    assert m(*a) == capi.I8QL_OK
    if not torch.cuda.is_available():
        assert m(*ok) == capi.I8QL_ERR_NO_DEVICE


def test_w8a8_linear_fused_argument_errors(lib):
    f = lib.w8a8_linear_fused
    ok = (A, B, C, None, D, None, None, None, 8, 16, 64, None)
    args = list(ok); args[8] = 9
    assert f(*args) == capi.I8QL_ERR_UNSUPPORTED          # more than 8 tokens
    args = list(ok); args[10] = 40
    assert f(*args) == capi.I8QL_ERR_UNSUPPORTED          # K % 16
    args = list(ok); args[0] = None
    assert f(*args) == capi.I8QL_ERR_INVALID_ARG
    args = list(ok); args[8] = 0
    assert f(*args) == capi.I8QL_OK


def test_early_weight_loads_setting(lib):
    """Process-wide option, off by default; setting it needs no device."""
    assert lib.i8ql_early_weight_loads() == 0
    lib.i8ql_set_early_weight_loads(1)
    try:
        assert lib.i8ql_early_weight_loads() == 1
    finally:
        lib.i8ql_set_early_weight_loads(0)
    assert lib.i8ql_early_weight_loads() == 0


def test_w8a8_linear_launches_argument_errors(lib):
    import ctypes
    n = ctypes.c_int32(-1)
    f = lib.i8ql_w8a8_linear_launches
    assert f(8, 16, 40, ctypes.byref(n)) == capi.I8QL_ERR_UNSUPPORTED   # K % 16
    assert f(8, 0, 64, ctypes.byref(n)) == capi.I8QL_ERR_INVALID_ARG    # N = 0
    assert f(-1, 16, 64, ctypes.byref(n)) == capi.I8QL_ERR_INVALID_ARG
    assert f(8, 16, 64, None) == capi.I8QL_ERR_INVALID_ARG
    assert f(0, 16, 64, ctypes.byref(n)) == capi.I8QL_OK and n.value == 0  # nothing to launch
    if not torch.cuda.is_available():
        assert f(8, 16, 64, ctypes.byref(n)) == capi.I8QL_ERR_NO_DEVICE


def test_binding_constants_match_the_header():
    text = open(HEADER).read()
    for name in ("I8QL_MAX_K", "I8QL_W8A8_DECODE_MAX_M"):
        m = re.search(rf"#define {name} (\d+)", text)
        assert m and int(m.group(1)) == getattr(capi, name), name
    m = re.search(r"#define I8QL_NOALLOC_MAX_ELEMENTS \((\d+) \* (\d+) \* (\d+)\)", text)
    assert m and int(m.group(1)) * int(m.group(2)) * int(m.group(3)) == capi.I8QL_NOALLOC_MAX_ELEMENTS


def test_every_declaration_cites_its_source():
    """Each comment that documents header declarations names the passage the
    operation follows ("Source:"), or says it has none on the pages."""
    text = open(HEADER).read()
    blocks = re.findall(r"/\*(.*?)\*/\s*(?:#define[^\n]*\n\s*)*"
                        r"((?:(?:i8ql_status|int32_t|const char\*|void)\s+\w+\s*\([^;]*\);\s*)+)", text, re.S)
    documented = set()
    for comment, decls in blocks:
        names = re.findall(r"(\w+)\s*\(", decls)
        flat = " ".join(" ".join(line.strip().lstrip("*").split()) for line in comment.splitlines()).strip()
        assert "Source:" in flat or "no counterpart on the pages" in flat.lower(), names
        documented.update(names)
    missing = set(_declared_functions()) - documented
    assert not missing, f"declarations without a comment: {sorted(missing)}"
