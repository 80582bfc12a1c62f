"""Python binding of ``libi8ql.so`` (argument marshalling only).

Each function keeps the name of its C entry point, takes torch CUDA tensors,
checks dtypes, shapes and contiguity, allocates any output the caller did not
pass (torch is only the device-memory and stream provider), and calls the C
ABI with raw device pointers and the current CUDA stream.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.  If the
library is missing, loading fails with an error that says how to build it.
"""

from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libi8ql.so")

I8QL_OK = 0
I8QL_ERR_INVALID_ARG = 1
I8QL_ERR_UNSUPPORTED = 2
I8QL_ERR_CUDA = 3
I8QL_ERR_TIMEOUT = 4
I8QL_ERR_BAD_OFFSETS = 5
I8QL_ERR_NO_DEVICE = 6
I8QL_ERR_WORKSPACE_LIMIT = 7
I8QL_MAX_K = 133144
I8QL_NOALLOC_MAX_ELEMENTS = 16 * 1024 * 1024
I8QL_W8A8_DECODE_MAX_M = 32  # w8a8_gemm runs the decode kernel up to this M

# Every symbol the C header declares, with its ctypes signature.
_P, _I64, _S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
SIGNATURES = {
    "quantize_weight_per_channel_int8": (_S, [_P, _I64, _I64, _P, _P, _P]),
    "quantize_act_per_token_int8": (_S, [_P, _I64, _I64, _P, _P, _P]),
    "w8a8_gemm": (_S, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w8a8_gemm_noalloc": (_S, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w8a8_linear": (_S, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w8a16_gemm": (_S, [_P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "grouped_w8a16_gemm": (_S, [_P, _P, _I64, _P, _P, _P, _I64, _I64, _I64, _P]),
    "i8ql_w8a8_plan": (_S, [_I64, _I64, _I64, _P, _P, _P]),
    "i8ql_fp8_plan": (_S, [_I64, _I64, _I64, _P, _P, _P]),
    "i8ql_w8a8_noalloc_plan": (_S, [_I64, _I64, _I64, _P, _P, _P]),
    "i8ql_w8a8_linear_launches": (_S, [_I64, _I64, _I64, _P]),
    "i8ql_get_device_error": (_S, [_P]),
    "i8ql_status_string": (ctypes.c_char_p, [_S]),
    "i8ql_version": (_S, []),
    "i8ql_debug_stream_k_timeout": (None, [_S]),
    "i8ql_set_early_weight_loads": (None, [_S]),
    "i8ql_early_weight_loads": (_S, []),
    "quantize_weight_per_channel_fp8": (_S, [_P, _I64, _I64, _P, _P, _P]),
    "quantize_act_per_token_fp8": (_S, [_P, _I64, _I64, _P, _P, _P]),
    "w8a8_fp8_gemm": (_S, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w8a8_fp8_linear": (_S, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "quantize_weight_w4_g128": (_S, [_P, _I64, _I64, _P, _P, _P]),
    "w4a16_gemm": (_S, [_P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w8a8_linear_fused": (_S, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "moe_route_topk": (_S, [_P, _I64, _I64, _I64, _I64, _P, _P, _P, _P, _P]),
    "grouped_w8a16_silu_mul": (_S, [_P, _P, _P, _I64, _P, _P, _P, _I64, _I64, _I64, _P]),
    "moe_combine": (_S, [_P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "moe_expert_mlp_w8a16": (_S, [_P, _P, _I64, _I64, _I64, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
}

_LIB = None


class I8qlError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIBRARY):
            raise ImportError(
                f"{LIBRARY} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        handle = ctypes.CDLL(LIBRARY)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


def status_string(status: int) -> str:
    return lib().i8ql_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != I8QL_OK:
        raise I8qlError(status, where)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, dtype: torch.dtype, shape: tuple, name: str) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.numel() and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _quant(fn_name: str, src: torch.Tensor, q, scale, stream):
    if src.dim() != 2:
        raise ValueError("input must be 2-D [rows, K]")
    rows, k = src.shape
    _need(src, torch.bfloat16, (rows, k), "input")
    if q is None:
        q = torch.empty((rows, k), dtype=torch.int8, device=src.device)
    if scale is None:
        scale = torch.empty((rows,), dtype=torch.float32, device=src.device)
    _need(q, torch.int8, (rows, k), "q")
    _need(scale, torch.float32, (rows,), "scale")
    st = getattr(lib(), fn_name)(_ptr(src), rows, k, _ptr(q), _ptr(scale), _stream(stream))
    _check(st, fn_name)
    return q, scale


def quantize_weight_per_channel_int8(w: torch.Tensor, q=None, scale=None, stream=None):
    """int8 codes [N, K] and fp32 per-output-channel scales [N] of bf16 w."""
    return _quant("quantize_weight_per_channel_int8", w, q, scale, stream)


def quantize_act_per_token_int8(x: torch.Tensor, q=None, scale=None, stream=None):
    """int8 codes [M, K] and fp32 per-token scales [M] of bf16 x."""
    return _quant("quantize_act_per_token_int8", x, q, scale, stream)


def w8a8_linear(x, qw, sw, bias=None, y=None, qx=None, sx=None, acc_debug=None, stream=None, fused=False):
    """bf16 y [M, N] = w8a8_gemm(quantize_act_per_token_int8(x), qw, sw, bias),
    with the quantization fused into the call; qx / sx, when given, receive
    the token codes and scales.  fused=True takes the one-launch entry point
    (w8a8_linear_fused, M <= 8)."""
    m, k = x.shape
    n = qw.shape[0]
    _need(x, torch.bfloat16, (m, k), "x")
    _need(qw, torch.int8, (n, k), "qw")
    _need(sw, torch.float32, (n,), "sw")
    if bias is not None:
        _need(bias, torch.bfloat16, (n,), "bias")
    if y is None:
        y = torch.empty((m, n), dtype=torch.bfloat16, device=qw.device)
    _need(y, torch.bfloat16, (m, n), "y")
    if qx is not None:
        _need(qx, torch.int8, (m, k), "qx")
    if sx is not None:
        _need(sx, torch.float32, (m,), "sx")
    if acc_debug is not None:
        _need(acc_debug, torch.int32, (m, n), "acc_debug")
    name = "w8a8_linear_fused" if fused else "w8a8_linear"
    st = getattr(lib(), name)(_ptr(x), _ptr(qw), _ptr(sw), _ptr(bias), _ptr(y), _ptr(qx), _ptr(sx),
                              _ptr(acc_debug), m, n, k, _stream(stream))
    _check(st, name)
    return y


def w8a8_gemm(qx, sx, qw, sw, bias=None, y=None, acc_debug=None, stream=None):
    """bf16 y [M, N] = ((float)(qx @ qw^T) * sx[:, None]) * sw[None, :] (+ bias)."""
    m, k = qx.shape
    n = qw.shape[0]
    _need(qx, torch.int8, (m, k), "qx")
    _need(sx, torch.float32, (m,), "sx")
    _need(qw, torch.int8, (n, k), "qw")
    _need(sw, torch.float32, (n,), "sw")
    if bias is not None:
        _need(bias, torch.bfloat16, (n,), "bias")
    if y is None:
        y = torch.empty((m, n), dtype=torch.bfloat16, device=qw.device)
    _need(y, torch.bfloat16, (m, n), "y")
    if acc_debug is not None:
        _need(acc_debug, torch.int32, (m, n), "acc_debug")
    st = lib().w8a8_gemm(_ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), _ptr(bias), _ptr(y),
                         _ptr(acc_debug), m, n, k, _stream(stream))
    _check(st, "w8a8_gemm")
    return y


def w8a8_gemm_noalloc(qx, sx, qw, sw, y, bias=None, acc_debug=None, stream=None):
    """w8a8_gemm through the entry point that allocates no device memory.

    For callers that cannot allocate while they run (graph replay with fixed
    memory, allocator-free serving loops): the output ``y`` must be passed in,
    and the large-M workspace comes from a fixed array inside the library, so
    ``M * K`` may not exceed ``I8QL_NOALLOC_MAX_ELEMENTS`` when M > 32.
    Calls that could overlap on the GPU must not be issued (they share it).
    """
    m, k = qx.shape
    n = qw.shape[0]
    _need(qx, torch.int8, (m, k), "qx")
    _need(sx, torch.float32, (m,), "sx")
    _need(qw, torch.int8, (n, k), "qw")
    _need(sw, torch.float32, (n,), "sw")
    _need(y, torch.bfloat16, (m, n), "y")
    if bias is not None:
        _need(bias, torch.bfloat16, (n,), "bias")
    if acc_debug is not None:
        _need(acc_debug, torch.int32, (m, n), "acc_debug")
    st = lib().w8a8_gemm_noalloc(_ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), _ptr(bias), _ptr(y),
                                 _ptr(acc_debug), m, n, k, _stream(stream))
    _check(st, "w8a8_gemm_noalloc")
    return y


def w8a16_gemm(x, qw, sw, y=None, stream=None):
    """bf16 y [M, N] = bf16(sw[n] * sum_k qw[n, k] * x[m, k])."""
    m, k = x.shape
    n = qw.shape[0]
    _need(x, torch.bfloat16, (m, k), "x")
    _need(qw, torch.int8, (n, k), "qw")
    _need(sw, torch.float32, (n,), "sw")
    if y is None:
        y = torch.empty((m, n), dtype=torch.bfloat16, device=qw.device)
    _need(y, torch.bfloat16, (m, n), "y")
    st = lib().w8a16_gemm(_ptr(x), _ptr(qw), _ptr(sw), _ptr(y), m, n, k, _stream(stream))
    _check(st, "w8a16_gemm")
    return y


def grouped_w8a16_gemm(x, offsets, qw, sw, y=None, stream=None):
    """Grouped W8A16: rows offsets[e] .. offsets[e+1] of x use expert e."""
    t, k = x.shape
    e, n, k2 = qw.shape
    if k2 != k:
        raise ValueError("qw and x disagree on K")
    _need(x, torch.bfloat16, (t, k), "x")
    _need(offsets, torch.int32, (e + 1,), "offsets")
    _need(qw, torch.int8, (e, n, k), "qw")
    _need(sw, torch.float32, (e, n), "sw")
    if y is None:
        y = torch.empty((t, n), dtype=torch.bfloat16, device=qw.device)
    _need(y, torch.bfloat16, (t, n), "y")
    st = lib().grouped_w8a16_gemm(_ptr(x), _ptr(offsets), e, _ptr(qw), _ptr(sw), _ptr(y), t, n, k,
                                  _stream(stream))
    _check(st, "grouped_w8a16_gemm")
    return y


def _plan(fn_name: str, m: int, n: int, k: int) -> tuple[int, int, int]:
    tile_n, split_k, pair = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    _check(getattr(lib(), fn_name)(m, n, k, ctypes.byref(tile_n), ctypes.byref(split_k), ctypes.byref(pair)),
           fn_name)
    return tile_n.value, split_k.value, pair.value


def i8ql_w8a8_plan(m: int, n: int, k: int) -> tuple[int, int, int]:
    """(tile width, split-K factor, CTA-pair mode: 0 single CTAs, 1 pairs,
    2 pairs with stream-K) w8a8_gemm uses for an M x N x K problem on the
    current device; (0, 0, 0) in the decode range (M <= I8QL_W8A8_DECODE_MAX_M)."""
    return _plan("i8ql_w8a8_plan", m, n, k)


def i8ql_fp8_plan(m: int, n: int, k: int) -> tuple[int, int, int]:
    """(tile width, split-K factor, CTA pairs 0/1) w8a8_fp8_gemm uses for an
    M x N x K problem on the current device."""
    return _plan("i8ql_fp8_plan", m, n, k)


def i8ql_w8a8_noalloc_plan(m: int, n: int, k: int) -> tuple[int, int, int]:
    """The same for w8a8_gemm_noalloc (never stream-K)."""
    return _plan("i8ql_w8a8_noalloc_plan", m, n, k)


def i8ql_w8a8_linear_launches(m: int, n: int, k: int) -> int:
    """Kernels one w8a8_linear call of this size launches on the current
    device: 1 with the quantization inside the decode GEMM, else 2 (0 for
    m == 0)."""
    launches = ctypes.c_int32(-1)
    _check(lib().i8ql_w8a8_linear_launches(m, n, k, ctypes.byref(launches)), "i8ql_w8a8_linear_launches")
    return launches.value


def i8ql_get_device_error(stream=None) -> int:
    """Wait for the stream, then read and clear the sticky kernel-fault word."""
    return int(lib().i8ql_get_device_error(_stream(stream)))


def i8ql_version() -> int:
    return int(lib().i8ql_version())


def i8ql_debug_stream_k_timeout(on: bool) -> None:
    """Test hook: while on, stream-K finishers wait for a flag nothing writes
    (1 ms limit), so the call records I8QL_ERR_TIMEOUT without hanging."""
    lib().i8ql_debug_stream_k_timeout(1 if on else 0)


def i8ql_set_early_weight_loads(on: bool) -> None:
    """Serving option: decode-size GEMMs load their first weights before
    waiting for the previous kernel on the stream (which must not write
    them).  Process-wide; off by default."""
    lib().i8ql_set_early_weight_loads(1 if on else 0)


def i8ql_early_weight_loads() -> bool:
    return bool(lib().i8ql_early_weight_loads())


# ---------------------------------------------------------------- FP8 E4M3

def _quant_fp8(fn_name: str, src: torch.Tensor, q, scale, stream):
    if src.dim() != 2:
        raise ValueError("input must be 2-D [rows, K]")
    rows, k = src.shape
    _need(src, torch.bfloat16, (rows, k), "input")
    if q is None:
        q = torch.empty((rows, k), dtype=torch.uint8, device=src.device)
    if scale is None:
        scale = torch.empty((rows,), dtype=torch.float32, device=src.device)
    _need(q, torch.uint8, (rows, k), "q")
    _need(scale, torch.float32, (rows,), "scale")
    _check(getattr(lib(), fn_name)(_ptr(src), rows, k, _ptr(q), _ptr(scale), _stream(stream)), fn_name)
    return q, scale


def quantize_weight_per_channel_fp8(w: torch.Tensor, q=None, scale=None, stream=None):
    """E4M3 codes [N, K] (uint8) and fp32 per-channel scales (absmax / 448)."""
    return _quant_fp8("quantize_weight_per_channel_fp8", w, q, scale, stream)


def quantize_act_per_token_fp8(x: torch.Tensor, q=None, scale=None, stream=None):
    """E4M3 codes [M, K] (uint8) and fp32 per-token scales (absmax / 448)."""
    return _quant_fp8("quantize_act_per_token_fp8", x, q, scale, stream)


def w8a8_fp8_gemm(qx, sx, qw, sw, bias=None, y=None, stream=None):
    """bf16 y [M, N] = ((sum_k e4m3(qx) e4m3(qw)) * sx[:, None]) * sw[None, :] (+ bias)."""
    m, k = qx.shape
    n = qw.shape[0]
    _need(qx, torch.uint8, (m, k), "qx")
    _need(sx, torch.float32, (m,), "sx")
    _need(qw, torch.uint8, (n, k), "qw")
    _need(sw, torch.float32, (n,), "sw")
    if bias is not None:
        _need(bias, torch.bfloat16, (n,), "bias")
    if y is None:
        y = torch.empty((m, n), dtype=torch.bfloat16, device=qw.device)
    _need(y, torch.bfloat16, (m, n), "y")
    _check(lib().w8a8_fp8_gemm(_ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), _ptr(bias), _ptr(y), m, n, k,
                               _stream(stream)), "w8a8_fp8_gemm")
    return y


def w8a8_fp8_linear(x, qw, sw, bias=None, y=None, qx=None, sx=None, stream=None):
    """bf16 y = w8a8_fp8_gemm(quantize_act_per_token_fp8(x), qw, sw, bias) in one call."""
    m, k = x.shape
    n = qw.shape[0]
    _need(x, torch.bfloat16, (m, k), "x")
    _need(qw, torch.uint8, (n, k), "qw")
    _need(sw, torch.float32, (n,), "sw")
    if bias is not None:
        _need(bias, torch.bfloat16, (n,), "bias")
    if y is None:
        y = torch.empty((m, n), dtype=torch.bfloat16, device=qw.device)
    _need(y, torch.bfloat16, (m, n), "y")
    if qx is not None:
        _need(qx, torch.uint8, (m, k), "qx")
    if sx is not None:
        _need(sx, torch.float32, (m,), "sx")
    _check(lib().w8a8_fp8_linear(_ptr(x), _ptr(qw), _ptr(sw), _ptr(bias), _ptr(y), _ptr(qx), _ptr(sx), m, n, k,
                                 _stream(stream)), "w8a8_fp8_linear")
    return y


# ---------------------------------------------------------------- W4A16, group 128

def quantize_weight_w4_g128(w: torch.Tensor, q=None, scale=None, stream=None):
    """Packed int4 codes [N, K/2] (uint8) and bf16 group scales [N, K/128]."""
    n, k = w.shape
    _need(w, torch.bfloat16, (n, k), "w")
    if q is None:
        q = torch.empty((n, k // 2), dtype=torch.uint8, device=w.device)
    if scale is None:
        scale = torch.empty((n, k // 128), dtype=torch.bfloat16, device=w.device)
    _need(q, torch.uint8, (n, k // 2), "q")
    _need(scale, torch.bfloat16, (n, k // 128), "scale")
    _check(lib().quantize_weight_w4_g128(_ptr(w), n, k, _ptr(q), _ptr(scale), _stream(stream)),
           "quantize_weight_w4_g128")
    return q, scale


def w4a16_gemm(x, q, scale, y=None, stream=None):
    """bf16 y [M, N] = bf16(sum_g scale[n, g] * sum_k q[n, k] * x[m, k])."""
    m, k = x.shape
    n = q.shape[0]
    _need(x, torch.bfloat16, (m, k), "x")
    _need(q, torch.uint8, (n, k // 2), "q")
    _need(scale, torch.bfloat16, (n, k // 128), "scale")
    if y is None:
        y = torch.empty((m, n), dtype=torch.bfloat16, device=q.device)
    _need(y, torch.bfloat16, (m, n), "y")
    _check(lib().w4a16_gemm(_ptr(x), _ptr(q), _ptr(scale), _ptr(y), m, n, k, _stream(stream)), "w4a16_gemm")
    return y


# ---------------------------------------------------------------- MoE expert MLP

def moe_route_topk(logits, top_k, n_shared, stream=None):
    """Device routing: (offsets [E+n_shared+1], row_token [T*S], token_row
    [T, S], slot_weight [T, S]) for fp32 logits [T, E]."""
    t, e = logits.shape
    _need(logits, torch.float32, (t, e), "logits")
    s = top_k + n_shared
    dev = logits.device
    offsets = torch.empty((e + n_shared + 1,), dtype=torch.int32, device=dev)
    row_token = torch.empty((t * s,), dtype=torch.int32, device=dev)
    token_row = torch.empty((t, s), dtype=torch.int32, device=dev)
    slot_weight = torch.empty((t, s), dtype=torch.float32, device=dev)
    _check(lib().moe_route_topk(_ptr(logits), t, e, top_k, n_shared, _ptr(offsets), _ptr(row_token),
                                _ptr(token_row), _ptr(slot_weight), _stream(stream)), "moe_route_topk")
    return offsets, row_token, token_row, slot_weight


def grouped_w8a16_silu_mul(x, row_token, offsets, qw, sw, h=None, rows=None, stream=None):
    """h [rows, I] = bf16(silu(gate) * up) of the grouped fused gate/up
    projection qw [E, 2I, K], gathering token rows through row_token."""
    e, two_i, k = qw.shape
    inter = two_i // 2
    if rows is None:
        rows = row_token.shape[0] if row_token is not None else x.shape[0]
    _need(x, torch.bfloat16, (x.shape[0], k), "x")
    _need(offsets, torch.int32, (e + 1,), "offsets")
    if row_token is not None:
        _need(row_token, torch.int32, (rows,), "row_token")
    _need(sw, torch.float32, (e, two_i), "sw")
    if h is None:
        h = torch.empty((rows, inter), dtype=torch.bfloat16, device=qw.device)
    _need(h, torch.bfloat16, (rows, inter), "h")
    _check(lib().grouped_w8a16_silu_mul(_ptr(x), _ptr(row_token), _ptr(offsets), e, _ptr(qw), _ptr(sw), _ptr(h),
                                        rows, inter, k, _stream(stream)), "grouped_w8a16_silu_mul")
    return h


def moe_combine(yd, token_row, slot_weight, out=None, stream=None):
    """out [T, H] = bf16(sum_s slot_weight[t, s] * yd[token_row[t, s]])."""
    t, s = token_row.shape
    h = yd.shape[1]
    _need(token_row, torch.int32, (t, s), "token_row")
    _need(slot_weight, torch.float32, (t, s), "slot_weight")
    _need(yd, torch.bfloat16, (yd.shape[0], h), "yd")
    if out is None:
        out = torch.empty((t, h), dtype=torch.bfloat16, device=yd.device)
    _need(out, torch.bfloat16, (t, h), "out")
    _check(lib().moe_combine(_ptr(yd), _ptr(token_row), _ptr(slot_weight), _ptr(out), t, s, h, _stream(stream)),
           "moe_combine")
    return out


def moe_expert_mlp_w8a16(x, logits, top_k, n_shared, qw_gate_up, sw_gate_up, qw_down, sw_down, out=None,
                         stream=None):
    """The MoE expert MLP end to end (routing, gate/up + SiLU gate, down,
    combine) for tokens x [T, H] with gate logits [T, E_routed]."""
    t, hid = x.shape
    e_r = logits.shape[1]
    e, two_i, k = qw_gate_up.shape
    inter = two_i // 2
    _need(x, torch.bfloat16, (t, hid), "x")
    _need(logits, torch.float32, (t, e_r), "logits")
    if e != e_r + n_shared or k != hid:
        raise ValueError("expert weights do not match the routing or the hidden size")
    _need(qw_gate_up, torch.int8, (e, two_i, hid), "qw_gate_up")
    _need(sw_gate_up, torch.float32, (e, two_i), "sw_gate_up")
    _need(qw_down, torch.int8, (e, hid, inter), "qw_down")
    _need(sw_down, torch.float32, (e, hid), "sw_down")
    if out is None:
        out = torch.empty((t, hid), dtype=torch.bfloat16, device=x.device)
    _need(out, torch.bfloat16, (t, hid), "out")
    _check(lib().moe_expert_mlp_w8a16(_ptr(x), _ptr(logits), e_r, top_k, n_shared, _ptr(qw_gate_up),
                                      _ptr(sw_gate_up), _ptr(qw_down), _ptr(sw_down), _ptr(out), t, hid, inter,
                                      _stream(stream)), "moe_expert_mlp_w8a16")
    return out
