"""ctypes front end of the C oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by the smoke check and by
the CPU baseline leg of ``bench.py``; never by the product path.  Arrays
are numpy; bf16 values travel as their raw ``uint16`` bit patterns.
"""

from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

_LIB = None

_ERRORS = {
    1: "non-finite input",
    2: "bad argument",
    3: "accumulator outside int32",
    4: "bad group offsets",
    5: "a nonzero group's scale underflows bf16",
}


def load(path: str):
    """Open an oracle build at ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_quant_rows.argtypes = [p, i64, i64, p, p]
    lib.oracle_int_acc.argtypes = [p, p, i64, i64, i64, p]
    lib.oracle_w8a8_epilogue.argtypes = [p, p, p, p, i64, i64, p, p]
    lib.oracle_w8a8_points.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, p, p, p, p]
    lib.oracle_w8a16.argtypes = [p, p, p, i64, i64, i64, p]
    lib.oracle_w8a16_points.argtypes = [p, p, p, i64, i64, i64, i64, p, p, p]
    lib.oracle_grouped_w8a16.argtypes = [p, p, i64, p, p, i64, i64, i64, p]
    lib.oracle_narrow_bf16.argtypes = [p, i64, p]
    lib.oracle_narrow_bf16.restype = None
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_fp8_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_fp8_decode.restype = ctypes.c_float
    lib.oracle_fp8_encode.argtypes = [ctypes.c_float]
    lib.oracle_fp8_encode.restype = ctypes.c_uint8
    lib.oracle_fp8_encode_array.argtypes = [p, i64, p]
    lib.oracle_fp8_encode_array.restype = None
    lib.oracle_fp8_decode_array.argtypes = [p, i64, p]
    lib.oracle_fp8_decode_array.restype = None
    lib.oracle_quant_rows_fp8.argtypes = [p, i64, i64, p, p]
    lib.oracle_w8a8_fp8_points.argtypes = [p, p, p, p, p, i64, i64, i64, i64, p, p, p, p]
    lib.oracle_quant_w4_g128.argtypes = [p, i64, i64, p, p]
    lib.oracle_w4_unpack.argtypes = [p, i64, i64, p]
    lib.oracle_w4_unpack.restype = None
    lib.oracle_w4a16.argtypes = [p, p, p, i64, i64, i64, p]
    lib.oracle_moe_route.argtypes = [p, i64, i64, i64, i64, p, p, p, p, p]
    lib.oracle_silu_mul.argtypes = [p, i64, i64, p]
    lib.oracle_silu_mul.restype = None
    lib.oracle_moe_combine.argtypes = [p, p, p, i64, i64, i64, p]
    lib.oracle_moe_combine.restype = None
    return lib


def _lib():
    global _LIB
    if _LIB is None:
        _LIB = load(_build.build())
    return _LIB


class OracleError(RuntimeError):
    pass


def _check(rc: int) -> None:
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"oracle error {rc}"))


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def quant_rows(src_bf16):
    """Per-row symmetric int8 codes and fp32 scales of a bf16 [R, K] array."""
    src = _c(src_bf16, np.uint16)
    rows, k = src.shape
    q = np.empty((rows, k), np.int8)
    s = np.empty((rows,), np.float32)
    _check(_lib().oracle_quant_rows(_ptr(src), rows, k, _ptr(q), _ptr(s)))
    return q, s


def int_acc(qx, qw) -> np.ndarray:
    """Exact int64 accumulator sum_k qx[m,k] * qw[n,k]."""
    qx, qw = _c(qx, np.int8), _c(qw, np.int8)
    m, k = qx.shape
    n, k2 = qw.shape
    assert k == k2
    acc = np.empty((m, n), np.int64)
    _check(_lib().oracle_int_acc(_ptr(qx), _ptr(qw), m, n, k, _ptr(acc)))
    return acc


def w8a8_epilogue(acc, sx, sw, bias_bf16=None):
    """fp32 epilogue values and their bf16 (RNE) bits for an int64 acc."""
    acc = _c(acc, np.int64)
    m, n = acc.shape
    sx, sw = _c(sx, np.float32), _c(sw, np.float32)
    b = None if bias_bf16 is None else _c(bias_bf16, np.uint16)
    f = np.empty((m, n), np.float32)
    y = np.empty((m, n), np.uint16)
    _check(_lib().oracle_w8a8_epilogue(_ptr(acc), _ptr(sx), _ptr(sw), _ptr(b), m, n,
                                       _ptr(f), _ptr(y)))
    return f, y


def w8a8(qx, sx, qw, sw, bias_bf16=None):
    """Full W8A8 layer: (int64 acc, fp32 epilogue, bf16 bits)."""
    acc = int_acc(qx, qw)
    f, y = w8a8_epilogue(acc, sx, sw, bias_bf16)
    return acc, f, y


def w8a8_points(qx, sx, qw, sw, bias_bf16, pm, pn):
    """W8A8 at output points (pm[i], pn[i]): (acc, f, y) per point."""
    qx, qw = _c(qx, np.int8), _c(qw, np.int8)
    m, k = qx.shape
    n = qw.shape[0]
    sx, sw = _c(sx, np.float32), _c(sw, np.float32)
    b = None if bias_bf16 is None else _c(bias_bf16, np.uint16)
    pm, pn = _c(pm, np.int64), _c(pn, np.int64)
    cnt = pm.shape[0]
    acc = np.empty(cnt, np.int64)
    f = np.empty(cnt, np.float32)
    y = np.empty(cnt, np.uint16)
    _check(_lib().oracle_w8a8_points(_ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), _ptr(b), m, n, k,
                                     cnt, _ptr(pm), _ptr(pn), _ptr(acc), _ptr(f), _ptr(y)))
    return acc, f, y


def w8a16(x_bf16, q, s) -> np.ndarray:
    """fp64 dequantize-then-matmul y[m,n] = sum_k (s[n] q[n,k]) x[m,k]."""
    x = _c(x_bf16, np.uint16)
    q, s = _c(q, np.int8), _c(s, np.float32)
    m, k = x.shape
    n = q.shape[0]
    y = np.empty((m, n), np.float64)
    _check(_lib().oracle_w8a16(_ptr(x), _ptr(q), _ptr(s), m, n, k, _ptr(y)))
    return y


def w8a16_points(x_bf16, q, s, pm, pn) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    q, s = _c(q, np.int8), _c(s, np.float32)
    m, k = x.shape
    n = q.shape[0]
    pm, pn = _c(pm, np.int64), _c(pn, np.int64)
    y = np.empty(pm.shape[0], np.float64)
    _check(_lib().oracle_w8a16_points(_ptr(x), _ptr(q), _ptr(s), m, n, k, pm.shape[0],
                                      _ptr(pm), _ptr(pn), _ptr(y)))
    return y


def grouped_w8a16(x_bf16, offsets, q, s) -> np.ndarray:
    """Grouped W8A16: rows offsets[e]..offsets[e+1] use expert e."""
    x = _c(x_bf16, np.uint16)
    off = _c(offsets, np.int32)
    q, s = _c(q, np.int8), _c(s, np.float32)
    t, k = x.shape
    e, n, k2 = q.shape
    assert k == k2 and off.shape[0] == e + 1
    y = np.empty((t, n), np.float64)
    _check(_lib().oracle_grouped_w8a16(_ptr(x), _ptr(off), e, _ptr(q), _ptr(s), t, n, k,
                                       _ptr(y)))
    return y


def narrow_bf16(f32) -> np.ndarray:
    """binary32 -> bf16 bits, round to nearest even."""
    f = _c(f32, np.float32)
    out = np.empty(f.shape, np.uint16)
    _lib().oracle_narrow_bf16(_ptr(f), f.size, _ptr(out))
    return out


def widen_bf16(bits) -> np.ndarray:
    """bf16 bits -> float32 (exact)."""
    return (_c(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def set_threads(n: int = 0) -> int:
    """Threads of the oracle's row loops (n <= 0: keep the current count);
    returns the count in effect (1 in a build without OpenMP)."""
    return int(_lib().oracle_set_threads(int(n)))


# ---------------------------------------------------------------- FP8 E4M3

def fp8_encode(v) -> np.ndarray:
    """E4M3 codes (uint8) of fp32 values: nearest, ties to even, saturating."""
    f = _c(v, np.float32)
    out = np.empty(f.shape, np.uint8)
    _lib().oracle_fp8_encode_array(_ptr(f), f.size, _ptr(out))
    return out


def fp8_decode(c) -> np.ndarray:
    """fp32 values of E4M3 codes (exact)."""
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float32)
    _lib().oracle_fp8_decode_array(_ptr(c), c.size, _ptr(out))
    return out


def quant_rows_fp8(src_bf16):
    """Per-row E4M3 codes (uint8) and fp32 scales (absmax / 448) of bf16 [R, K]."""
    src = _c(src_bf16, np.uint16)
    rows, k = src.shape
    q = np.empty((rows, k), np.uint8)
    s = np.empty((rows,), np.float32)
    _check(_lib().oracle_quant_rows_fp8(_ptr(src), rows, k, _ptr(q), _ptr(s)))
    return q, s


def w8a8_fp8_points(qx, sx, qw, sw, bias_bf16, pm, pn):
    """FP8 W8A8 at output points: (exact fp64 dot products, fp64 outputs)."""
    qx, qw = _c(qx, np.uint8), _c(qw, np.uint8)
    m, k = qx.shape
    n = qw.shape[0]
    sx, sw = _c(sx, np.float32), _c(sw, np.float32)
    b = None if bias_bf16 is None else _c(bias_bf16, np.uint16)
    pm, pn = _c(pm, np.int64), _c(pn, np.int64)
    acc = np.empty(pm.shape[0], np.float64)
    y = np.empty(pm.shape[0], np.float64)
    _check(_lib().oracle_w8a8_fp8_points(_ptr(qx), _ptr(sx), _ptr(qw), _ptr(sw), _ptr(b), m, n, k,
                                         pm.shape[0], _ptr(pm), _ptr(pn), _ptr(acc), _ptr(y)))
    return acc, y


def w8a8_fp8(qx, sx, qw, sw, bias_bf16=None):
    """FP8 W8A8 over the whole [M, N] output: (exact acc, fp64 y)."""
    m, n = np.asarray(qx).shape[0], np.asarray(qw).shape[0]
    pm, pn = np.meshgrid(np.arange(m), np.arange(n), indexing="ij")
    acc, y = w8a8_fp8_points(qx, sx, qw, sw, bias_bf16, pm.ravel(), pn.ravel())
    return acc.reshape(m, n), y.reshape(m, n)


# ---------------------------------------------------------------- W4A16, group 128

def quant_w4_g128(src_bf16):
    """Packed int4 codes [R, K/2] (uint8) and bf16 group scales [R, K/128]."""
    src = _c(src_bf16, np.uint16)
    rows, k = src.shape
    packed = np.empty((rows, k // 2), np.uint8)
    scale = np.empty((rows, k // 128), np.uint16)
    _check(_lib().oracle_quant_w4_g128(_ptr(src), rows, k, _ptr(packed), _ptr(scale)))
    return packed, scale


def w4_unpack(packed, k):
    """Signed codes [R, K] of packed int4 storage."""
    packed = _c(packed, np.uint8)
    rows = packed.shape[0]
    codes = np.empty((rows, k), np.int8)
    _lib().oracle_w4_unpack(_ptr(packed), rows, k, _ptr(codes))
    return codes


def w4a16(x_bf16, packed, scale) -> np.ndarray:
    """fp64 dequantize-then-matmul of the group-128 int4 weights."""
    x = _c(x_bf16, np.uint16)
    packed, scale = _c(packed, np.uint8), _c(scale, np.uint16)
    m, k = x.shape
    n = packed.shape[0]
    y = np.empty((m, n), np.float64)
    _check(_lib().oracle_w4a16(_ptr(x), _ptr(packed), _ptr(scale), m, n, k, _ptr(y)))
    return y


# ---------------------------------------------------------------- MoE expert MLP

class Route:
    """Routing of T tokens: sel/prob [T, topk], offsets [E + shared + 1],
    row_token [rows], token_row [T, topk + shared], row_weight [rows]."""

    def __init__(self, sel, prob, offsets, row_token, token_row, shared):
        self.sel, self.prob, self.offsets = sel, prob, offsets
        self.row_token, self.token_row = row_token, token_row
        t, topk = sel.shape
        self.slot_weight = np.concatenate([prob, np.ones((t, shared))], axis=1)  # [T, topk + shared]
        self.row_weight = np.empty(row_token.shape[0], np.float64)
        self.row_weight[token_row.ravel()] = self.slot_weight.ravel()


def moe_route(logits, topk, shared) -> Route:
    lg = _c(logits, np.float32)
    t, e = lg.shape
    s = topk + shared
    sel = np.empty((t, topk), np.int32)
    prob = np.empty((t, topk), np.float64)
    offsets = np.empty(e + shared + 1, np.int32)
    row_token = np.empty(t * s, np.int32)
    token_row = np.empty((t, s), np.int32)
    _check(_lib().oracle_moe_route(_ptr(lg), t, e, topk, shared, _ptr(sel), _ptr(prob), _ptr(offsets),
                                   _ptr(row_token), _ptr(token_row)))
    return Route(sel, prob, offsets, row_token, token_row, shared)


def silu_mul(gu) -> np.ndarray:
    """h = silu(gate) * up of a fused [rows, 2I] gate/up output (fp64)."""
    gu = _c(gu, np.float64)
    rows, two_i = gu.shape
    h = np.empty((rows, two_i // 2), np.float64)
    _lib().oracle_silu_mul(_ptr(gu), rows, two_i // 2, _ptr(h))
    return h


def moe_combine(yd, token_row, slot_weight) -> np.ndarray:
    """out[t] = sum_s w[t, s] * yd[token_row[t, s]] (fp64)."""
    yd = _c(yd, np.float64)
    tr = _c(token_row, np.int32)
    w = _c(slot_weight, np.float64)
    t, s = tr.shape
    h = yd.shape[1]
    out = np.empty((t, h), np.float64)
    _lib().oracle_moe_combine(_ptr(yd), _ptr(tr), _ptr(w), t, s, h, _ptr(out))
    return out
