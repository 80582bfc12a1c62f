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
