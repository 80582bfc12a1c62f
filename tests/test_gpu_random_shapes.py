"""Seeded random shapes for every GEMM family, through the C ABI, against
the oracle: the launch planners (decode or tensor-core W8A8 and its tile
widths, split-K and CTA pairs; FP8 tile widths, split-K clusters and pairs;
grouped slot mappings) meet shapes nobody picked by hand, ragged in every
dimension.  Bars as in the per-family test files: int8 accumulators
bit-exact, W8A8 outputs within one bf16 ulp, the others within their
accumulation bound plus one bf16 rounding (and the relative Frobenius bar
on outputs of at least 1,024 elements).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from int8_quantized_linear_gb300 import capi, synthetic
from tests import util
from tests.test_gpu_fp8 import _fp8_codes
from tests.test_gpu_fp8 import check_gemm as check_fp8_gemm
from tests.test_gpu_parity import _abs_inputs, _points, check_elementwise, gpu_grouped, gpu_w8a8, gpu_w8a16
from tests.test_gpu_w4 import check_gemm as check_w4_gemm

pytestmark = pytest.mark.gpu

CASES = 32


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    from int8_quantized_linear_gb300 import build
    build.build()
    capi.lib()
    assert capi.i8ql_get_device_error() == capi.I8QL_OK
    yield
    assert capi.i8ql_get_device_error() == capi.I8QL_OK


def _shape(seed, m_max, n_max, k_unit, k_units):
    g = np.random.default_rng(seed)
    return int(g.integers(1, m_max + 1)), int(g.integers(1, n_max + 1)), k_unit * int(g.integers(1, k_units + 1))


@pytest.mark.parametrize("case", range(CASES))
def test_w8a8_random(case):
    m, n, k = _shape(1000 + case, 300, 700, 16, 200)
    qx, sx = oracle.quant_rows(util.bits(synthetic.activations(m, k, case)))
    qw, sw = oracle.quant_rows(util.bits(synthetic.weight(n, k, 50 + case)))
    bias = util.bits(synthetic.bias(n, case)) if case % 2 else None
    acc, y = gpu_w8a8(qx, sx, qw, sw, bias)
    pm, pn = (a.ravel() for a in np.meshgrid(np.arange(m), np.arange(n), indexing="ij"))
    if pm.size > 20000:
        pm, pn = _points(m, n, 3000, case)
    ref_acc, _, ref_y = oracle.w8a8_points(qx, sx, qw, sw, bias, pm, pn)
    assert np.array_equal(acc[pm, pn].astype(np.int64), ref_acc), (m, n, k)
    assert util.max_ulp_diff(y[pm, pn], ref_y) <= 1, (m, n, k)


@pytest.mark.parametrize("case", range(CASES))
def test_w8a16_random(case):
    m, n, k = _shape(2000 + case, 64, 700, 16, 200)
    qw, sw = oracle.quant_rows(util.bits(synthetic.weight(n, k, 60 + case)))
    x = synthetic.activations(m, k, 70 + case)
    y = gpu_w8a16(x, qw, sw)
    xb = util.bits(x)
    ref = oracle.w8a16(xb, qw, sw)
    if ref.size >= 1024:
        assert util.rel_frobenius(y, ref) <= util.frob_bar(ref, 2e-3), (m, n, k)
    ax, aq = _abs_inputs(xb, qw)
    check_elementwise(y, ref, oracle.w8a16(ax, aq, sw), k)


@pytest.mark.parametrize("case", range(CASES))
def test_fp8_random(case):
    m, n, k = _shape(3000 + case, 300, 700, 16, 250)
    qx, sx = _fp8_codes(m, k, 80 + case)
    qw, sw = _fp8_codes(n, k, 90 + case, 0.02)
    bias = util.bits(synthetic.bias(n, case)) if case % 2 == 0 else None
    pm = pn = None
    if m * n > 20000:
        pm, pn = _points(m, n, 3000, case)
    check_fp8_gemm(qx, sx, qw, sw, bias, pm, pn)


@pytest.mark.parametrize("case", range(CASES))
def test_w4a16_random(case):
    m, n, k = _shape(4000 + case, 64, 400, 128, 16)
    q, s = oracle.quant_w4_g128(util.bits(synthetic.weight(n, k, 100 + case)))
    check_w4_gemm(synthetic.activations(m, k, 110 + case), q, s)


@pytest.mark.parametrize("case", range(CASES))
def test_grouped_random(case):
    g = np.random.default_rng(5000 + case)
    e_count = int(g.integers(1, 41))
    n = int(g.integers(16, 301))
    k = 16 * int(g.integers(1, 101))
    counts = g.integers(0, 5, e_count) * (g.random(e_count) < 0.6)  # many empty experts
    heavy = g.random(e_count) < 0.1
    counts = np.where(heavy, g.integers(9, 70, e_count), counts)
    if counts.sum() == 0:
        counts[-1] = 1
    off = np.zeros(e_count + 1, np.int32)
    off[1:] = np.cumsum(counts)
    q = np.empty((e_count, n, k), np.int8)
    s = np.empty((e_count, n), np.float32)
    for e in range(e_count):
        q[e], s[e] = oracle.quant_rows(util.bits(synthetic.weight(n, k, 200 + 41 * case + e)))
    x = synthetic.activations(int(off[-1]), k, 120 + case)
    y = gpu_grouped(x, off, q, s)
    assert capi.i8ql_get_device_error() == capi.I8QL_OK
    xb = util.bits(x)
    ref = oracle.grouped_w8a16(xb, off, q, s)
    if ref.size >= 1024:
        assert util.rel_frobenius(y, ref) <= util.frob_bar(ref, 2e-3), (e_count, n, k, counts.tolist())
    ax, aq = _abs_inputs(xb, q)
    check_elementwise(y, ref, oracle.grouped_w8a16(ax, off, aq, s), k)
