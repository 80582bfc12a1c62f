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


@pytest.mark.parametrize("case", range(CASES))
def test_w8a8_linear_random(case):
    """The linear layer (its quantization inside the call: one launch, two,
    or the tensor-core path's fp16 codes, by shape) equals the two calls bit
    for bit and the oracle's codes and scales."""
    m, n, k = _shape(6000 + case, 300, 600, 16, 160)
    if case % 4 == 0:
        m = 1 + case % 8  # the one-launch range
    x = synthetic.activations(m, k, 130 + case)
    qw, sw = oracle.quant_rows(util.bits(synthetic.weight(n, k, 140 + case)))
    qw_d, sw_d = torch.from_numpy(qw).cuda(), torch.from_numpy(sw).cuda()
    qx = torch.empty((m, k), dtype=torch.int8, device="cuda")
    sx = torch.empty((m,), dtype=torch.float32, device="cuda")
    y = capi.w8a8_linear(x.cuda(), qw_d, sw_d, qx=qx, sx=sx)
    q2, s2 = capi.quantize_act_per_token_int8(x.cuda())
    y2 = capi.w8a8_gemm(q2, s2, qw_d, sw_d)
    torch.cuda.synchronize()
    qx_ref, sx_ref = oracle.quant_rows(util.bits(x))
    assert np.array_equal(qx.cpu().numpy(), qx_ref) and np.array_equal(sx.cpu().numpy(), sx_ref)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), (m, n, k)


@pytest.mark.parametrize("case", range(CASES // 2))
def test_moe_layer_random(case):
    """Random MoE layers (experts, top-k, shared experts, tokens, widths):
    the routing is bit-exact, the layer equals its four stages called one by
    one, and the whole chain is within the three stages' bars of the fp64
    oracle chain."""
    g = np.random.default_rng(7000 + case)
    e_r = int(g.integers(1, 65))
    topk = int(g.integers(1, min(8, e_r) + 1))
    shared = int(g.integers(0, 3))
    tokens = int(g.integers(1, 101))
    hid = 16 * int(g.integers(1, 33))
    inter = 16 * int(g.integers(1, 33))
    e_all = e_r + shared
    qgu = np.empty((e_all, 2 * inter, hid), np.int8)
    sgu = np.empty((e_all, 2 * inter), np.float32)
    qd = np.empty((e_all, hid, inter), np.int8)
    sd = np.empty((e_all, hid), np.float32)
    for e in range(e_all):
        qgu[e], sgu[e] = oracle.quant_rows(util.bits(synthetic.weight(2 * inter, hid, 300 + 70 * case + e)))
        qd[e], sd[e] = oracle.quant_rows(util.bits(synthetic.weight(hid, inter, 900 + 70 * case + e)))
    x = synthetic.activations(tokens, hid, 150 + case)
    logits = synthetic.gate_logits(tokens, e_r, 160 + case).numpy()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    off, row_token, token_row, w = capi.moe_route_topk(dev(logits), topk, shared)
    ref = oracle.moe_route(logits, topk, shared)
    torch.cuda.synchronize()
    assert np.array_equal(off.cpu().numpy(), ref.offsets)
    assert np.array_equal(row_token.cpu().numpy(), ref.row_token)
    assert np.array_equal(token_row.cpu().numpy(), ref.token_row)
    h = capi.grouped_w8a16_silu_mul(x.cuda(), row_token, off, dev(qgu), dev(sgu))
    yd = capi.grouped_w8a16_gemm(h, off, dev(qd), dev(sd))
    staged = capi.moe_combine(yd, token_row, w)
    out = capi.moe_expert_mlp_w8a16(x.cuda(), dev(logits), topk, shared, dev(qgu), dev(sgu), dev(qd), dev(sd))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), staged.view(torch.int16))
    xg = util.bits(x)[ref.row_token]
    h64 = oracle.silu_mul(oracle.grouped_w8a16(xg, ref.offsets, qgu, sgu))
    yd64 = np.zeros((h64.shape[0], hid))
    for e in range(e_all):
        a, b = ref.offsets[e], ref.offsets[e + 1]
        if b > a:
            yd64[a:b] = h64[a:b] @ (qd[e].astype(np.float64) * sd[e][:, None].astype(np.float64)).T
    out64 = oracle.moe_combine(yd64, ref.token_row, ref.slot_weight)
    got = util.from_bits(util.bits(out.cpu())).double().numpy()
    assert util.rel_frobenius(got, out64) <= util.frob_bar(out64, 6e-3), (e_r, topk, shared, tokens, hid, inter)
