"""GPU parity of the FP8 E4M3 path (quantization and the tcgen05
kind::f8f6f4 GEMM) against the CPU oracle, through the C ABI.

Bars:
 * E4M3 codes and fp32 scales: bit-exact.
 * GEMM outputs: every product of two E4M3 values is exact in fp32, so the
   GPU differs from the oracle's exact fp64 result only by fp32
   accumulation and the epilogue's roundings: per element
   |y - y_exact| <= K * 2^-23 * sum_k |p_k| * sx * sw + 2^-8 * |y_exact|
   (any accumulation order, then one bf16 rounding), and the relative
   Frobenius error of the output stays within 2e-3.  With small-integer
   codes every partial sum is an integer below 2^24, so the accumulator is
   exact and the output must be within one bf16 ulp of the fp32 epilogue
   of the exact sum.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from int8_quantized_linear_gb300 import capi, synthetic
from tests import util
from tests.golden import load as golden

pytestmark = pytest.mark.gpu

FROB = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    from int8_quantized_linear_gb300 import build
    build.build()
    capi.lib()
    assert capi.i8ql_get_device_error() == capi.I8QL_OK
    yield
    assert capi.i8ql_get_device_error() == capi.I8QL_OK


def _gpu_quant(src_bf16: torch.Tensor, weight: bool):
    rows, k = src_bf16.shape
    qbuf, q = util.guarded((rows, k), torch.uint8, "cuda", 0x7F)
    sbuf, s = util.guarded((rows,), torch.float32, "cuda", -3.0)
    fn = capi.quantize_weight_per_channel_fp8 if weight else capi.quantize_act_per_token_fp8
    fn(src_bf16.cuda(), q=q, scale=s)
    torch.cuda.synchronize()
    assert util.guard_intact(qbuf, rows * k, 0x7F) and util.guard_intact(sbuf, rows, -3.0)
    return q.cpu().numpy(), s.cpu().numpy()


def check_quant(src_bf16: torch.Tensor, weight: bool = True):
    q, s = _gpu_quant(src_bf16, weight)
    q_ref, s_ref = oracle.quant_rows_fp8(util.bits(src_bf16))
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32)), "scales differ"
    bad = np.argwhere(q != q_ref)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:3].tolist()}: " \
        f"{[(hex(q[i, j]), hex(q_ref[i, j])) for i, j in bad[:3]]}"
    return q, s


@pytest.mark.parametrize("case", golden.fp8_rows(), ids=lambda c: c[0])
def test_fp8_quant_golden_rows_on_gpu(case):
    name, row, scale, codes = case
    vals = np.zeros((1, 16), np.float64)
    vals[0, :len(row)] = row
    src = torch.tensor(vals, dtype=torch.float64).to(torch.bfloat16)
    for weight in (True, False):
        q, s = _gpu_quant(src, weight)
        assert s[0] == np.float32(scale), name
        assert q[0, :len(codes)].tolist() == codes, name


def _adversarial(rows, k, seed):
    w = synthetic.weight(rows, k, seed).float()
    g = torch.Generator().manual_seed(seed)
    w[0] = 0.0
    if rows > 2:
        w[1] *= 1e-35  # tiny and subnormal magnitudes keep their full grid
    if rows > 3:
        w[2] = torch.randint(-64, 65, (k,), generator=g).float() * 0.0625  # many exact midpoints
        w[2, 0] = 448.0
    return w.to(torch.bfloat16)


@pytest.mark.parametrize("rows,k", [(1, 16), (3, 48), (33, 1040), (129, 4096), (7, 12288), (5, 16400),
                                    (300, 256), (1000, 2560), (4100, 2992), (40, 9744)])
def test_fp8_quant_shapes(rows, k):
    check_quant(_adversarial(rows, k, rows * 7 + k), True)
    check_quant(synthetic.activations(rows, k, rows + k), False)


def test_fp8_quant_full_size():
    n, k = synthetic.QWEN3_4B_SHAPES["gate_up"]
    check_quant(synthetic.weight(n, k, 1), True)
    check_quant(synthetic.activations(4096, 2560, 2), False)


# ------------------------------------------------------------------ GEMM

def _gpu_gemm(qx, sx, qw, sw, bias_bits=None):
    m, n = qx.shape[0], qw.shape[0]
    ybuf, y = util.guarded((m, n), torch.int16, "cuda", 0x7F7F)
    bias = None if bias_bits is None else util.from_bits(bias_bits, "cuda")
    capi.w8a8_fp8_gemm(torch.from_numpy(qx).cuda(), torch.from_numpy(sx).cuda(), torch.from_numpy(qw).cuda(),
                       torch.from_numpy(sw).cuda(), bias=bias, y=y.view(torch.bfloat16))
    torch.cuda.synchronize()
    assert util.guard_intact(ybuf, m * n, 0x7F7F)
    return y.cpu().numpy().view(np.uint16)


def _bound(qx, sx, qw, sw, pm, pn, k):
    """K * 2^-23 * sum_k |products| * |sx sw| at the points (magnitudes from
    the oracle applied to the codes' absolute values)."""
    mag, _ = oracle.w8a8_fp8_points(qx & np.uint8(0x7F), np.ones_like(sx), qw & np.uint8(0x7F),
                                    np.ones_like(sw), None, pm, pn)
    return mag * np.abs(sx[pm].astype(np.float64) * sw[pn]) * (k * 2.0 ** -23)


def check_gemm(qx, sx, qw, sw, bias_bits=None, pm=None, pn=None):
    m, k = qx.shape
    n = qw.shape[0]
    y = oracle.widen_bf16(_gpu_gemm(qx, sx, qw, sw, bias_bits)).astype(np.float64)
    if pm is None and m * n <= 65536:
        pm, pn = (a.ravel() for a in np.meshgrid(np.arange(m), np.arange(n), indexing="ij"))
    elif pm is None:
        g = np.random.default_rng(m * n + k)
        pm = np.concatenate([g.integers(0, m, 4000), [0, m - 1, m - 1, 0]])
        pn = np.concatenate([g.integers(0, n, 4000), [0, n - 1, 0, n - 1]])
    _, ref = oracle.w8a8_fp8_points(qx, sx, qw, sw, bias_bits, pm, pn)
    got = y[pm, pn]
    assert util.rel_frobenius(got, ref) <= util.frob_bar(ref, FROB)
    bound = _bound(qx, sx, qw, sw, pm, pn, k) + np.abs(ref) * 2.0 ** -8 + 1e-30
    worst = np.argmax(np.abs(got - ref) - bound)
    assert np.all(np.abs(got - ref) <= bound), (pm[worst], pn[worst], got[worst], ref[worst], bound[worst])
    return y


def _fp8_codes(rows, k, seed, scale=1.0):
    """E4M3 codes of a seeded N(0, scale) matrix (through the oracle)."""
    g = torch.Generator().manual_seed(seed)
    v = (torch.randn(rows, k, generator=g) * scale).to(torch.bfloat16)
    return oracle.quant_rows_fp8(util.bits(v))


def _scales(n, seed, lo=1e-4, hi=2e-2):
    g = np.random.default_rng(seed)
    return (lo + (hi - lo) * g.random(n)).astype(np.float32)


def test_fp8_gemm_small_integers_exact():
    """Codes of +-1 .. +-16 (products are integers up to 256, every partial
    sum an integer below 2^24): the fp32 accumulator is exact, so the output
    is the fp32 epilogue of the exact sum to within one bf16 ulp.  This pins
    the operand layout, descriptors and tile edges (ragged M, N, K, down to a
    single output channel)."""
    ints = np.arange(1, 17, dtype=np.float32)
    codes = oracle.fp8_encode(ints)
    assert np.array_equal(oracle.fp8_decode(codes), ints)
    for (m, n, k) in [(1, 16, 16), (7, 40, 48), (129, 300, 1040), (256, 256, 4096), (300, 513, 2064),
                      (64, 640, 4096), (128, 520, 9728), (1, 1, 16), (40, 1, 16), (300, 3, 64),
                      (2048, 5, 128)]:
        g = np.random.default_rng(m + n + k)
        qx = codes[g.integers(0, 16, (m, k))] | (g.integers(0, 2, (m, k)) * 0x80).astype(np.uint8)
        qw = codes[g.integers(0, 16, (n, k))] | (g.integers(0, 2, (n, k)) * 0x80).astype(np.uint8)
        sx, sw = _scales(m, m, 0.5, 1.0), _scales(n, n, 1e-3, 1e-2)
        bias = util.bits(synthetic.bias(n, n)) if m % 2 else None
        y = _gpu_gemm(qx, sx, qw, sw, bias)
        pm, pn = (a.ravel() for a in np.meshgrid(np.arange(m), np.arange(n), indexing="ij"))
        acc, _ = oracle.w8a8_fp8_points(qx, sx, qw, sw, None, pm, pn)
        assert np.all(np.abs(acc) < 2 ** 24)
        f = (acc.astype(np.float32) * sx[pm]).astype(np.float32) * sw[pn]
        f = f.astype(np.float32)
        if bias is not None:
            f = (f + oracle.widen_bf16(bias)[pn]).astype(np.float32)
        want = oracle.narrow_bf16(f)
        assert util.max_ulp_diff(y[pm, pn], want) <= 1, (m, n, k)


@pytest.mark.parametrize("m,n,k", [(1, 256, 1024), (7, 300, 2064), (64, 513, 1040), (128, 200, 4096),
                                   (129, 2560, 2560), (300, 1000, 4160), (512, 768, 9728)])
def test_fp8_gemm_shapes(m, n, k):
    qx, sx = _fp8_codes(m, k, m + k)
    qw, sw = _fp8_codes(n, k, n + 2 * k, 0.02)
    bias = util.bits(synthetic.bias(n, n + 1)) if (m + n) % 2 else None
    check_gemm(qx, sx, qw, sw, bias)


@pytest.mark.parametrize("m,n,k", [(300, 1000, 2560), (2048, 512, 1024), (64, 24, 512)])
def test_fp8_gemm_unaligned_scales_and_bias(m, n, k):
    """Weight scales and bias that start off a 16-byte boundary (4- and
    2-byte aligned, the least the boundary allows) give, bit for bit, the
    output of the call with 16-byte-aligned copies, for several launch
    forms (CTA pairs, single CTAs)."""
    qx, sx = _fp8_codes(m, k, m + 1)
    qw, sw = _fp8_codes(n, k, n + 2, 0.02)
    bias = synthetic.bias(n, n + 3).cuda()
    qx_d, sx_d, qw_d = (torch.from_numpy(a).cuda() for a in (qx, sx, qw))
    sw_al = torch.from_numpy(sw).cuda()
    sw_buf = torch.zeros(n + 1, dtype=torch.float32, device="cuda")
    sw_buf[1:] = sw_al
    b_buf = torch.zeros(n + 1, dtype=torch.bfloat16, device="cuda")
    b_buf[1:] = bias
    y_al = capi.w8a8_fp8_gemm(qx_d, sx_d, qw_d, sw_al, bias=bias)
    y_un = capi.w8a8_fp8_gemm(qx_d, sx_d, qw_d, sw_buf[1:], bias=b_buf[1:])
    y_nb = capi.w8a8_fp8_gemm(qx_d, sx_d, qw_d, sw_buf[1:])
    y_nb_al = capi.w8a8_fp8_gemm(qx_d, sx_d, qw_d, sw_al)
    torch.cuda.synchronize()
    assert torch.equal(y_al.view(torch.int16), y_un.view(torch.int16))
    assert torch.equal(y_nb.view(torch.int16), y_nb_al.view(torch.int16))


@pytest.mark.parametrize("m,n,k", [(3, 40, 131072), (130, 257, 65552)])
def test_fp8_gemm_longest_k(m, n, k):
    """The longest K the exact oracle covers (2^17 products: its fp64 sum of
    multiples of 2^-18 below 2^18 is exact up to there), and a long K on the
    split-K path: the fp32 accumulation over the whole range stays within
    its bound."""
    qx, sx = _fp8_codes(m, k, m + 3)
    qw, sw = _fp8_codes(n, k, n + 4, 0.02)
    pm, pn = (a.ravel() for a in np.meshgrid(np.arange(m), np.arange(n), indexing="ij"))
    if pm.size > 4000:
        g = np.random.default_rng(k)
        pm, pn = g.integers(0, m, 4000), g.integers(0, n, 4000)
    check_gemm(qx, sx, qw, sw, None, pm, pn)


def test_fp8_plans_cover_split_k_tile_widths_and_pairs():
    """The prefill shapes exercise every launch form: split-K clusters of
    single CTAs at both tile widths (few tiles), persistent single CTAs, and
    CTA pairs with 256- and 192-wide tiles."""
    plans = {capi.i8ql_fp8_plan(m, n, k) for m in (1, 64, 128, 512, 2048, 4096)
             for n, k in synthetic.QWEN3_4B_SHAPES.values()}
    assert any(s > 1 and t == 128 for t, s, _ in plans), plans
    assert any(s > 1 and t == 256 for t, s, _ in plans), plans
    assert any(s == 1 and p == 0 for _, s, p in plans), plans
    assert any(p == 1 and t == 256 for t, _, p in plans), plans
    assert any(p == 1 and t == 192 for t, _, p in plans), plans
    assert all(s == 1 for _, s, p in plans if p == 1)
    for m, n, k in [(1, 2560, 9728), (128, 2560, 2560), (128, 2560, 9728)]:
        assert capi.i8ql_fp8_plan(m, n, k)[1] > 1, (m, n, k)


@pytest.mark.parametrize("m", [128, 512, 2048])
@pytest.mark.parametrize("shape", list(synthetic.QWEN3_4B_SHAPES))
def test_fp8_gemm_qwen3_4b_prefill_sampled(shape, m):
    """Qwen3-4B prefill shapes (outlier weights and activation channels),
    bias on, sampled outputs against the exact oracle; M = 128 and 512 run
    split-K clusters, M = 2048 CTA pairs (192-wide tiles for N = 2560)."""
    n, k = synthetic.QWEN3_4B_SHAPES[shape]
    qw, sw = oracle.quant_rows_fp8(util.bits(synthetic.weight(n, k, 1)))
    qx, sx = oracle.quant_rows_fp8(util.bits(synthetic.activations(m, k, 2)))
    bias = util.bits(synthetic.bias(n, 3))
    g = np.random.default_rng(n + m)
    pm = np.concatenate([g.integers(0, m, 3000), [0, m - 1]])
    pn = np.concatenate([g.integers(0, n, 3000), [n - 1, 0]])
    check_gemm(qx, sx, qw, sw, bias, pm, pn)


@pytest.mark.parametrize("m,n,k", [(1, 256, 1024), (64, 513, 1040), (300, 1000, 4160), (2048, 2560, 2560)])
def test_fp8_linear_matches_quantize_then_gemm(m, n, k):
    """The fused call gives the two-call result bit for bit, with the
    oracle's token codes and scales."""
    x = synthetic.activations(m, k, m + 5)
    qw, sw = oracle.quant_rows_fp8(util.bits(synthetic.weight(n, k, n + 5)))
    qw_d, sw_d = torch.from_numpy(qw).cuda(), torch.from_numpy(sw).cuda()
    bias = synthetic.bias(n, 7).cuda() if m % 2 == 0 else None
    qx = torch.empty((m, k), dtype=torch.uint8, device="cuda")
    sx = torch.empty((m,), dtype=torch.float32, device="cuda")
    y1 = capi.w8a8_fp8_linear(x.cuda(), qw_d, sw_d, bias=bias, qx=qx, sx=sx)
    y2 = capi.w8a8_fp8_linear(x.cuda(), qw_d, sw_d, bias=bias)
    q2, s2 = capi.quantize_act_per_token_fp8(x.cuda())
    y3 = capi.w8a8_fp8_gemm(q2, s2, qw_d, sw_d, bias=bias)
    torch.cuda.synchronize()
    qx_ref, sx_ref = oracle.quant_rows_fp8(util.bits(x))
    assert np.array_equal(qx.cpu().numpy(), qx_ref) and np.array_equal(sx.cpu().numpy(), sx_ref)
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))
    assert torch.equal(y2.view(torch.int16), y3.view(torch.int16))


def test_fp8_empty_and_zero_rows():
    capi.w8a8_fp8_gemm(torch.empty((0, 64), dtype=torch.uint8, device="cuda"),
                       torch.empty((0,), device="cuda"), torch.zeros((32, 64), dtype=torch.uint8, device="cuda"),
                       torch.ones(32, device="cuda"), y=torch.empty((0, 32), dtype=torch.bfloat16, device="cuda"))
    x = torch.zeros((3, 128), dtype=torch.bfloat16)
    q, s = _gpu_quant(x, False)
    assert (q == 0).all() and (s == 1.0).all()
