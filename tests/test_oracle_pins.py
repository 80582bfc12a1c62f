"""Pins of the CPU oracle against what the pages and mathematics fix.

None of these tests compares the oracle with itself: each checks it against
a hand-derived fixture, a closed form, an invariant, a printed figure, exact
rational arithmetic, or an independent library routine.  A plausible mistake
anywhere in the oracle (a dropped term, a reciprocal instead of a division,
bf16 scale arithmetic, a transposed operand, a wrong scale index) fails at
least one of them.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from int8_quantized_linear_gb300 import synthetic
from tests.golden import load as golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _bf16(values) -> np.ndarray:
    """float values (already bf16-exact) -> bf16 bits, checked exact."""
    t = torch.tensor(np.asarray(values, np.float64), dtype=torch.float64)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.to(torch.float64), t), "fixture value not exact in bf16"
    return synthetic.bf16_bits(b)


def _random_rows(seed: int, rows: int, k: int) -> np.ndarray:
    w = synthetic.weight(rows, k, seed)
    return synthetic.bf16_bits(w)


# --------------------------------------------------------------------------
# Per-row quantization: "Day 6 -- Quantize It Yourself", mechanism blocks 1
# and 4; "Phase 5a: int8 weight-only quantization", Summary (fp32 arithmetic,
# zero-channel guard without a floor).
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", golden.quant_rows(), ids=lambda c: c[0])
def test_quant_golden_rows(case):
    name, row, scale, codes = case
    q, s = oracle.quant_rows(_bf16([row]))
    assert s[0] == np.float32(scale), (name, float(s[0]).hex())
    assert q[0].tolist() == codes, name


def _quant_inputs():
    yield "weights", _random_rows(11, 96, 320)
    yield "acts", synthetic.bf16_bits(synthetic.activations(64, 512, 12))
    g = torch.Generator().manual_seed(13)
    wide = torch.exp(torch.randn(64, 256, generator=g) * 20) * torch.sign(torch.randn(64, 256, generator=g))
    yield "wide_dynamic_range", synthetic.bf16_bits(wide.clamp(-1e30, 1e30).to(torch.bfloat16))


@pytest.mark.parametrize("name,bits", list(_quant_inputs()), ids=lambda v: v if isinstance(v, str) else "")
def test_quant_round_trip_bound(name, bits):
    """|w - s*q| <= s/2 up to the one fp32 rounding of w/s (the ideal bound
    that the "Phase 5a" Summary says bf16 arithmetic exceeds by up to 1.5x)."""
    q, s = oracle.quant_rows(bits)
    w = oracle.widen_bf16(bits).astype(np.float64)
    err = np.abs(w - s.astype(np.float64)[:, None] * q.astype(np.float64))
    bound = s.astype(np.float64)[:, None] * (0.5 + 128.0 * 2.0 ** -24)
    assert np.all(err <= bound), name


def test_quant_scale_is_fp32_absmax_over_127():
    """s = fl32(absmax / 127): within half an fp32 ulp of the exact ratio.
    bf16 scale arithmetic would miss by up to 2^-9 relative."""
    bits = _random_rows(21, 128, 256)
    q, s = oracle.quant_rows(bits)
    w = oracle.widen_bf16(bits).astype(np.float64)
    a = np.abs(w).max(axis=1)
    exact = a / 127.0
    rel = np.abs(s.astype(np.float64) - exact) / exact
    assert np.all(rel <= 2.0 ** -24)
    # the scale really carries fp32 precision, not bf16's 8 bits
    s_bits = s.view(np.uint32)
    assert np.any((s_bits & 0xFFFF) != 0)


def test_quant_argmax_maps_to_full_scale():
    bits = _random_rows(22, 64, 192)
    q, _ = oracle.quant_rows(bits)
    w = oracle.widen_bf16(bits)
    j = np.abs(w).argmax(axis=1)
    r = np.arange(w.shape[0])
    assert np.all(q[r, j] == np.where(w[r, j] > 0, 127, -127))
    assert q.min() >= -127 and q.max() <= 127


def test_quant_sign_symmetry_and_power_of_two_scaling():
    bits = _random_rows(23, 32, 256)
    q, s = oracle.quant_rows(bits)
    qn, sn = oracle.quant_rows(bits ^ np.uint16(0x8000))
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)
    w = torch.from_numpy(oracle.widen_bf16(bits).copy())
    for j in (-20, 3, 40):
        scaled = synthetic.bf16_bits((w * 2.0 ** j).to(torch.bfloat16))
        q2, s2 = oracle.quant_rows(scaled)
        assert np.array_equal(q2, q)
        assert np.array_equal(s2, (s.astype(np.float64) * 2.0 ** j).astype(np.float32))


def test_quant_zero_row_guard_and_nonfinite_rejected():
    bits = np.zeros((3, 32), np.uint16)
    bits[1] = _bf16([[0.25] * 32])[0]
    q, s = oracle.quant_rows(bits)
    assert s[0] == 1.0 and s[2] == 1.0 and not np.any(np.isnan(s))
    assert not q[0].any() and not q[2].any()
    assert np.all(q[1] == 127)
    bad = bits.copy()
    bad[1, 5] = 0x7FC0  # NaN
    with pytest.raises(oracle.OracleError):
        oracle.quant_rows(bad)


def test_quant_matches_ieee_binary32_library_arithmetic():
    """Cross-check with numpy's IEEE binary32 division and rint (ties to
    even) on many rows, including near-ties found by search."""
    bits = _random_rows(24, 256, 512)
    q, s = oracle.quant_rows(bits)
    w = oracle.widen_bf16(bits)
    a = np.abs(w).max(axis=1)
    s_np = np.where(a == 0, np.float32(1), a / np.float32(127)).astype(np.float32)
    q_np = np.clip(np.rint(w / s_np[:, None]), -127, 127).astype(np.int8)
    assert np.array_equal(s, s_np)
    assert np.array_equal(q, q_np)


def test_quant_reciprocal_would_differ_somewhere():
    """Rows where w * (1/s) and w / s round differently: the oracle follows
    the division (the page writes w / s)."""
    rows = []
    for a in (72.0, 74.0, 74.5, 87.5, 89.5):
        rows.append([a, a / 2, -a / 2])
    q, s = oracle.quant_rows(_bf16(rows))
    w = oracle.widen_bf16(_bf16(rows))
    div = np.rint(w / s[:, None])
    rec = np.rint(w * (np.float32(1) / s)[:, None])
    assert np.array_equal(q, div.astype(np.int8))
    assert not np.array_equal(div, rec)


def test_storage_reduction_closed_form():
    """int8 codes plus one fp32 scale per output channel over a DeepSeek-MoE
    expert (gate [1408,2048], up [1408,2048], down [2048,1408]) saves 49.89 %
    of the bf16 bytes ("Phase 5a", Summary: 49.89 % expert-weight memory
    reduction).  bf16 scales (49.94 %) or per-input-channel scales (49.87 %)
    would not."""
    shapes = [(1408, 2048), (1408, 2048), (2048, 1408)]
    before = after = 0
    for i, (n, k) in enumerate(shapes):
        w = synthetic.weight(n, k, 100 + i, outlier_frac=0.0)
        bits = synthetic.bf16_bits(w)
        q, s = oracle.quant_rows(bits)
        assert q.shape == (n, k) and s.shape == (n,)
        before += bits.nbytes
        after += q.nbytes + s.nbytes
    reduction = 100.0 * (1.0 - after / before)
    assert f"{reduction:.2f}" == "49.89"


# --------------------------------------------------------------------------
# W8A8: "feat(quantization): support compressed-tensors W8A8 and mixed
# modules", Design and Supported Execution Scheme; "Day 6", block 5.
# --------------------------------------------------------------------------

def _codes(seed, rows, k):
    g = np.random.default_rng(seed)
    return g.integers(-127, 128, size=(rows, k), dtype=np.int64).astype(np.int8)


def test_int_acc_matches_integer_matmul():
    qx, qw = _codes(1, 7, 48), _codes(2, 5, 48)
    acc = oracle.int_acc(qx, qw)
    ref = qx.astype(np.int64) @ qw.astype(np.int64).T
    assert acc.shape == (7, 5) and np.array_equal(acc, ref)


def test_int_acc_closed_forms():
    k = 1024
    qx = np.full((2, k), 127, np.int8)
    qw = np.full((3, k), -127, np.int8)
    assert np.all(oracle.int_acc(qx, qw) == -16129 * k)
    # a one-hot token picks a column of the weight codes
    qw = _codes(3, 9, 64)
    for j in (0, 17, 63):
        e = np.zeros((1, 64), np.int8)
        e[0, j] = 1
        assert np.array_equal(oracle.int_acc(e, qw)[0], qw[:, j].astype(np.int64))


def test_int32_range_limit():
    """K = 133,144 is the largest depth whose worst-case sum fits int32."""
    k = 133144
    qx = np.full((1, k), 127, np.int8)
    acc = oracle.int_acc(qx, qx)
    assert acc[0, 0] == 127 * 127 * k <= 2 ** 31 - 1
    f, _ = oracle.w8a8_epilogue(acc, np.ones(1, np.float32), np.ones(1, np.float32))
    assert np.isfinite(f).all()
    with pytest.raises(oracle.OracleError):
        oracle.w8a8_epilogue(acc + 127 * 127, np.ones(1, np.float32), np.ones(1, np.float32))


@pytest.mark.parametrize("with_bias", [False, True])
def test_w8a8_int_path_equals_dequantize_then_matmul(with_bias):
    """Exact rationals: sx*sw*sum(qx*qw) == sum((sx*qx)*(sw*qw)); the
    oracle's fp32 epilogue is that value up to its two or three fp32
    roundings, and its bf16 output is that fp32 value rounded once."""
    m, n, k = 6, 5, 16
    g = np.random.default_rng(5)
    qx, qw = _codes(6, m, k), _codes(7, n, k)
    sx = (g.random(m) * 0.1 + 0.01).astype(np.float32)
    sw = (g.random(n) * 0.001 + 1e-4).astype(np.float32)
    bias = synthetic.bf16_bits(synthetic.bias(n, 8)) if with_bias else None
    acc, f, y = oracle.w8a8(qx, sx, qw, sw, bias)
    bias_f = oracle.widen_bf16(bias) if with_bias else np.zeros(n, np.float32)
    for i in range(m):
        for j in range(n):
            dq = sum((Fraction(float(sx[i])) * int(qx[i, t])) * (Fraction(float(sw[j])) * int(qw[j, t]))
                     for t in range(k))
            ip = Fraction(float(sx[i])) * Fraction(float(sw[j])) * sum(int(qx[i, t]) * int(qw[j, t]) for t in range(k))
            assert dq == ip
            exact = ip + Fraction(float(bias_f[j]))
            rel = 3 * 2.0 ** -24 if with_bias else 2 * 2.0 ** -24
            tol = abs(float(ip)) * rel + (2.0 ** -149)
            assert abs(Fraction(float(f[i, j])) - exact) <= Fraction(tol)
    ref_bits = synthetic.bf16_bits(torch.from_numpy(f).to(torch.bfloat16))
    assert np.array_equal(y, ref_bits)


def test_w8a8_scale_indices_not_swapped():
    """sx is per token (row m), sw per output channel (column n)."""
    qx = np.ones((2, 16), np.int8)
    qw = np.ones((3, 16), np.int8)
    sx = np.array([1.0, 2.0], np.float32)
    sw = np.array([1.0, 10.0, 100.0], np.float32)
    _, f, _ = oracle.w8a8(qx, sx, qw, sw)
    assert np.array_equal(f, np.array([[16, 160, 1600], [32, 320, 3200]], np.float32))


def test_bf16_narrowing_matches_torch():
    g = torch.Generator().manual_seed(9)
    vals = torch.randn(4096, generator=g) * torch.exp(torch.randn(4096, generator=g) * 10)
    ties = torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 2 ** -130 * 3, 65280.5, 0.0, -0.0],
                        dtype=torch.float32)
    v = torch.cat([vals, ties]).numpy()
    ref = synthetic.bf16_bits(torch.from_numpy(v).to(torch.bfloat16))
    assert np.array_equal(oracle.narrow_bf16(v), ref)


def test_w8a8_points_agree_with_full():
    qx, qw = _codes(10, 9, 32), _codes(11, 7, 32)
    sx = np.linspace(0.01, 0.5, 9).astype(np.float32)
    sw = np.linspace(1e-3, 2e-3, 7).astype(np.float32)
    bias = synthetic.bf16_bits(synthetic.bias(7, 3))
    acc, f, y = oracle.w8a8(qx, sx, qw, sw, bias)
    pm = np.array([0, 8, 3, 5]); pn = np.array([6, 0, 2, 2])
    pa, pf, py = oracle.w8a8_points(qx, sx, qw, sw, bias, pm, pn)
    assert np.array_equal(pa, acc[pm, pn]) and np.array_equal(pf, f[pm, pn]) and np.array_equal(py, y[pm, pn])


# --------------------------------------------------------------------------
# W8A16 and its grouped form: "Day 6", block 5 (dequantize inside the kernel,
# multiply on bf16 math); "Phase 5a", Summary (grouped expert GEMM).
# --------------------------------------------------------------------------

def test_w8a16_equals_float64_dequantized_matmul():
    x = synthetic.bf16_bits(synthetic.activations(5, 96, 31))
    q, s = oracle.quant_rows(_random_rows(32, 40, 96))
    y = oracle.w8a16(x, q, s)
    w = s.astype(np.float64)[:, None] * q.astype(np.float64)
    ref = oracle.widen_bf16(x).astype(np.float64) @ w.T
    assert y.shape == (5, 40)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-300)


def test_w8a16_closed_forms():
    q, s = oracle.quant_rows(_random_rows(33, 12, 64))
    for j in (0, 31, 63):
        e = np.zeros((1, 64), np.float32)
        e[0, j] = 1.0
        y = oracle.w8a16(oracle.narrow_bf16(e), q, s)
        assert np.array_equal(y[0], s.astype(np.float64) * q[:, j].astype(np.float64))
    ones = oracle.narrow_bf16(np.ones((1, 64), np.float32))
    y = oracle.w8a16(ones, q, s)
    assert np.array_equal(y[0], s.astype(np.float64) * q.astype(np.float64).sum(axis=1))


def test_w8a16_points_agree_with_full():
    x = synthetic.bf16_bits(synthetic.activations(4, 64, 34))
    q, s = oracle.quant_rows(_random_rows(35, 10, 64))
    y = oracle.w8a16(x, q, s)
    pm = np.array([0, 3, 2]); pn = np.array([9, 0, 4])
    assert np.array_equal(oracle.w8a16_points(x, q, s, pm, pn), y[pm, pn])


def test_grouped_is_blockwise_per_expert():
    e_count, n, k = 4, 24, 64
    q = np.empty((e_count, n, k), np.int8)
    s = np.empty((e_count, n), np.float32)
    for e in range(e_count):
        q[e], s[e] = oracle.quant_rows(_random_rows(40 + e, n, k))
        s[e] *= (e + 1)  # make experts easy to tell apart
    off = np.array([0, 3, 3, 7, 9], np.int32)  # expert 1 is empty
    x = synthetic.bf16_bits(synthetic.activations(9, k, 44))
    y = oracle.grouped_w8a16(x, off, q, s)
    for e in range(e_count):
        lo, hi = off[e], off[e + 1]
        if hi > lo:
            assert np.array_equal(y[lo:hi], oracle.w8a16(x[lo:hi], q[e], s[e]))
    # the wrong expert gives a different answer
    assert not np.allclose(y[0:3], oracle.w8a16(x[0:3], q[2], s[2]))


@pytest.mark.parametrize("off", [[1, 3, 3, 7, 9], [0, 3, 2, 7, 9], [0, 3, 3, 7, 8]])
def test_grouped_rejects_bad_offsets(off):
    q = np.zeros((4, 8, 16), np.int8)
    s = np.ones((4, 8), np.float32)
    x = np.zeros((9, 16), np.uint16)
    with pytest.raises(oracle.OracleError):
        oracle.grouped_w8a16(x, np.array(off, np.int32), q, s)


# --------------------------------------------------------------------------
# The synthetic routing (input generation, not the method).
# --------------------------------------------------------------------------

@pytest.mark.parametrize("tokens", [1, 8, 64])
def test_routing_synthesis_invariants(tokens):
    r = synthetic.moe_routing(tokens, seed=3)
    r2 = synthetic.moe_routing(tokens, seed=3)
    assert np.array_equal(r.offsets, r2.offsets) and np.array_equal(r.rows, r2.rows)
    assert r.experts == 66 and r.offsets[0] == 0 and r.total_rows == 8 * tokens
    assert np.all(np.diff(r.offsets) >= 0)
    for t in range(tokens):
        assert len(set(r.topk[t].tolist())) == 6 and r.topk[t].max() < 64
    counts = np.diff(r.offsets)
    assert counts[64] == tokens and counts[65] == tokens
    # every routed (token, expert) pair appears once, in its expert's block
    for e in range(64):
        toks = r.rows[r.offsets[e]:r.offsets[e + 1]]
        assert sorted(toks.tolist()) == [t for t in range(tokens) if e in r.topk[t]]
    # the chosen experts are the six most probable
    g = torch.Generator().manual_seed(3)
    logits = torch.randn((tokens, 64), generator=g).double().numpy()
    for t in range(tokens):
        chosen = logits[t, r.topk[t]]
        others = np.delete(logits[t], r.topk[t])
        assert chosen.min() >= others.max()
