"""Pins of the oracle's FP8 E4M3, W4A16-g128 and MoE expert-MLP functions.

As for the int8 functions, nothing here compares the oracle with itself:
hand-derived fixtures (``tests/golden/fp8_rows.txt``,
``tests/golden/w4_groups.txt``), closed forms, invariants and independent
library routines (torch's float8_e4m3fn and bf16 conversions, numpy matmul
and softmax, the numpy routing of the input recipe) fix every function, so
that a plausible mistake (a wrong exponent bias, ties away from zero, an
fp32 instead of a bf16 group scale, swapped nibbles, a wrong group size, a
top-k tie broken the other way, a dropped gate or weight) fails one of them.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from int8_quantized_linear_gb300 import synthetic
from tests.golden import load as golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _bf16(values) -> np.ndarray:
    t = torch.tensor(np.asarray(values, np.float64), dtype=torch.float64)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.to(torch.float64), t), "fixture value not exact in bf16"
    return synthetic.bf16_bits(b)


# --------------------------------------------------------------------------
# FP8 E4M3: "Day 6 -- Quantize It Yourself", The mechanism, blocks 1, 2, 5.
# --------------------------------------------------------------------------

def test_fp8_decode_closed_forms():
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x39: 1.125,
             0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0, 0x77: 240.0}
    got = oracle.fp8_decode(np.array(list(cases), np.uint8))
    assert got.tolist() == list(cases.values())
    assert np.isnan(oracle.fp8_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    assert np.signbit(oracle.fp8_decode(np.array([0x80], np.uint8)))[0]


def test_fp8_codes_match_torch_float8_e4m3fn():
    """Library cross-check: decoding agrees with torch for every code, and
    encoding agrees with torch's round-to-nearest-even cast on random values
    of every magnitude inside the range and on every exact midpoint."""
    codes = np.arange(256, dtype=np.uint8)
    finite = codes[(codes & 0x7F) != 0x7F]
    mine = oracle.fp8_decode(finite)
    theirs = torch.from_numpy(finite.copy()).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(mine, theirs)
    g = np.random.default_rng(5)
    v = (g.standard_normal(200000) * np.exp(g.uniform(-12, 6, 200000))).astype(np.float32)
    v = np.clip(v, -448, 448)
    pos = np.sort(np.unique(np.abs(mine)))
    mids = ((pos[1:].astype(np.float64) + pos[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, pos, -pos])
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.fp8_encode(v), want)


def test_fp8_encode_saturates_and_keeps_zero_sign():
    got = oracle.fp8_encode(np.array([448.0, 449.0, 464.0, 1e30, -500.0, -0.0, 0.0, -1e-30], np.float32))
    assert got.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x00, 0x80]


@pytest.mark.parametrize("case", golden.fp8_rows(), ids=lambda c: c[0])
def test_fp8_golden_rows(case):
    name, row, scale, codes = case
    q, s = oracle.quant_rows_fp8(_bf16([row]))
    assert s[0] == np.float32(scale), (name, float(s[0]).hex())
    assert q[0].tolist() == codes, name


def test_fp8_quant_invariants():
    """s = fl32(absmax / 448); the absmax element maps to +-448; every code
    is the nearest grid point of the binary32 quotient (within half the grid
    spacing at its magnitude); the zero row is guarded."""
    w = synthetic.weight(64, 512, 21).float()
    w[3] = 0.0
    bits = synthetic.bf16_bits(w.to(torch.bfloat16))
    q, s = oracle.quant_rows_fp8(bits)
    wf = oracle.widen_bf16(bits)
    a = np.abs(wf).max(axis=1)
    want_s = np.where(a == 0, np.float32(1), (a / np.float32(448)).astype(np.float32))
    assert np.array_equal(s, want_s)
    assert q[3].tolist() == [0] * 512
    nz = np.arange(64) != 3
    amax = np.argmax(np.abs(wf), axis=1)
    assert set((q[nz, amax[nz]] & 0x7F).tolist()) == {0x7E}
    t = (wf / s[:, None]).astype(np.float32).astype(np.float64)
    d = oracle.fp8_decode(q).astype(np.float64)
    mag = np.abs(t)
    e = np.floor(np.log2(np.maximum(mag, 2.0 ** -6)))
    half_spacing = 2.0 ** (e - 3) / 2
    assert np.all(np.abs(d - t) <= half_spacing * (1 + 1e-12))


def test_fp8_w8a8_exact_against_numpy_and_closed_form():
    g = np.random.default_rng(8)
    qx = g.integers(0, 256, (5, 96)).astype(np.uint8)
    qw = g.integers(0, 256, (7, 96)).astype(np.uint8)
    qx[(qx & 0x7F) == 0x7F] = 0x38
    qw[(qw & 0x7F) == 0x7F] = 0xB8
    sx = g.uniform(0.01, 1, 5).astype(np.float32)
    sw = g.uniform(1e-4, 1e-2, 7).astype(np.float32)
    bias = _bf16(np.round(g.standard_normal(7) * 8) / 8)
    acc, y = oracle.w8a8_fp8(qx, sx, qw, sw, bias)
    dx = torch.from_numpy(qx.copy()).view(torch.float8_e4m3fn).double().numpy()
    dw = torch.from_numpy(qw.copy()).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(acc, dx @ dw.T)
    want = (dx @ dw.T) * sx[:, None].astype(np.float64) * sw[None, :].astype(np.float64) + \
        oracle.widen_bf16(bias).astype(np.float64)[None, :]
    assert np.allclose(y, want, rtol=1e-15, atol=0)
    # all ones (0x38) and all 448 (0x7e): sums K and K * 448^2 exactly
    ones = np.full((2, 64), 0x38, np.uint8)
    big = np.full((3, 64), 0x7E, np.uint8)
    acc1, _ = oracle.w8a8_fp8(ones, np.ones(2, np.float32), big, np.ones(3, np.float32))
    assert (acc1 == 64 * 448.0).all()
    acc2, _ = oracle.w8a8_fp8(big, np.ones(3, np.float32), big, np.ones(3, np.float32))
    assert (acc2 == 64 * 448.0 * 448.0).all()


# --------------------------------------------------------------------------
# W4A16 group 128: "Day 6", The mechanism, blocks 1 and 5.
# --------------------------------------------------------------------------

@pytest.mark.parametrize("case", golden.w4_groups(), ids=lambda c: c[0])
def test_w4_golden_groups(case):
    name, row, scales, groups, nbytes = case
    packed, sc = oracle.quant_w4_g128(_bf16([row]))
    assert oracle.widen_bf16(sc[0]).tolist() == scales, name
    codes = oracle.w4_unpack(packed, len(row))[0]
    for gi, want in enumerate(groups):
        assert codes[gi * 128: gi * 128 + len(want)].tolist() == want, (name, gi)
    assert packed[0, :len(nbytes)].tolist() == nbytes, name


def test_w4_scale_is_bf16_of_fp32_absmax_over_7_per_group():
    """Library cross-check of the scale (torch's bf16 cast of the fp32
    quotient), per group of 128 along K: an outlier moves only its group."""
    w = synthetic.weight(16, 512, 31).float()
    w[5, 300] = 3.0
    bits = synthetic.bf16_bits(w.to(torch.bfloat16))
    packed, sc = oracle.quant_w4_g128(bits)
    wf = torch.from_numpy(oracle.widen_bf16(bits)).view(16, 4, 128)
    a = wf.abs().amax(dim=2)
    want = (a / torch.tensor(7.0, dtype=torch.float32)).to(torch.bfloat16)
    want = torch.where(a == 0, torch.ones_like(want), want)
    assert np.array_equal(sc, synthetic.bf16_bits(want))
    assert oracle.widen_bf16(sc[5, 2]) == np.float32(torch.tensor(3.0 / 7, dtype=torch.float32).to(
        torch.bfloat16).float().item())
    assert (oracle.widen_bf16(sc[5, [0, 1, 3]]) < 0.05).all()


def test_w4_round_trip_bound_and_range():
    """|w - s q| <= s / 2 with the stored scale; codes in [-7, 7], the group
    absmax mapping to +-7."""
    bits = synthetic.bf16_bits(synthetic.weight(32, 1024, 33))
    packed, sc = oracle.quant_w4_g128(bits)
    q = oracle.w4_unpack(packed, 1024).astype(np.float64)
    s = np.repeat(oracle.widen_bf16(sc).astype(np.float64), 128, axis=1)
    w = oracle.widen_bf16(bits).astype(np.float64)
    assert np.all(np.abs(w - s * q) <= s / 2 * (1 + 2.0 ** -20))
    assert q.min() >= -7 and q.max() <= 7
    wg = np.abs(w).reshape(32, 8, 128).argmax(axis=2)
    qg = np.abs(q).reshape(32, 8, 128)
    assert (np.take_along_axis(qg, wg[..., None], axis=2) == 7).all()


def test_w4_packing_against_independent_unpack():
    bits = synthetic.bf16_bits(synthetic.weight(8, 256, 34))
    packed, _ = oracle.quant_w4_g128(bits)
    lo = (packed & 15).astype(np.int16)
    hi = (packed >> 4).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    codes = np.stack([lo, hi], axis=2).reshape(8, 256)
    assert np.array_equal(codes, oracle.w4_unpack(packed, 256))


def test_w4a16_equals_float64_dequantized_matmul():
    bits = synthetic.bf16_bits(synthetic.weight(24, 384, 35))
    packed, sc = oracle.quant_w4_g128(bits)
    x = synthetic.bf16_bits(synthetic.activations(5, 384, 36))
    # independent dequantization: numpy nibbles and torch bf16 widening
    lo = (packed & 15).astype(np.int16)
    hi = (packed >> 4).astype(np.int16)
    codes = np.stack([np.where(lo >= 8, lo - 16, lo), np.where(hi >= 8, hi - 16, hi)], axis=2).reshape(24, 384)
    s = torch.from_numpy(sc.view(np.int16)).view(torch.bfloat16).double().numpy()
    wd = codes * np.repeat(s, 128, axis=1)
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.allclose(oracle.w4a16(x, packed, sc), xd @ wd.T, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# MoE expert MLP around the grouped GEMM: "Phase 5a", Summary, and the
# DeepSeek-MoE-16B configuration (top-6 of 64 routed + 2 shared experts).
# --------------------------------------------------------------------------

def test_moe_route_hand_derived_ties():
    logits = np.array([[0.5, 2.0, 2.0, -1.0, 3.0, 0.0, 2.0, 1.0],
                       [1.0] * 8], np.float32)
    r = oracle.moe_route(logits, topk=3, shared=1)
    assert r.sel.tolist() == [[4, 1, 2], [0, 1, 2]]  # equal logits: lower index first
    assert r.offsets.tolist() == [0, 1, 3, 5, 5, 6, 6, 6, 6, 8]
    assert r.row_token.tolist() == [1, 0, 1, 0, 1, 0, 0, 1]
    assert r.token_row.tolist() == [[5, 1, 3, 6], [0, 2, 4, 7]]
    assert r.prob[1].tolist() == [0.125] * 3
    z = np.exp(logits[0].astype(np.float64) - 3.0)
    assert np.allclose(r.prob[0], z[[4, 1, 2]] / z.sum(), rtol=1e-15)
    assert r.row_weight.tolist() == [0.125, r.prob[0, 1], 0.125, r.prob[0, 2], 0.125, r.prob[0, 0], 1.0, 1.0]


@pytest.mark.parametrize("tokens", [1, 8, 64])
def test_moe_route_matches_input_recipe_routing(tokens):
    """Library cross-check: numpy's stable sort of the softmax probabilities
    (the input recipe's routing) selects and groups the same rows."""
    ref = synthetic.moe_routing(tokens, seed=3)
    logits = synthetic.gate_logits(tokens, 64, 3).numpy()
    r = oracle.moe_route(logits, topk=6, shared=2)
    assert np.array_equal(r.sel, ref.topk)
    assert np.array_equal(r.offsets, ref.offsets)
    assert np.array_equal(r.row_token, ref.rows)
    z = logits.astype(np.float64) - logits.max(axis=1, keepdims=True)
    p = np.exp(z) / np.exp(z).sum(axis=1, keepdims=True)
    assert np.allclose(r.prob, np.take_along_axis(p, ref.topk, axis=1), rtol=1e-14)
    # every (token, slot) row holds that token
    assert np.array_equal(r.row_token[r.token_row], np.repeat(np.arange(tokens)[:, None], 8, axis=1))


def test_silu_mul_closed_forms():
    g = np.array([0.0, 1.0, -1.0, 40.0, -40.0, 2.5])
    u = np.array([3.0, 2.0, 2.0, 0.5, 7.0, -1.0])
    h = oracle.silu_mul(np.concatenate([g, u])[None, :])[0]
    want = g * (1 / (1 + np.exp(-g))) * u
    assert np.allclose(h, want, rtol=1e-15, atol=0)
    assert h[0] == 0.0 and abs(h[3] - 20.0) < 1e-12 and abs(h[4]) < 40 * 7 * np.exp(-40.0) * 1.01
    assert abs(h[1] - 2.0 / (1.0 + np.exp(-1.0))) < 1e-15  # gate first, then up


def test_moe_combine_closed_forms():
    yd = np.arange(12, dtype=np.float64).reshape(4, 3)
    token_row = np.array([[2, 0], [1, 3]], np.int32)
    w = np.array([[0.25, 1.0], [0.5, 2.0]])
    out = oracle.moe_combine(yd, token_row, w)
    assert out.tolist() == [[0.25 * 6 + 0, 0.25 * 7 + 1, 0.25 * 8 + 2],
                            [0.5 * 3 + 2 * 9, 0.5 * 4 + 2 * 10, 0.5 * 5 + 2 * 11]]
