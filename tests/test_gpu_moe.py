"""GPU parity of the MoE expert MLP around the grouped GEMM (routing, the
fused gate/up SiLU-gated product, down, weighted combine) against the CPU
oracle, through the C ABI, on the DeepSeek-MoE-16B shapes (64 routed + 2
shared experts, top-6, hidden 2048, expert intermediate 1408).

Bars:
 * routing: offsets, grouped rows and (token, slot) rows bit-exact (the
   choice is made on the fp32 logits themselves, ties to the lower index);
   slot weights within 2e-6 relative of the fp64 softmax (fp32 exp and sum);
 * each GEMM stage on the previous stage's GPU output: relative Frobenius
   error <= 2e-3 (the weight-only bar) and every element within the fp32
   accumulation bound plus one bf16 rounding (for the SiLU-gated product,
   propagated through silu(g) * u with |silu'| <= 1.1);
 * the whole layer: identical, bit for bit, to the four stages called one by
   one, and within 6e-3 relative Frobenius of the all-fp64 oracle chain
   (three bf16-rounded stage outputs, each <= 2e-3).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from int8_quantized_linear_gb300 import capi, synthetic
from tests import util

pytestmark = pytest.mark.gpu

ROUTED, SHARED, TOPK = 64, 2, 6
H, INTER = 2048, 1408


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    from int8_quantized_linear_gb300 import build
    build.build()
    capi.lib()
    assert capi.i8ql_get_device_error() == capi.I8QL_OK
    yield
    assert capi.i8ql_get_device_error() == capi.I8QL_OK


_EXPERTS = {}


def experts():
    """Oracle-quantized DS-MoE expert weights (gate/up then down), cached."""
    if not _EXPERTS:
        e = ROUTED + SHARED
        for name, (n, k), seed in (("gu", (2 * INTER, H), 1000), ("d", (H, INTER), 1100)):
            q = np.empty((e, n, k), np.int8)
            s = np.empty((e, n), np.float32)
            for i in range(e):
                q[i], s[i] = oracle.quant_rows(util.bits(synthetic.weight(n, k, seed + i)))
            _EXPERTS[name] = (q, s)
    return _EXPERTS


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


# ------------------------------------------------------------------ routing

def check_route(logits: np.ndarray, topk=TOPK, shared=SHARED):
    off, row_token, token_row, w = capi.moe_route_topk(dev(logits), topk, shared)
    torch.cuda.synchronize()
    ref = oracle.moe_route(logits, topk, shared)
    assert np.array_equal(off.cpu().numpy(), ref.offsets)
    assert np.array_equal(row_token.cpu().numpy(), ref.row_token)
    assert np.array_equal(token_row.cpu().numpy(), ref.token_row)
    got_w = w.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got_w - ref.slot_weight) <= 2e-6 * np.abs(ref.slot_weight))
    return ref


@pytest.mark.parametrize("tokens", [1, 8, 64, 512, 4096])
def test_route_matches_oracle(tokens):
    check_route(synthetic.gate_logits(tokens, ROUTED, 3 + tokens).numpy())


def test_route_ties_and_small_shapes():
    logits = np.array([[0.5, 2.0, 2.0, -1.0, 3.0, 0.0, 2.0, 1.0], [1.0] * 8], np.float32)
    ref = check_route(logits, topk=3, shared=1)
    assert ref.token_row.tolist() == [[5, 1, 3, 6], [0, 2, 4, 7]]
    g = np.random.default_rng(9)
    ties = np.round(g.standard_normal((300, 40)) * 2).astype(np.float32)  # many equal logits
    check_route(ties, topk=8, shared=0)
    check_route(g.standard_normal((33, 256)).astype(np.float32), topk=32, shared=64)


def test_route_empty():
    off, _, _, _ = capi.moe_route_topk(torch.empty((0, ROUTED), dtype=torch.float32, device="cuda"), TOPK, SHARED)
    torch.cuda.synchronize()
    assert (off.cpu() == 0).all()


# ------------------------------------------------------------------ stages

def gpu_stages(x_bf16, logits):
    """The four stages called one by one: (route, h, yd, out) on the device."""
    (qgu, sgu), (qd, sd) = experts()["gu"], experts()["d"]
    off, row_token, token_row, w = capi.moe_route_topk(dev(logits), TOPK, SHARED)
    h = capi.grouped_w8a16_silu_mul(x_bf16.cuda(), row_token, off, dev(qgu), dev(sgu))
    yd = capi.grouped_w8a16_gemm(h, off, dev(qd), dev(sd))
    out = capi.moe_combine(yd, token_row, w)
    torch.cuda.synchronize()
    return (off, row_token, token_row, w), h, yd, out


@pytest.mark.parametrize("tokens", [1, 8, 64])
def test_moe_stages_against_oracle(tokens):
    x = synthetic.activations(tokens, H, 700 + tokens)
    logits = synthetic.gate_logits(tokens, ROUTED, 800 + tokens).numpy()
    (qgu, sgu), (qd, sd) = experts()["gu"], experts()["d"]
    route, h, yd, out = gpu_stages(x, logits)
    ref = oracle.moe_route(logits, TOPK, SHARED)
    xg = util.bits(x)[ref.row_token]  # the gathered token rows
    # gate/up with the SiLU-gated product
    gu = oracle.grouped_w8a16(xg, ref.offsets, qgu, sgu)
    h_ref = oracle.silu_mul(gu)
    h_gpu = util.from_bits(util.bits(h.cpu())).double().numpy()
    assert util.rel_frobenius(h_gpu, h_ref) <= util.frob_bar(h_ref, 2e-3)
    mag = oracle.grouped_w8a16(xg & np.uint16(0x7FFF), ref.offsets, np.abs(qgu.astype(np.int16)).astype(np.int8), sgu)
    eg, eu = mag[:, :INTER] * H * 2.0 ** -23, mag[:, INTER:] * H * 2.0 ** -23
    g_ref, u_ref = gu[:, :INTER], gu[:, INTER:]
    silu = g_ref / (1 + np.exp(-g_ref))
    bound = 1.1 * eg * np.abs(u_ref) + eu * np.abs(silu) + eg * eu + np.abs(h_ref) * (2.0 ** -8 + 1e-6) + 1e-30
    assert np.all(np.abs(h_gpu - h_ref) <= bound)
    # down on the GPU's h
    hb = util.bits(h.cpu())
    yd_ref = oracle.grouped_w8a16(hb, ref.offsets, qd, sd)
    yd_gpu = util.from_bits(util.bits(yd.cpu())).double().numpy()
    assert util.rel_frobenius(yd_gpu, yd_ref) <= util.frob_bar(yd_ref, 2e-3)
    # combine of the GPU's expert outputs
    out_ref = oracle.moe_combine(yd_gpu, ref.token_row, ref.slot_weight)
    out_gpu = util.from_bits(util.bits(out.cpu())).double().numpy()
    assert util.rel_frobenius(out_gpu, out_ref) <= util.frob_bar(out_ref, 2e-3)
    mag_c = oracle.moe_combine(np.abs(yd_gpu), ref.token_row, ref.slot_weight)
    bound_c = mag_c * ((TOPK + SHARED) * 2.0 ** -23 + 2e-6) + np.abs(out_ref) * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(out_gpu - out_ref) <= bound_c)


@pytest.mark.parametrize("tokens", [1, 8, 64])
def test_moe_layer_one_call(tokens):
    """moe_expert_mlp_w8a16 equals the staged calls bit for bit, and the
    all-fp64 oracle chain within three stages' bars."""
    x = synthetic.activations(tokens, H, 900 + tokens)
    logits = synthetic.gate_logits(tokens, ROUTED, 950 + tokens).numpy()
    (qgu, sgu), (qd, sd) = experts()["gu"], experts()["d"]
    _, _, _, out_staged = gpu_stages(x, logits)
    out = capi.moe_expert_mlp_w8a16(x.cuda(), dev(logits), TOPK, SHARED, dev(qgu), dev(sgu), dev(qd), dev(sd))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_staged.view(torch.int16))
    ref = oracle.moe_route(logits, TOPK, SHARED)
    xg = util.bits(x)[ref.row_token]
    h64 = oracle.silu_mul(oracle.grouped_w8a16(xg, ref.offsets, qgu, sgu))
    # the fp64 chain: down of the unrounded h, by its definition (sum over k of s q h)
    yd64 = np.empty((h64.shape[0], H))
    for e in range(ROUTED + SHARED):
        a, b = ref.offsets[e], ref.offsets[e + 1]
        if b > a:
            yd64[a:b] = h64[a:b] @ (qd[e].astype(np.float64) * sd[e][:, None].astype(np.float64)).T
    out64 = oracle.moe_combine(yd64, ref.token_row, ref.slot_weight)
    got = util.from_bits(util.bits(out.cpu())).double().numpy()
    assert util.rel_frobenius(got, out64) <= 6e-3
