"""The relative-Frobenius bar of the GPU tests: where the correctly rounded
bf16 value of the exact result already misses 2e-3, the bar is that rounding
floor (with 5 % room), computed from the oracle alone."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from int8_quantized_linear_gb300 import synthetic
from tests import util


def test_bar_is_the_stated_one_on_typical_outputs():
    g = np.random.default_rng(0)
    ref = g.standard_normal((64, 300))
    assert util.frob_bar(ref, 2e-3) == 2e-3


def test_bar_follows_the_rounding_floor_of_concentrated_outputs():
    # a W4A16 output whose energy sits in a few large elements (outlier
    # activation channels): even the exact result rounded once to bf16
    # misses 2e-3
    m, n, k = 7, 269, 2048
    q, s = oracle.quant_w4_g128(util.bits(synthetic.weight(n, k, 131)))
    ref = oracle.w4a16(util.bits(synthetic.activations(m, k, 141)), q, s)
    rounded = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    floor = util.rel_frobenius(rounded, ref)
    assert floor > 2e-3
    assert util.frob_bar(ref, 2e-3) == 1.05 * floor
    # a result off by one more bf16 ulp on its largest element fails the bar
    worse = rounded.copy()
    i = np.unravel_index(np.argmax(np.abs(ref)), ref.shape)
    worse[i] = worse[i] * (1 + 2.0 ** -7)
    assert util.rel_frobenius(worse, ref) > util.frob_bar(ref, 2e-3)
