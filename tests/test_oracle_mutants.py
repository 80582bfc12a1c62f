"""Mutation check of the oracle's pins (the check "Phase 5a: int8 weight-only
quantization" lists as deferred in its Summary).

Each mutant is the oracle's C source with one plausible mistake planted by
text substitution, compiled on the CPU into a temporary library.  The pin
suite is then run against it, and at least one pin must fail.  Nothing here
touches a GPU.
"""

from __future__ import annotations

import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from oracle import build as obuild
from tests import test_oracle_pins as pins
from tests import test_oracle_pins_next as pins_next
from tests.golden import load as golden

MUTANTS = {
    "reciprocal_multiply": ("widen_bf16(row[j]) / scale;", "widen_bf16(row[j]) * (1.0f / scale);"),
    "round_half_away": ("float c = round_half_even(t);", "float c = roundf(t);"),
    "bf16_scale_arithmetic": (
        "float scale = (a == 0.0f) ? 1.0f : a / 127.0f;",
        "float scale = (a == 0.0f) ? 1.0f : widen_bf16(narrow_bf16_rne(a / 127.0f));"),
    "small_channel_floor": (
        "float scale = (a == 0.0f) ? 1.0f : a / 127.0f;",
        "float scale = (a < 1e-20f) ? 1.0f : a / 127.0f;"),
    # (The clamp to [-127, 127] is never active: with s = fl32(a / 127) the
    # quotient stays within 127 * (1 + 2^-23), so removing it is an
    # equivalent mutant and is not listed.)
    "signed_max_not_absmax": ("float av = fabsf(widen_bf16(row[j]));", "float av = widen_bf16(row[j]);"),
    "transposed_weight_operand": (
        "acc[m * n_rows + n] = sum;",
        "acc[n * m_rows + m] = sum;"),
    "dropped_bias": ("if (bias) f = f + widen_bf16(bias[n]);", "(void)bias;"),
    "token_scale_twice": ("f = f * sw;", "f = f * sx;"),
    "w8a16_scale_dropped": ("double w = (double)s[n] * (double)q[n * k + j];\n                sum += w * (double)widen_bf16(x[m * k + j]);\n            }\n            y[m * n_rows + n] = sum;",
                            "double w = (double)q[n * k + j];\n                sum += w * (double)widen_bf16(x[m * k + j]);\n            }\n            y[m * n_rows + n] = sum;"),
    "grouped_wrong_expert": ("const int8_t* qe = q + e * n_rows * k;", "const int8_t* qe = q;"),
    "grouped_no_offset_check": ("if (off[e + 1] < off[e]) return ORACLE_ERR_OFFSETS;", "(void)0;"),
    # FP8 E4M3
    "fp8_exponent_bias_8": ("ldexpf(1.0f + (float)m / 8.0f, e - 7)", "ldexpf(1.0f + (float)m / 8.0f, e - 8)"),
    "fp8_ties_to_upper": ("((lo & 1) == 0 ? lo : hi)", "hi"),
    "fp8_scale_over_127": ("(a == 0.0f) ? 1.0f : a / 448.0f;", "(a == 0.0f) ? 1.0f : a / 127.0f;"),
    # (Dropping the explicit saturation at 448 is an equivalent mutant: the
    # bisection then ends between 0x7d and 0x7e with 0x7e the nearer code.)
    "fp8_zero_sign_dropped": ("uint8_t sign = signbit(v) ? 0x80 : 0x00;", "uint8_t sign = (v < 0) ? 0x80 : 0x00;"),
    "fp8_w8a8_scale_dropped": ("double f = sum * (double)sx[m] * (double)sw[n];", "double f = sum * (double)sx[m];"),
    # W4A16, group 128
    "w4_fp32_scale_not_stored_bf16": ("float sv = widen_bf16(sb);", "float sv = (a == 0.0f) ? 1.0f : a / 7.0f;"),
    "w4_absmax_half_group": ("for (int j = 0; j < 128; ++j) {\n                float av", "for (int j = 0; j < 64; ++j) {\n                float av"),
    "w4_nibbles_swapped": ("(uint8_t)((c[0] & 15) | ((c[1] & 15) << 4))", "(uint8_t)((c[1] & 15) | ((c[0] & 15) << 4))"),
    "w4_divide_by_8": ("narrow_bf16_rne(a / 7.0f)", "narrow_bf16_rne(a / 8.0f)"),
    "w4a16_first_group_scale": ("(double)widen_bf16(scale[n * (k / 128) + j / 128])", "(double)widen_bf16(scale[n * (k / 128)])"),
    # MoE expert MLP
    "route_ties_to_higher_index": ("(best < 0 || l[e] > l[best])", "(best < 0 || l[e] >= l[best])"),
    "route_unnormalised_probability": ("prob[t * topk + s] = exp((double)l[best] - mx) / den;",
                                       "prob[t * topk + s] = exp((double)l[best] - mx);"),
    "silu_gate_dropped": ("h[r * inter + j] = g / (1.0 + exp(-g)) * u;", "h[r * inter + j] = g * u;"),
    "silu_up_as_gate": ("double g = gu[r * 2 * inter + j];", "double g = gu[r * 2 * inter + inter + j];"),
    "combine_unweighted": ("sum += w[t * S + s] * yd[", "sum += yd["),
}


def _pin_calls():
    calls = [(f"golden:{c[0]}", lambda c=c: pins.test_quant_golden_rows(c)) for c in golden.quant_rows()]
    for name, bits in pins._quant_inputs():
        calls.append((f"bound:{name}", lambda n=name, b=bits: pins.test_quant_round_trip_bound(n, b)))
    for fn in (pins.test_quant_scale_is_fp32_absmax_over_127, pins.test_quant_argmax_maps_to_full_scale,
               pins.test_quant_sign_symmetry_and_power_of_two_scaling,
               pins.test_quant_zero_row_guard_and_nonfinite_rejected,
               pins.test_quant_matches_ieee_binary32_library_arithmetic,
               pins.test_quant_reciprocal_would_differ_somewhere, pins.test_storage_reduction_closed_form,
               pins.test_int_acc_matches_integer_matmul, pins.test_int_acc_closed_forms,
               pins.test_w8a8_scale_indices_not_swapped, pins.test_bf16_narrowing_matches_torch,
               pins.test_w8a16_equals_float64_dequantized_matmul, pins.test_w8a16_closed_forms,
               pins.test_grouped_is_blockwise_per_expert):
        calls.append((fn.__name__, fn))
    for wb in (False, True):
        calls.append((f"w8a8_rational:{wb}", lambda wb=wb: pins.test_w8a8_int_path_equals_dequantize_then_matmul(wb)))
    calls += [(f"fp8_golden:{c[0]}", lambda c=c: pins_next.test_fp8_golden_rows(c)) for c in golden.fp8_rows()]
    calls += [(f"w4_golden:{c[0]}", lambda c=c: pins_next.test_w4_golden_groups(c)) for c in golden.w4_groups()]
    for t in (1, 8, 64):
        calls.append((f"route_recipe:{t}", lambda t=t: pins_next.test_moe_route_matches_input_recipe_routing(t)))
    for fn in (pins_next.test_fp8_decode_closed_forms, pins_next.test_fp8_codes_match_torch_float8_e4m3fn,
               pins_next.test_fp8_encode_saturates_and_keeps_zero_sign, pins_next.test_fp8_quant_invariants,
               pins_next.test_fp8_w8a8_exact_against_numpy_and_closed_form,
               pins_next.test_w4_scale_is_bf16_of_fp32_absmax_over_7_per_group,
               pins_next.test_w4_round_trip_bound_and_range, pins_next.test_w4_packing_against_independent_unpack,
               pins_next.test_w4a16_equals_float64_dequantized_matmul, pins_next.test_moe_route_hand_derived_ties,
               pins_next.test_silu_mul_closed_forms, pins_next.test_moe_combine_closed_forms):
        calls.append((fn.__name__, fn))
    for off in ([0, 3, 2, 7, 9],):
        calls.append(("grouped_bad_offsets", lambda off=off: pins.test_grouped_rejects_bad_offsets(off)))
    return calls


def _build_mutant(src: str, old: str, new: str, out: str) -> None:
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = src.replace(old, new, 1)
    cfile = out[:-3] + ".c"
    with open(cfile, "w") as fh:
        fh.write(mutated)
    subprocess.run([os.environ.get("CC", "gcc"), *obuild.FLAGS, *obuild.OPENMP, "-w", cfile, "-o", out, "-lm"],
                   check=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_mutant_fails_a_pin(name):
    with open(obuild.SOURCE) as fh:
        src = fh.read()
    old, new = MUTANTS[name]
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, f"mut_{name}.so")
        _build_mutant(src, old, new, path)
        saved = oracle._LIB
        oracle._LIB = oracle.load(path)
        failed = []
        try:
            for label, call in _pin_calls():
                try:
                    with np.errstate(all="ignore"):
                        call()
                except (AssertionError, oracle.OracleError, pytest.fail.Exception) as exc:  # noqa: PERF203
                    failed.append(label)
                    del exc
        finally:
            oracle._LIB = saved
    assert failed, f"mutant {name} survived every pin"


def test_unmutated_oracle_passes_every_pin():
    for label, call in _pin_calls():
        call()
