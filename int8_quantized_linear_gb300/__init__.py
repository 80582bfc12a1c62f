"""int8 quantized linear layers for GB300 (sm_103a).

The compute lives in ``libi8ql.so`` (hand-written CUDA kernels behind a C
ABI, declared in ``include/i8ql.h``); this package only marshals torch
tensors into it.  Build the library with ``int8_quantized_linear_gb300.build``.
"""

from .capi import (  # noqa: F401
    I8qlError,
    grouped_w8a16_gemm,
    grouped_w8a16_silu_mul,
    i8ql_early_weight_loads,
    i8ql_fp8_plan,
    i8ql_get_device_error,
    i8ql_set_early_weight_loads,
    i8ql_version,
    i8ql_w8a8_linear_launches,
    i8ql_w8a8_noalloc_plan,
    i8ql_w8a8_plan,
    moe_combine,
    moe_expert_mlp_w8a16,
    moe_route_topk,
    quantize_act_per_token_fp8,
    quantize_act_per_token_int8,
    quantize_weight_per_channel_fp8,
    quantize_weight_per_channel_int8,
    quantize_weight_w4_g128,
    w4a16_gemm,
    w8a8_fp8_gemm,
    w8a8_fp8_linear,
    w8a8_gemm,
    w8a8_gemm_noalloc,
    w8a8_linear,
    w8a16_gemm,
)
