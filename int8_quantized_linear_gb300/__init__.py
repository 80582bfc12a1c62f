"""int8 quantized linear layers for GB300 (sm_103a).

The compute lives in ``libi8ql.so`` (hand-written CUDA kernels behind a C
ABI, declared in ``include/i8ql.h``); this package only marshals torch
tensors into it.  Build the library with ``int8_quantized_linear_gb300.build``.
"""

from .capi import (  # noqa: F401
    I8qlError,
    grouped_w8a16_gemm,
    i8ql_get_device_error,
    i8ql_version,
    quantize_act_per_token_int8,
    quantize_weight_per_channel_int8,
    w8a16_gemm,
    w8a8_gemm,
)
