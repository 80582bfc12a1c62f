"""The W8A8 entry point that allocates no device memory (w8a8_gemm_noalloc).

It exists for callers that cannot allocate while they run (graph replay with
memory fixed at capture, allocator-free serving loops): it must give what
w8a8_gemm gives, take its large-M workspace from the library's fixed array,
and refuse problems that do not fit that array.  Two calls in a row check
that the shared array carries nothing over from one call to the next.

This file is collected last on purpose, and passes both alone in a fresh
process and after the rest of the suite.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from int8_quantized_linear_gb300 import capi
from tests import util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library(cuda_device):
    from int8_quantized_linear_gb300 import build
    build.build()
    capi.lib()
    yield
    assert capi.i8ql_get_device_error() == capi.I8QL_OK


def _problem(m, n, k, seed):
    g = torch.Generator().manual_seed(seed)
    qx = torch.randint(-127, 128, (m, k), generator=g, dtype=torch.int16).to(torch.int8)
    qw = torch.randint(-127, 128, (n, k), generator=g, dtype=torch.int16).to(torch.int8)
    sx = (torch.rand(m, generator=g) * 0.1 + 0.01).float()
    sw = (torch.rand(n, generator=g) * 0.001 + 1e-4).float()
    bias = (torch.randn(n, generator=g) * 0.02).to(torch.bfloat16)
    return [t.cuda() for t in (qx, sx, qw, sw, bias)]


def _both(qx, sx, qw, sw, bias):
    m, n = qx.shape[0], qw.shape[0]
    acc_ref = torch.empty((m, n), dtype=torch.int32, device="cuda")
    y_ref = capi.w8a8_gemm(qx, sx, qw, sw, bias=bias, acc_debug=acc_ref)
    acc = torch.full((m, n), -7, dtype=torch.int32, device="cuda")
    y = torch.full((m, n), 3.0, dtype=torch.bfloat16, device="cuda")
    capi.w8a8_gemm_noalloc(qx, sx, qw, sw, y, bias=bias, acc_debug=acc)
    torch.cuda.synchronize()
    return (acc.cpu().numpy(), util.bits(y.cpu()), acc_ref.cpu().numpy(), util.bits(y_ref.cpu()))


@pytest.mark.parametrize("shapes", [
    [(300, 513, 1040), (200, 1024, 2064)],   # both take the workspace path (M > 32)
    [(129, 6144, 1024), (8, 2560, 2560)],     # workspace path, then the decode path
])
def test_noalloc_matches_w8a8_gemm_on_consecutive_calls(shapes):
    for i, (m, n, k) in enumerate(shapes):
        acc, y, acc_ref, y_ref = _both(*_problem(m, n, k, 100 + i))
        assert np.array_equal(acc, acc_ref), f"call {i}: accumulators differ"
        # identical int32 sums through the same epilogue: bit-identical outputs
        assert np.array_equal(y, y_ref), f"call {i}: outputs differ"


def test_noalloc_rejects_problems_beyond_its_array():
    k = 4096
    m = capi.I8QL_NOALLOC_MAX_ELEMENTS // k + 1  # m * k just over the limit
    n = 48
    qx = torch.zeros((m, k), dtype=torch.int8, device="cuda")
    qw = torch.zeros((n, k), dtype=torch.int8, device="cuda")
    sx = torch.ones(m, device="cuda")
    sw = torch.ones(n, device="cuda")
    y = torch.zeros((m, n), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(capi.I8qlError) as err:
        capi.w8a8_gemm_noalloc(qx, sx, qw, sw, y)
    assert err.value.status == capi.I8QL_ERR_WORKSPACE_LIMIT
    # the decode range needs no workspace, whatever M * K would be
    qx8, sx8 = qx[:8].contiguous(), sx[:8].contiguous()
    y8 = torch.zeros((8, n), dtype=torch.bfloat16, device="cuda")
    capi.w8a8_gemm_noalloc(qx8, sx8, qw, sw, y8)
    torch.cuda.synchronize()
    assert not torch.isnan(y8.float()).any()
