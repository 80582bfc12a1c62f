"""Host-side consistency of bench.py's accounting (no GPU): the kernel
classes, the source lists the DRAM-traffic table is keyed by, the table
itself, and the algorithmic byte counts against their definitions."""

from __future__ import annotations

import json
import os

import numpy as np

import bench


def test_traffic_table_keys_are_known_classes():
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.json")
    table = json.load(open(path))
    for part, entries in table.items():
        if part.startswith("_"):
            continue
        assert part in bench.PART_CLASSES, part
        for kernel, entry in entries.items():
            assert kernel in bench.PART_CLASSES[part], (part, kernel)
            assert kernel in bench.KERNEL_SOURCES[part], (part, kernel)
            assert entry["dram_bytes_per_launch"] > 0
            assert len(entry["source_sha256_16"]) == 16


def test_kernel_source_lists_name_existing_files():
    for part, kernels in bench.KERNEL_SOURCES.items():
        assert part in bench.PART_CLASSES, part
        for kernel, files in kernels.items():
            assert kernel in bench.PART_CLASSES[part], (part, kernel)
            for f in files:
                assert os.path.exists(os.path.join(bench.ROOT, "int8_quantized_linear_gb300", "csrc", f)), f
            assert len(bench.kernel_source_hash(kernel, part)) == 16


def test_tensor_classes_are_classes():
    for part, kernel in bench.TENSOR_CLASSES:
        assert kernel in bench.PART_CLASSES[part]


def test_byte_counts():
    """The algorithmic bytes of each call, recounted from the tensors it
    reads and writes once."""
    m, n, k = 3, 40, 256
    assert bench.bytes_quant(n, k) == 2 * n * k + n * k + 4 * n                 # bf16 in, int8 + fp32 out
    assert bench.bytes_w8a8(m, n, k, True) == m * k + n * k + 4 * m + 4 * n + 2 * m * n + 2 * n
    assert bench.bytes_w8a16(m, n, k) == 2 * m * k + n * k + 4 * n + 2 * m * n
    assert bench.bytes_w4a16(m, n, k) == 2 * m * k + n * k // 2 + 2 * n * (k // 128) + 2 * m * n
    assert bench.bytes_quant_w4(n, k) == 2 * n * k + n * k // 2 + 2 * n * (k // 128)
    assert bench.bytes_linear_fused(m, n, k, False) == 2 * m * k + n * k + 4 * n + 2 * m * n
    counts = np.array([0, 2, 0, 5])
    # experts without rows read nothing
    assert bench.bytes_grouped(counts, n, k) == 2 * (n * k + 4 * n) + 2 * 7 * (k + n)


def _res(per, peaks=None):
    return {"per": per, "peaks": (peaks or {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0,
                                             "bf16_tflops_sustained": 1800.0}, "measured")}


def test_roofline_hbm_class():
    """An HBM-bound class: achieved = algorithmic bytes per launch / mean
    launch time, against the copy peak; the dominant class is the one with
    the most time."""
    per = {"w8a16": {"ms": 2.0, "launches": 4, "bytes": 4 * 24e6, "flops": 0.0},
           "grouped": {"ms": 6.0, "launches": 2, "bytes": 2 * 150e6, "flops": 0.0}}
    r = bench.roofline("decode", _res(per))
    assert r["kernel"] == "grouped" and r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - 150e6 / 3e-3 / 1e9) < 1e-9          # 50 GB/s
    assert abs(r["frac"] - r["achieved"] / 6000.0) < 1e-12
    assert r["algorithmic_bytes_per_launch"] == 150e6
    r16 = bench.roofline("decode", _res(per), "w8a16")
    assert abs(r16["achieved"] - 24e6 / 0.5e-3 / 1e9) < 1e-9


def test_roofline_tensor_classes_take_their_pipe_peak():
    per = {"fp8": {"ms": 1.0, "launches": 10, "bytes": 1e9, "flops": 2e12}}
    r = bench.roofline("fp8", _res(per))
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 2000.0) < 1e-9                       # 2e12 flop in 1 ms
    assert r["peak"] == 2 * 2000.0 and abs(r["frac"] - 0.5) < 1e-12  # the 8-bit pipe: twice bf16
    per = {"w8a8": {"ms": 1.0, "launches": 10, "bytes": 1e9, "flops": 1e12}}
    r = bench.roofline("prefill", _res(per))
    assert r["peak"] == 2000.0 and abs(r["frac"] - 0.5) < 1e-12
