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
