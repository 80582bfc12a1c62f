#!/usr/bin/env python
"""Benchmark of the int8 quantized linear layer on GB300.

The default run (``--workload all``) measures the whole metric, "int8 GEMM
TOPS (prefill) & weight GB/s (decode)", in three parts, each captured as a
CUDA graph of one step and timed on its own, and prints ONE JSON line:

  decode (top-level value, GB/s): the Qwen3-4B decode linears plus the
  DeepSeek-MoE-16B grouped experts, one pass of every row of the path:
    * per-channel weight quantization of the four bf16 projection weights
      (fused QKV [6144, 2560], o [2560, 2560], fused gate_up [19456, 2560],
      down [2560, 9728]);
    * for M in {1, 4, 8} and each projection: per-token activation
      quantization, the W8A8 GEMM and the W8A16 GEMM;
    * the grouped W8A16 GEMM over 66 experts (64 routed, top-6, + 2 shared)
      for T in {1, 8, 64} decode tokens, gate_up [2816, 2048] then down
      [2048, 1408].
  prefill (block "prefill", TOPS): Qwen3-4B W8A8 prefill, bias on: for M in
    {128, 512, 2048, 4096} and each projection, the W8A8 linear layer from
    bf16 activations (w8a8_linear: per-token quantization fused into the
    call).
  Qwen3-8B sweep (block "qwen3_8b_sweep"): fused QKV [6144, 4096],
    o [4096, 4096], fused gate_up [24576, 4096], down [4096, 12288]; W8A16
    for M in {1, 2, 4, 8, 16, 32, 64} and the W8A8 linear layer for M in
    {1, 2, 4, 8, 16, 32, 64, 128, 512, 2048, 8192}.
  FP8 prefill (block "fp8_prefill", TOPS against the 8-bit pipe): the
    Qwen3-4B prefill shapes through the FP8 E4M3 linear layer.
  W4A16 decode (block "w4a16_decode", GB/s): int4 group-128 quantization of
    the Qwen3-8B weights and the W4A16 GEMM at M in {1, 4, 8}.
  MoE expert MLP (block "moe_mlp", GB/s): the DeepSeek-MoE-16B layer for
    T in {1, 8, 64}: device routing, gate/up with the SiLU-gated product,
    down, weighted combine, one call each.
  One-launch W8A8 (block "w8a8_linear_one_launch", GB/s): the Qwen3-4B
    decode shapes through w8a8_linear_fused, the per-token quantization
    inside the decode GEMM (the decode part runs the faster two launches).

Every GEMM launch of a step reads its own copy of the int8 weights, and each
part touches more than the 129 MB L2 per step, so no launch finds its
weights in L2 (between timed steps nothing is reused either).  The timed
region replays K steps of the part's graph back to back.  Launches of one
kernel class run back to back (programmatic dependent launch overlaps their
prologues), and an external CUDA event pair around each class's batch times
it live: average launch duration = batch time / launches.  The decode,
sweep and one-launch parts run with the library's early weight loads on
(i8ql_set_early_weight_loads: split-K decode GEMMs start their weight
stream before waiting for the previous kernel, whose outputs they do not
read as weights); config.early_weight_loads names those parts.

value (decode) = algorithmic HBM bytes of all launches / step time (GB/s);
prefill TOPS = 2*M*N*K summed over the W8A8 launches / step time.
Algorithmic bytes per launch: quantization 3*R*K + 4*R; W8A8
M*K + N*K + 4*(M+N) + 2*M*N (+2*N bias); the W8A8 linear layer adds the
quantization pass of its activations, except in one launch (decode), where
it reads the bf16 tokens once: 2*M*K + N*K + 4*N + 2*M*N; W8A16
N*K + 4*N + 2*M*K + 2*M*N; grouped sum over experts with rows of
(N*K + 4*N) + 2*rows*(K+N); W4A16 N*K/2 + 2*N*K/128 + 2*M*K + 2*M*N; the
expert MLP its experts' weights and scales plus its row traffic.

cpu_baseline times the CPU oracle (the only reference implementation: the
pages ship no code) on the host cores, with one thread and with every core,
on a bounded sample of the same workload; --impl reference times it with
every core.

Other modes: --single KIND:DIMS times one call eagerly (for ncu captures of
one kernel); --shapes GROUPS prints one JSON line per shape and call of
every path (CUDA-graph replays over weight copies larger than L2), the
per-call tables of the measured results.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "int8 GEMM TOPS (prefill) & weight GB/s (decode) vs GB300 roofline"
DECODE_MS = (1, 4, 8)
PREFILL_MS = (128, 512, 2048, 4096)
MOE_TOKENS = (1, 8, 64)
SWEEP_W8A16_MS = (1, 2, 4, 8, 16, 32, 64)
W4_MS = (1, 4, 8)
SWEEP_W8A8_MS = (1, 2, 4, 8, 16, 32, 64, 128, 512, 2048, 8192)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Kernel classes of each part, in launch order; "tensor" classes are
# contractions on the tensor-core kernel (TOPS against the bf16-pipe peak),
# the others stream weights (GB/s against HBM).
PART_CLASSES = {
    "decode": ("quant_w", "quant_x", "w8a8", "w8a16", "grouped"),
    "prefill": ("w8a8",),
    "sweep8b": ("w8a16", "w8a8_decode", "w8a8_prefill"),
    "fp8": ("fp8",),
    "w4": ("quant_w4", "w4a16"),
    "moe": ("moe_mlp",),
    "fused": ("w8a8_fused",),
}
# tensor-bound classes and the peak each is measured against: the int8
# W8A8 kernel runs on the fp16 pipe (the bf16 rate), FP8 on the 8-bit pipe
# (twice the bf16 rate, the nominal ratio)
TENSOR_CLASSES = {("prefill", "w8a8"): 1.0, ("sweep8b", "w8a8_prefill"): 1.0, ("fp8", "fp8"): 2.0}


# ---------------------------------------------------------------- accounting

def bytes_quant(r, k):
    return 3 * r * k + 4 * r


def bytes_w8a8(m, n, k, bias):
    return m * k + n * k + 4 * (m + n) + 2 * m * n + (2 * n if bias else 0)


def bytes_w8a16(m, n, k):
    return n * k + 4 * n + 2 * m * k + 2 * m * n


def bytes_grouped(counts, n, k):
    active = [int(c) for c in counts if c > 0]
    return len(active) * (n * k + 4 * n) + 2 * sum(active) * (k + n)


def bytes_linear_fused(m, n, k, bias):
    """W8A8 from bf16 tokens in one pass: the tokens are read once as bf16
    and their codes never leave the kernel."""
    return 2 * m * k + n * k + 4 * n + 2 * m * n + (2 * n if bias else 0)


def bytes_w4a16(m, n, k):
    return n * k // 2 + 2 * n * (k // 128) + 2 * m * k + 2 * m * n


def bytes_quant_w4(n, k):
    return 2 * n * k + n * k // 2 + 2 * n * (k // 128)


def bytes_moe(counts, tokens, hidden, inter, routed):
    """The expert MLP: the weights and scales of every expert with rows
    (gate/up and down), the gathered tokens, h written and read, the down
    outputs written and read by the combine, the outputs and the logits."""
    active = [int(c) for c in counts if c > 0]
    rows = sum(active)
    weights = len(active) * (2 * inter * hidden + 8 * inter + hidden * inter + 4 * hidden)
    return weights + 2 * rows * hidden + 4 * rows * inter + 4 * rows * hidden + 2 * tokens * hidden + 4 * tokens * routed


def workload_name(part):
    if part == "decode":
        return ("Qwen3-4B decode linears (QKV 6144x2560, o 2560x2560, gate_up 19456x2560, "
                "down 9728->2560; M in {1,4,8}; weight quant + act quant + W8A8 + W8A16) + "
                "DeepSeek-MoE-16B grouped W8A16 (66 experts, top-6 + 2 shared, T in {1,8,64}; "
                "gate_up 2816x2048, down 2048x1408)")
    if part == "prefill":
        return ("Qwen3-4B prefill W8A8 (QKV 6144x2560, o 2560x2560, gate_up 19456x2560, down 9728->2560; "
                "M in {128,512,2048,4096}; W8A8 linear from bf16 activations (per-token act quant fused), bias on)")
    if part == "fp8":
        return ("Qwen3-4B prefill FP8 E4M3 W8A8 (same four shapes, M in {128,512,2048,4096}, per-token dynamic "
                "FP8 activations and per-channel FP8 weights, bias on; FP8 linear from bf16 activations)")
    if part == "w4":
        return ("Qwen3-8B W4A16 group-128 decode (QKV 6144x4096, o 4096x4096, gate_up 24576x4096, down 12288->4096; "
                "M in {1,4,8}; int4 weight quantization + W4A16 GEMM)")
    if part == "fused":
        return ("Qwen3-4B decode W8A8 linear layer in one launch (per-token quantization inside the decode GEMM; "
                "the four shapes, M in {1,4,8})")
    if part == "moe":
        return ("DeepSeek-MoE-16B expert MLP, int8 weight-only (66 experts, top-6 + 2 shared; device routing, "
                "gate_up 2816x2048 with the SiLU-gated product, down 2048x1408, weighted combine; T in {1,8,64})")
    return ("Qwen3-8B sweep (QKV 6144x4096, o 4096x4096, gate_up 24576x4096, down 12288->4096; "
            "W8A16 for M in {1,2,4,8,16,32,64}; W8A8 linear from bf16 activations for "
            "M in {1,2,4,8,16,32,64,128,512,2048,8192})")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# CUDA sources each kernel class runs (W8A8 in the decode range runs on the
# decode kernel; above it on the tensor-core kernel).
KERNEL_SOURCES = {
    "decode": {"w8a8": ["decode_gemm.cu"], "w8a16": ["decode_gemm.cu"], "grouped": ["decode_gemm.cu"],
               "quant_w": ["quant.cu"], "quant_x": ["quant.cu"]},
    "prefill": {"w8a8": ["w8a8.cu", "w8a8_fused.cu", "tc_common.cuh", "quant.cu"]},
    "sweep8b": {"w8a16": ["decode_gemm.cu"], "w8a8_decode": ["decode_gemm.cu", "quant.cu"],
                "w8a8_prefill": ["w8a8.cu", "w8a8_fused.cu", "tc_common.cuh", "quant.cu"]},
    "w4": {"w4a16": ["w4a16.cu"], "quant_w4": ["w4a16.cu", "quant_math.cuh"]},
    "fp8": {"fp8": ["fp8_gemm.cu", "tc_common.cuh", "quant.cu", "quant_math.cuh"]},
    "moe": {"moe_mlp": ["moe.cu", "decode_gemm.cu"]},
    "fused": {"w8a8_fused": ["decode_gemm.cu", "quant_math.cuh"]},
}


def kernel_source_hash(kernel, part):
    h = hashlib.sha256()
    for src in KERNEL_SOURCES[part][kernel]:
        with open(os.path.join(ROOT, "int8_quantized_linear_gb300", "csrc", src), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, part):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        table = json.load(fh)
    entry = table.get(part, {}).get(kernel)
    if not entry or kernel not in KERNEL_SOURCES.get(part, {}) or \
            entry.get("source_sha256_16") != kernel_source_hash(kernel, part):
        return None
    return entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- GPU workload

class Launch:
    __slots__ = ("kernel", "fn", "bytes", "flops", "label", "gpu_kernels")

    def __init__(self, kernel, fn, nbytes, flops, label, gpu_kernels=1):
        self.kernel, self.fn, self.bytes, self.flops, self.label = kernel, fn, nbytes, flops, label
        self.gpu_kernels = gpu_kernels  # library kernels one call launches


class Workload:
    """Device buffers and the ordered launch list of one step of a part."""

    def __init__(self, part, device, seed=1):
        from int8_quantized_linear_gb300 import capi
        self._capi = capi
        self.part = part
        self.device = device
        self.launches: list[Launch] = []
        self.h2d: list[tuple[torch.Tensor, torch.Tensor]] = []  # (pinned host, device) inputs
        self.d2h: list[tuple[torch.Tensor, torch.Tensor]] = []  # (device, pinned host) results
        getattr(self, "_" + part)(seed)
        # Launches of one kernel class run back to back (stable order
        # otherwise), so that consecutive launches can overlap through
        # programmatic dependent launch and a pair of events brackets each
        # class's batch.
        order = {k: i for i, k in enumerate(PART_CLASSES[part])}
        self.launches.sort(key=lambda l: order[l.kernel])
        self.batches = []
        for l in self.launches:
            if not self.batches or self.batches[-1][0] != l.kernel:
                self.batches.append((l.kernel, []))
            self.batches[-1][1].append(l)
        torch.cuda.synchronize()

    def _pin_in(self, t):
        self.h2d.append((torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t), t))

    def _pin_out(self, t):
        self.d2h.append((t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True)))

    def _weight_copies(self, n, k, seed, copies):
        from int8_quantized_linear_gb300 import capi, synthetic
        w = synthetic.weight(n, k, seed, device=self.device)
        qs = [torch.empty((n, k), dtype=torch.int8, device=self.device) for _ in range(copies)]
        s = torch.empty((n,), dtype=torch.float32, device=self.device)
        capi.quantize_weight_per_channel_int8(w, q=qs[0], scale=s)
        for c in range(1, copies):
            qs[c].copy_(qs[0])
        return w, qs, s

    def _linear(self, kernel, x, q, s, bias, label):
        """The W8A8 linear layer from bf16 activations (quantization fused)."""
        from int8_quantized_linear_gb300 import capi
        m, k = x.shape
        n = q.shape[0]
        y = torch.empty((m, n), dtype=torch.bfloat16, device=self.device)
        self.launches.append(Launch(
            kernel, lambda x=x, q=q, s=s, b=bias, y=y: capi.w8a8_linear(x, q, s, bias=b, y=y),
            bytes_quant(m, k) + bytes_w8a8(m, n, k, bias is not None), 2 * m * n * k, f"{label} M={m}",
            gpu_kernels=capi.i8ql_w8a8_linear_launches(m, n, k)))
        self._pin_out(y)

    def _w8a16(self, kernel, x, q, s, label):
        from int8_quantized_linear_gb300 import capi
        m, k = x.shape
        n = q.shape[0]
        y = torch.empty((m, n), dtype=torch.bfloat16, device=self.device)
        self.launches.append(Launch(kernel, lambda x=x, q=q, s=s, y=y: capi.w8a16_gemm(x, q, s, y=y),
                                    bytes_w8a16(m, n, k), 2 * m * n * k, f"{label} M={m}"))
        self._pin_out(y)

    def _decode(self, seed):
        from int8_quantized_linear_gb300 import capi, synthetic
        dev = self.device
        for si, (name, (n, k)) in enumerate(synthetic.QWEN3_4B_SHAPES.items()):
            w, qs, s = self._weight_copies(n, k, seed + si, 2 * len(DECODE_MS))
            self.launches.append(Launch(
                "quant_w", lambda w=w, q=qs[0], s=s: capi.quantize_weight_per_channel_int8(w, q=q, scale=s),
                bytes_quant(n, k), 0, f"quant_w {name} {n}x{k}"))
            self._pin_in(w)
            for mi, m in enumerate(DECODE_MS):
                x = synthetic.activations(m, k, 100 * seed + 10 * si + mi, device=dev)
                self._pin_in(x)
                qx = torch.empty((m, k), dtype=torch.int8, device=dev)
                sx = torch.empty((m,), dtype=torch.float32, device=dev)
                self.launches.append(Launch(
                    "quant_x", lambda x=x, qx=qx, sx=sx: capi.quantize_act_per_token_int8(x, q=qx, scale=sx),
                    bytes_quant(m, k), 0, f"quant_x {name} M={m}"))
                y8 = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
                self.launches.append(Launch(
                    "w8a8", lambda qx=qx, sx=sx, q=qs[2 * mi], s=s, y=y8: capi.w8a8_gemm(qx, sx, q, s, y=y),
                    bytes_w8a8(m, n, k, False), 2 * m * n * k, f"w8a8 {name} M={m}"))
                self._pin_out(y8)
                self._w8a16("w8a16", x, qs[2 * mi + 1], s, f"w8a16 {name}")
        # DeepSeek-MoE grouped experts: one weight set per token count
        for ti, tokens in enumerate(MOE_TOKENS):
            route = synthetic.moe_routing(tokens, seed=3 + ti)
            counts = np.diff(route.offsets)
            off = torch.from_numpy(route.offsets).to(dev)
            self._pin_in(off)
            for pi, (proj, (n, k)) in enumerate(synthetic.DSMOE_SHAPES.items()):
                e_count = route.experts
                q = torch.empty((e_count, n, k), dtype=torch.int8, device=dev)
                s = torch.empty((e_count, n), dtype=torch.float32, device=dev)
                for e in range(e_count):
                    we = synthetic.weight(n, k, 1000 + 100 * pi + e, device=dev)
                    capi.quantize_weight_per_channel_int8(we, q=q[e], scale=s[e])
                x_tok = synthetic.activations(tokens, k, 900 + 10 * ti + pi, device=dev)
                x = x_tok[torch.from_numpy(route.rows).to(dev)].contiguous()
                self._pin_in(x)
                y = torch.empty((x.shape[0], n), dtype=torch.bfloat16, device=dev)
                self.launches.append(Launch(
                    "grouped", lambda x=x, off=off, q=q, s=s, y=y: capi.grouped_w8a16_gemm(x, off, q, s, y=y),
                    bytes_grouped(counts, n, k), 2 * int(counts.sum()) * n * k, f"grouped {proj} T={tokens}"))
                self._pin_out(y)

    def _prefill(self, seed):
        from int8_quantized_linear_gb300 import synthetic
        for si, (name, (n, k)) in enumerate(synthetic.QWEN3_4B_SHAPES.items()):
            w, qs, s = self._weight_copies(n, k, seed + si, len(PREFILL_MS))
            del w
            bias = synthetic.bias(n, seed + si, device=self.device)
            for mi, m in enumerate(PREFILL_MS):
                x = synthetic.activations(m, k, 100 * seed + 10 * si + mi, device=self.device)
                self._pin_in(x)
                self._linear("w8a8", x, qs[mi], s, bias, f"w8a8_linear {name}")

    def _sweep8b(self, seed):
        from int8_quantized_linear_gb300 import capi, synthetic
        seed += 40
        for si, (name, (n, k)) in enumerate(synthetic.QWEN3_8B_SHAPES.items()):
            w, qs, s = self._weight_copies(n, k, seed + si, len(SWEEP_W8A16_MS) + len(SWEEP_W8A8_MS))
            del w
            c = 0
            for m in SWEEP_W8A16_MS:
                x = synthetic.activations(m, k, 100 * seed + 10 * si + m, device=self.device)
                self._pin_in(x)
                self._w8a16("w8a16", x, qs[c], s, f"w8a16 {name}")
                c += 1
            for m in SWEEP_W8A8_MS:
                x = synthetic.activations(m, k, 100 * seed + 10 * si + m + 1, device=self.device)
                self._pin_in(x)
                # above the decode range a W8A8 call runs on the tensor-core kernel
                kind = "w8a8_decode" if m <= capi.I8QL_W8A8_DECODE_MAX_M else "w8a8_prefill"
                self._linear(kind, x, qs[c], s, None, f"w8a8_linear {name}")
                c += 1

    def _fp8(self, seed):
        from int8_quantized_linear_gb300 import capi, synthetic
        for si, (name, (n, k)) in enumerate(synthetic.QWEN3_4B_SHAPES.items()):
            w = synthetic.weight(n, k, seed + si, device=self.device)
            q0, s = capi.quantize_weight_per_channel_fp8(w)
            del w
            bias = synthetic.bias(n, seed + si, device=self.device)
            for mi, m in enumerate(PREFILL_MS):
                q = q0 if mi == 0 else q0.clone()
                x = synthetic.activations(m, k, 100 * seed + 10 * si + mi, device=self.device)
                self._pin_in(x)
                y = torch.empty((m, n), dtype=torch.bfloat16, device=self.device)
                self.launches.append(Launch(
                    "fp8", lambda x=x, q=q, s=s, b=bias, y=y: capi.w8a8_fp8_linear(x, q, s, bias=b, y=y),
                    bytes_quant(m, k) + bytes_w8a8(m, n, k, True), 2 * m * n * k, f"fp8_linear {name} M={m}",
                    gpu_kernels=2))
                self._pin_out(y)

    def _w4(self, seed):
        from int8_quantized_linear_gb300 import capi, synthetic
        seed += 40
        for si, (name, (n, k)) in enumerate(synthetic.QWEN3_8B_SHAPES.items()):
            w = synthetic.weight(n, k, seed + si, device=self.device)
            self._pin_in(w)
            q0, s0 = capi.quantize_weight_w4_g128(w)
            self.launches.append(Launch(
                "quant_w4", lambda w=w, q=q0, s=s0: capi.quantize_weight_w4_g128(w, q=q, scale=s),
                bytes_quant_w4(n, k), 0, f"quant_w4 {name}"))
            for mi, m in enumerate(W4_MS):
                q = q0.clone()
                x = synthetic.activations(m, k, 100 * seed + 10 * si + mi, device=self.device)
                self._pin_in(x)
                y = torch.empty((m, n), dtype=torch.bfloat16, device=self.device)
                self.launches.append(Launch(
                    "w4a16", lambda x=x, q=q, s=s0, y=y: capi.w4a16_gemm(x, q, s, y=y),
                    bytes_w4a16(m, n, k), 2 * m * n * k, f"w4a16 {name} M={m}"))
                self._pin_out(y)

    def _fused(self, seed):
        from int8_quantized_linear_gb300 import synthetic
        for si, (name, (n, k)) in enumerate(synthetic.QWEN3_4B_SHAPES.items()):
            w, qs, s = self._weight_copies(n, k, seed + si, len(DECODE_MS))
            del w
            for mi, m in enumerate(DECODE_MS):
                x = synthetic.activations(m, k, 100 * seed + 10 * si + mi, device=self.device)
                self._pin_in(x)
                y = torch.empty((m, n), dtype=torch.bfloat16, device=self.device)
                self.launches.append(Launch(
                    "w8a8_fused", lambda x=x, q=qs[mi], s=s, y=y: self._capi.w8a8_linear(x, q, s, y=y, fused=True),
                    bytes_linear_fused(m, n, k, False), 2 * m * n * k, f"w8a8_linear_fused {name} M={m}"))
                self._pin_out(y)

    def _moe(self, seed):
        from int8_quantized_linear_gb300 import capi, synthetic
        dev = self.device
        (inter2, hidden), (_, inter) = synthetic.DSMOE_SHAPES["gate_up"], synthetic.DSMOE_SHAPES["down"]
        e_count = synthetic.DSMOE_ROUTED + synthetic.DSMOE_SHARED
        for ti, tokens in enumerate(MOE_TOKENS):
            weights = []
            for pi, (proj, (n, k)) in enumerate(synthetic.DSMOE_SHAPES.items()):
                q = torch.empty((e_count, n, k), dtype=torch.int8, device=dev)
                s = torch.empty((e_count, n), dtype=torch.float32, device=dev)
                for e in range(e_count):
                    we = synthetic.weight(n, k, 1000 + 100 * pi + e, device=dev)
                    capi.quantize_weight_per_channel_int8(we, q=q[e], scale=s[e])
                weights += [q, s]
            x = synthetic.activations(tokens, hidden, 600 + ti, device=dev)
            logits = synthetic.gate_logits(tokens, synthetic.DSMOE_ROUTED, 3 + ti).to(dev)
            self._pin_in(x)
            self._pin_in(logits)
            out = torch.empty((tokens, hidden), dtype=torch.bfloat16, device=dev)
            counts = np.diff(synthetic.moe_routing(tokens, seed=3 + ti).offsets)
            rows = int(counts.sum())
            self.launches.append(Launch(
                "moe_mlp", lambda x=x, lg=logits, w=weights, o=out: capi.moe_expert_mlp_w8a16(
                    x, lg, synthetic.DSMOE_TOPK, synthetic.DSMOE_SHARED, w[0], w[1], w[2], w[3], out=o),
                bytes_moe(counts, tokens, hidden, inter, synthetic.DSMOE_ROUTED),
                2 * rows * (inter2 * hidden + hidden * inter), f"moe_mlp T={tokens}",
                gpu_kernels=4 if tokens <= 32 else 5))  # routing is one launch up to 32 tokens
            self._pin_out(out)

    def run(self, events=None):
        """One step; events[b] = (start, end) brackets batch b."""
        for b, (_, launches) in enumerate(self.batches):
            if events is not None:
                events[b][0].record()
            for l in launches:
                l.fn()
            if events is not None:
                events[b][1].record()

    @property
    def step_bytes(self):
        return sum(l.bytes for l in self.launches)

    def step_flops(self, classes):
        return sum(l.flops for l in self.launches if l.kernel in classes)


def _event(external):
    try:
        return torch.cuda.Event(enable_timing=True, external=external)
    except TypeError:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "", 1).isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4) if r[5 + j].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- oracle (CPU) arm

def oracle_step(sample):
    """Time the CPU oracle over a row sample of a workload; returns
    (algorithmic bytes, GEMM ops 2*M*N*K, seconds)."""
    import oracle
    total_b, total_ops, total_s = 0, 0, 0.0
    for item in sample:
        t0 = time.perf_counter()
        kind = item[0]
        if kind == "quant":
            _, src = item
            oracle.quant_rows(src)
            total_b += bytes_quant(*src.shape)
        elif kind in ("w8a8", "linear"):
            # per-token quantization then the W8A8 GEMM, counted as the GPU
            # step counts it (one pass over bf16 tokens for "linear")
            _, xb, qw, sw, bias = item
            qx, sx = oracle.quant_rows(xb)
            oracle.w8a8(qx, sx, qw, sw, bias)
            m, k = xb.shape
            if kind == "linear":
                total_b += bytes_linear_fused(m, qw.shape[0], k, bias is not None)
            else:
                total_b += bytes_quant(m, k) + bytes_w8a8(m, qw.shape[0], k, bias is not None)
            total_ops += 2 * m * qw.shape[0] * k
        elif kind == "w8a16":
            _, xb, qw, sw = item
            oracle.w8a16(xb, qw, sw)
            total_b += bytes_w8a16(xb.shape[0], qw.shape[0], xb.shape[1])
            total_ops += 2 * xb.shape[0] * qw.shape[0] * xb.shape[1]
        elif kind == "grouped":
            _, xb, off, q, s = item
            oracle.grouped_w8a16(xb, off, q, s)
            total_b += bytes_grouped(np.diff(off), q.shape[1], q.shape[2])
            total_ops += 2 * xb.shape[0] * q.shape[1] * q.shape[2]
        total_s += time.perf_counter() - t0
    return total_b, total_ops, total_s


def oracle_rate(part, nbytes, ops, seconds):
    """The oracle's rate in the part's unit: GB/s for decode, TOPS (2*M*N*K
    of the W8A8 GEMMs) for prefill."""
    if part == "decode":
        return nbytes / seconds / 1e9, "GB/s"
    return ops / seconds / 1e12, "TOPS"


def build_oracle_sample(part, row_frac, seed=1):
    """The part's workload with every weight cut to a fraction of its output
    rows (prefill: every M too; grouped experts: a fraction of their rows),
    drawn on the CPU from the same generators."""
    import oracle
    from int8_quantized_linear_gb300 import synthetic
    sample = []
    ms = DECODE_MS if part == "decode" else PREFILL_MS
    for si, (name, (n, k)) in enumerate(synthetic.QWEN3_4B_SHAPES.items()):
        nr = max(16, int(n * row_frac))
        w = synthetic.bf16_bits(synthetic.weight(nr, k, seed + si))
        qw, sw = oracle.quant_rows(w)
        bias = None if part == "decode" else synthetic.bf16_bits(synthetic.bias(nr, seed + si))
        if part == "decode":
            sample.append(("quant", w))
        for mi, m in enumerate(ms):
            mr = m if part == "decode" else max(1, int(m * row_frac))
            xb = synthetic.bf16_bits(synthetic.activations(mr, k, 100 * seed + 10 * si + mi))
            sample.append(("w8a8", xb, qw, sw, bias))
            if part == "decode":
                sample.append(("w8a16", xb, qw, sw))
    if part == "decode":
        experts = {}  # the same expert weights serve every token count
        for ti, tokens in enumerate(MOE_TOKENS):
            route = synthetic.moe_routing(tokens, seed=3 + ti)
            for pi, (proj, (n, k)) in enumerate(synthetic.DSMOE_SHAPES.items()):
                nr = max(16, int(n * row_frac))
                if pi not in experts:
                    q = np.empty((route.experts, nr, k), np.int8)
                    s = np.empty((route.experts, nr), np.float32)
                    for e in range(route.experts):
                        q[e], s[e] = oracle.quant_rows(
                            synthetic.bf16_bits(synthetic.weight(nr, k, 1000 + 100 * pi + e)))
                    experts[pi] = (q, s)
                q, s = experts[pi]
                x_tok = synthetic.activations(tokens, k, 900 + 10 * ti + pi)
                xb = synthetic.bf16_bits(x_tok[torch.from_numpy(route.rows)])
                sample.append(("grouped", xb, route.offsets, q, s))
    return sample


def cpu_baseline(part, row_frac, min_seconds=3.0):
    """The oracle on a bounded sample of the part, first on one thread, then
    on every core: {value (all cores), cores, single_thread {...}, ...}."""
    import oracle
    sample = build_oracle_sample(part, row_frac)
    scope = ("the whole workload" if row_frac >= 1 else
             f"the workload with every weight cut to {row_frac:.4g} of its output rows"
             + (" and every M to the same fraction" if part == "prefill" else " (grouped experts too)"))
    out = {}
    for label, threads in (("single", 1), ("all", os.cpu_count() or 1)):
        used = oracle.set_threads(threads)
        b, o, s, passes = 0, 0, 0.0, 0
        while passes == 0 or (label == "all" and s < min_seconds and passes < 10):
            bb, oo, ss = oracle_step(sample)
            b, o, s, passes = b + bb, o + oo, s + ss, passes + 1
        rate, unit = oracle_rate(part, b, o, s)
        out[label] = {"value": rate, "unit": unit, "cores": used, "seconds": s, "passes": passes}
    oracle.set_threads(os.cpu_count() or 1)
    a, one = out["all"], out["single"]
    return {"value": a["value"], "unit": a["unit"], "cores": a["cores"], "kind": "oracle",
            "sample": f"{a['passes']} pass(es) of {scope}; {a['seconds']:.1f} s on {a['cores']} threads",
            "nproc": os.cpu_count(),
            "single_thread": {"value": one["value"], "unit": one["unit"], "cores": 1,
                              "sample": f"{one['passes']} pass(es); {one['seconds']:.1f} s on 1 thread"}}


# ---------------------------------------------------------------- distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (the slowest rank sets the job time)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- arms

def run_reference(args, world, rank):
    """The oracle on the host cores (every core): each step is one pass over
    a bounded row sample of the decode part (the top-level metric)."""
    if rank != 0:
        return 0
    import oracle
    part = "prefill" if args.workload in ("prefill", "fp8") else "decode"
    frac = args.ref_row_frac
    sample = build_oracle_sample(part, frac)
    cores = oracle.set_threads(os.cpu_count() or 1)
    for _ in range(args.warmup):
        oracle_step(sample)
    b_tot, o_tot, s_tot = 0, 0, 0.0
    for _ in range(args.steps):
        b, o, s = oracle_step(sample)
        b_tot += b
        o_tot += o
        s_tot += s
    rate, unit = oracle_rate(part, b_tot, o_tot, s_tot)
    desc = (f"every weight cut to {frac:.4g} of its output rows (grouped experts too), "
            f"{'M in {1,4,8}' if part == 'decode' else 'M scaled by the same fraction'}; "
            f"C oracle on {cores} threads")
    line = {
        "metric": METRIC, "value": rate, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000 * s_tot / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": workload_name(part), "sample": desc},
        "cpu_baseline": {"value": rate, "unit": unit, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": rate, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# Parts whose decode GEMMs run with early weight loads (the serving option of
# i8ql_set_early_weight_loads): their weights are static during the step, and
# no GEMM follows a kernel that writes its weights.
EARLY_WEIGHT_PARTS = ("decode", "sweep8b", "fused")


def time_part(part, args, world, local, stream):
    """Build, capture and time one part; returns its measurements."""
    from int8_quantized_linear_gb300 import capi
    capi.i8ql_set_early_weight_loads(part in EARLY_WEIGHT_PARTS)
    try:
        return _time_part(part, args, world, local, stream)
    finally:
        capi.i8ql_set_early_weight_loads(False)


def _time_part(part, args, world, local, stream):
    from int8_quantized_linear_gb300 import capi
    device = torch.device("cuda", local)
    wl = Workload(part, device)
    n_launch = sum(l.gpu_kernels for l in wl.launches)  # library kernels per step
    n_batch = len(wl.batches)

    # eager pass: per-device initialisation happens outside graph capture
    with torch.cuda.stream(stream):
        wl.run()
    torch.cuda.synchronize()
    if capi.i8ql_get_device_error(stream) != capi.I8QL_OK:
        raise RuntimeError(f"{part}: kernel fault word set after the eager pass")

    external = _event(True) is not None
    use_graph = not args.no_graph and external
    steps = args.steps
    if use_graph:
        g_warm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_warm, stream=stream):
            wl.run()
        events = [[(_event(True), _event(True)) for _ in range(n_batch)] for _ in range(steps)]
        g_timed = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_timed, stream=stream):
            for s in range(steps):
                wl.run(events[s])
    else:
        g_warm = None
        events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n_batch)] for _ in range(steps)]

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            if use_graph:
                g_warm.replay()
            else:
                wl.run()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start
    if args.profile_timed:
        torch.cuda.profiler.start()
    with torch.cuda.stream(stream):
        start.record(stream)
        if use_graph:
            g_timed.replay()
        else:
            for s in range(steps):
                wl.run(events[s])
        end.record(stream)
    torch.cuda.synchronize()
    if args.profile_timed:
        torch.cuda.profiler.stop()
    clk = clocks.stop()
    barrier(world)
    ms_step = max_over_ranks(start.elapsed_time(end), world) / steps
    fault = capi.i8ql_get_device_error(stream)
    if fault != capi.I8QL_OK:
        raise RuntimeError(f"{part}: kernel fault word set: {capi.status_string(fault)}")

    # per-class live timings over the timed region
    per = {}
    for s in range(steps):
        for b, (kernel, launches) in enumerate(wl.batches):
            a, z = events[s][b]
            e = per.setdefault(kernel, {"launches": 0, "ms": 0.0, "bytes": 0, "flops": 0})
            e["launches"] += len(launches)
            e["ms"] += a.elapsed_time(z)
            e["bytes"] += sum(l.bytes for l in launches)
            e["flops"] += sum(l.flops for l in launches)
    peaks, peak_src = load_peaks()
    kernels = {}
    for name, e in per.items():
        gbs = e["bytes"] / (e["ms"] / 1e3) / 1e9
        entry = {"launches": e["launches"], "us_per_launch": 1e3 * e["ms"] / e["launches"],
                 "share": e["ms"] / sum(v["ms"] for v in per.values()),
                 "GB/s": gbs, "hbm_frac": gbs / peaks["hbm_gbs"]}
        if e["flops"]:
            tops = e["flops"] / (e["ms"] / 1e3) / 1e12
            entry["TOPS"] = tops
            if (part, name) in TENSOR_CLASSES:
                entry["tensor_frac"] = tops / (peaks["bf16_tflops"] * TENSOR_CLASSES[(part, name)])
        kernels[name] = entry

    e2e = run_e2e(args, wl, stream, g_warm, world, part)
    out = {"wl": wl, "per": per, "kernels": kernels, "ms_step": ms_step, "clocks": clk, "e2e": e2e,
           "launches": n_launch * steps, "graph": use_graph, "peaks": (peaks, peak_src)}
    del g_warm
    if use_graph:
        del g_timed
    return out


def roofline(part, res, kernel=None):
    """Roofline of the dominant kernel class of a part (or of `kernel`)."""
    per = res["per"]
    peaks, peak_src = res["peaks"]
    dom = kernel or max(per, key=lambda k: per[k]["ms"])
    d = per[dom]
    per_launch_bytes = d["bytes"] / d["launches"]
    if (part, dom) in TENSOR_CLASSES:
        ratio = TENSOR_CLASSES[(part, dom)]
        achieved = d["flops"] / (d["ms"] / 1e3) / 1e12
        peak = peaks["bf16_tflops"] * ratio
        pipe = "fp8 kind::f8f6f4 pipe" if ratio == 2.0 else "fp16 kind::f16 pipe"
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "peak_source": f"{peak_src} bf16_tflops burst x {ratio:g} ({pipe}, nominal ratio {ratio:g})",
                "kernel": dom}
    else:
        achieved = per_launch_bytes / (d["ms"] / d["launches"] / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peak_src} hbm_gbs", "kernel": dom}
    roof["traffic"] = ncu_traffic(dom, part)
    roof["algorithmic_bytes_per_launch"] = per_launch_bytes
    return roof


ALL_PARTS = ("decode", "prefill", "sweep8b", "fp8", "w4", "moe", "fused")


def part_value(part, wl, ms, world):
    """The part's throughput in its unit: TOPS (2*M*N*K of the tensor-core
    launches) for the prefill parts, algorithmic GB/s otherwise."""
    if part in ("prefill", "fp8"):
        return world * wl.step_flops(set(PART_CLASSES[part])) / (ms / 1e3) / 1e12, "TOPS"
    return world * wl.step_bytes / (ms / 1e3) / 1e9, "GB/s"


def run_ours(args, world, rank, local):
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    stream = torch.cuda.Stream(device)
    parts = ALL_PARTS if args.workload == "all" else (args.workload,)
    results = {}
    for part in parts:
        results[part] = time_part(part, args, world, local, stream)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    top = parts[0]
    r = results[top]
    value, unit = part_value(top, r["wl"], r["ms_step"], world)
    reasons = sorted({x for res in results.values() for x in res["clocks"].get("reasons", [])})
    clocks = dict(r["clocks"])
    clocks["reasons"] = reasons
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": " + ".join(workload_name(p) for p in parts), "parallelism": f"replicas x{world}",
                   "top_level": workload_name(top),
                   "l2": "inputs larger than L2: every GEMM launch reads its own weight copy, "
                         ">1 GB touched per step of each part",
                   "early_weight_loads": list(EARLY_WEIGHT_PARTS),
                   "graph": r["graph"]},
        "roofline": roofline(top, r),
        "kernels": r["kernels"],
        "gpu_launches": sum(res["launches"] for res in results.values()),
        "clocks": clocks,
        "e2e": r["e2e"],
    }
    if "prefill" in results and top != "prefill":
        p = results["prefill"]
        tops = world * p["wl"].step_flops({"w8a8"}) / (p["ms_step"] / 1e3) / 1e12
        line["prefill"] = {"workload": workload_name("prefill"), "value": tops, "unit": "TOPS",
                           "ms_per_step": p["ms_step"], "roofline": roofline("prefill", p),
                           "kernels": p["kernels"], "e2e": p["e2e"], "clocks": p["clocks"],
                           "gpu_launches": p["launches"]}
    if "sweep8b" in results:
        sw = results["sweep8b"]
        block = {"workload": workload_name("sweep8b"), "ms_per_step": sw["ms_step"], "kernels": sw["kernels"],
                 "e2e": sw["e2e"], "clocks": sw["clocks"], "gpu_launches": sw["launches"],
                 "roofline": {k: roofline("sweep8b", sw, k) for k in sw["per"]}}
        dec = [l for l in sw["wl"].launches if l.kernel != "w8a8_prefill"]
        pre = [l for l in sw["wl"].launches if l.kernel == "w8a8_prefill"]
        ms_dec = sum(sw["per"][k]["ms"] for k in ("w8a16", "w8a8_decode")) / args.steps
        ms_pre = sw["per"]["w8a8_prefill"]["ms"] / args.steps
        block["decode_GB/s"] = world * sum(l.bytes for l in dec) / (ms_dec / 1e3) / 1e9
        block["prefill_TOPS"] = world * sum(l.flops for l in pre) / (ms_pre / 1e3) / 1e12
        if top == "sweep8b":
            line.update({k: v for k, v in block.items() if k in ("kernels",)})
        else:
            line["qwen3_8b_sweep"] = block
    for part, key in (("fp8", "fp8_prefill"), ("w4", "w4a16_decode"), ("moe", "moe_mlp"),
                      ("fused", "w8a8_linear_one_launch")):
        if part in results and top != part:
            b = results[part]
            v, u = part_value(part, b["wl"], b["ms_step"], world)
            line[key] = {"workload": workload_name(part), "value": v, "unit": u, "ms_per_step": b["ms_step"],
                         "roofline": roofline(part, b), "kernels": b["kernels"], "e2e": b["e2e"],
                         "clocks": b["clocks"], "gpu_launches": b["launches"]}
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        frac = args.cpu_row_frac if args.cpu_row_frac is not None else (1 / 8 if top in ("prefill", "fp8") else 1 / 2)
        cpu_part = "prefill" if top in ("prefill", "fp8") else "decode"
        line["cpu_baseline"] = cpu_baseline(cpu_part, frac)
        if "prefill" in line:
            line["prefill"]["cpu_baseline"] = cpu_baseline("prefill", 1 / 8)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


class _Staging:
    """One pinned host buffer and one device buffer holding a list of
    tensors back to back (256-byte aligned), so that a step's transfers are
    one host<->device copy each way plus device-side copies to and from the
    tensors themselves (dozens of small host copies each cost far more than
    their bytes)."""

    def __init__(self, tensors, device, host=True):
        self.spans = []
        off = 0
        for t in tensors:
            n = t.numel() * t.element_size()
            self.spans.append((off, n))
            off += (n + 255) // 256 * 256
        self.host = torch.empty(max(off, 1), dtype=torch.uint8, pin_memory=True) if host else None
        self.dev = torch.empty(max(off, 1), dtype=torch.uint8, device=device)

    def views(self, buf, tensors):
        return [buf[o:o + n].view(t.dtype).view(t.shape) for (o, n), t in zip(self.spans, tensors)]


def run_e2e(args, wl, stream, graph, world, part):
    """Same step through the public API with host buffers: every input comes
    from pinned host memory and every result goes back to it, inside the
    timed region.  Each way is one host<->device copy of a staging buffer
    plus device-side copies to or from the step's tensors, and the copies
    are pipelined the way a serving loop runs them: step s+1's inputs go up
    (copy stream) and step s-1's results come down (a second copy stream)
    while step s computes, through two device staging buffers each way."""
    steps = max(1, min(args.steps, 10))
    h2d = sum(h.numel() * h.element_size() for h, _ in wl.h2d)
    d2h = sum(h.numel() * h.element_size() for _, h in wl.d2h)
    device = wl.device
    in_t, out_t = [h for h, _ in wl.h2d], [h for _, h in wl.d2h]
    ins = [_Staging(in_t, device, host=(i == 0)) for i in range(2)]
    outs = [_Staging(out_t, device, host=(i == 0)) for i in range(2)]
    for v, host in zip(ins[0].views(ins[0].host, in_t), in_t):
        v.copy_(host)  # the inputs' host bytes, once, outside the timed region
    in_dev = [st.views(st.dev, in_t) for st in ins]
    out_dev = [st.views(st.dev, out_t) for st in outs]
    up, down = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    ev = lambda: torch.cuda.Event()
    in_ready, in_free = [ev(), ev()], [ev(), ev()]
    out_ready, out_free = [ev(), ev()], [ev(), ev()]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    start.record(stream)
    up.wait_event(start)
    down.wait_event(start)
    for s in range(steps):
        b = s % 2
        with torch.cuda.stream(up):
            if s >= 2:
                up.wait_event(in_free[b])
            ins[b].dev.copy_(ins[0].host, non_blocking=True)
            in_ready[b].record(up)
        with torch.cuda.stream(stream):
            stream.wait_event(in_ready[b])
            for src, (_, devt) in zip(in_dev[b], wl.h2d):
                devt.copy_(src, non_blocking=True)
            in_free[b].record(stream)
            if graph is not None:
                graph.replay()
            else:
                wl.run()
            if s >= 2:
                stream.wait_event(out_free[b])
            for dst, (devt, _) in zip(out_dev[b], wl.d2h):
                dst.copy_(devt, non_blocking=True)
            out_ready[b].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(out_ready[b])
            outs[0].host.copy_(outs[b].dev, non_blocking=True)
            out_free[b].record(down)
    stream.wait_stream(up)
    stream.wait_stream(down)
    end.record(stream)
    torch.cuda.synchronize()
    for v, (_, host) in zip(outs[0].views(outs[0].host, out_t), wl.d2h):
        host.copy_(v)  # results where the caller keeps them (outside the timed region)
    ms = max_over_ranks(start.elapsed_time(end), world) / steps
    value, unit = part_value(part, wl, ms, world)
    return {"value": value, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": steps, "pipelined": True}


def run_single(args, local):
    """One kernel at one shape, eager launches timed with CUDA events; the
    weights rotate through enough copies to exceed L2.  Used for profiling."""
    from int8_quantized_linear_gb300 import capi, synthetic
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    parts = args.single.split(":")
    kind, dims = parts[0], [int(v) for v in parts[1:]]
    l2 = 256 << 20
    if kind in ("w8a8", "w8a16", "linear"):
        m, n, k = dims
        copies = max(1, -(-l2 // (n * k)))
        w = synthetic.weight(n, k, 1, device=dev)
        q0, s = capi.quantize_weight_per_channel_int8(w)
        del w
        qs = [q0] + [q0.clone() for _ in range(copies - 1)]
        x = synthetic.activations(m, k, 2, device=dev)
        qx, sx = capi.quantize_act_per_token_int8(x)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        if kind == "w8a8":
            fns = [lambda q=q: capi.w8a8_gemm(qx, sx, q, s, y=y) for q in qs]
            nbytes, flops = bytes_w8a8(m, n, k, False), 2 * m * n * k
        elif kind == "linear":
            fns = [lambda q=q: capi.w8a8_linear(x, q, s, y=y) for q in qs]
            nbytes, flops = bytes_quant(m, k) + bytes_w8a8(m, n, k, False), 2 * m * n * k
        else:
            fns = [lambda q=q: capi.w8a16_gemm(x, q, s, y=y) for q in qs]
            nbytes, flops = bytes_w8a16(m, n, k), 2 * m * n * k
    elif kind in ("w4a16", "fp8"):
        m, n, k = dims
        w = synthetic.weight(n, k, 1, device=dev)
        x = synthetic.activations(m, k, 2, device=dev)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        if kind == "w4a16":
            q0, s = capi.quantize_weight_w4_g128(w)
            copies = max(1, -(-l2 // (n * k // 2)))
            qs = [q0] + [q0.clone() for _ in range(copies - 1)]
            fns = [lambda q=q: capi.w4a16_gemm(x, q, s, y=y) for q in qs]
            nbytes, flops = bytes_w4a16(m, n, k), 2 * m * n * k
        else:
            q0, s = capi.quantize_weight_per_channel_fp8(w)
            copies = max(1, -(-l2 // (n * k)))
            qs = [q0] + [q0.clone() for _ in range(copies - 1)]
            fns = [lambda q=q: capi.w8a8_fp8_linear(x, q, s, y=y) for q in qs]
            nbytes, flops = bytes_quant(m, k) + bytes_w8a8(m, n, k, False), 2 * m * n * k
        del w
    elif kind == "quant_w4":
        r, k = dims
        copies = max(1, -(-l2 // (2 * r * k)))
        ws = [synthetic.weight(r, k, 1 + c, device=dev) for c in range(copies)]
        q = torch.empty((r, k // 2), dtype=torch.uint8, device=dev)
        sc = torch.empty((r, k // 128), dtype=torch.bfloat16, device=dev)
        fns = [lambda w=w: capi.quantize_weight_w4_g128(w, q=q, scale=sc) for w in ws]
        nbytes, flops = bytes_quant_w4(r, k), 0
    elif kind == "moe":
        (tokens,) = dims
        (inter2, hidden), (_, inter) = synthetic.DSMOE_SHAPES["gate_up"], synthetic.DSMOE_SHAPES["down"]
        e_count = synthetic.DSMOE_ROUTED + synthetic.DSMOE_SHARED
        weights = []
        for pi, (n, k) in enumerate(synthetic.DSMOE_SHAPES.values()):
            q = torch.empty((e_count, n, k), dtype=torch.int8, device=dev)
            sc = torch.empty((e_count, n), dtype=torch.float32, device=dev)
            for e in range(e_count):
                capi.quantize_weight_per_channel_int8(synthetic.weight(n, k, 1000 + 100 * pi + e, device=dev),
                                                      q=q[e], scale=sc[e])
            weights += [q, sc]
        x = synthetic.activations(tokens, hidden, 600, device=dev)
        logits = synthetic.gate_logits(tokens, synthetic.DSMOE_ROUTED, 3).to(dev)
        out = torch.empty((tokens, hidden), dtype=torch.bfloat16, device=dev)
        fns = [lambda: capi.moe_expert_mlp_w8a16(x, logits, synthetic.DSMOE_TOPK, synthetic.DSMOE_SHARED,
                                                 *weights, out=out)]
        counts = np.diff(synthetic.moe_routing(tokens, seed=3).offsets)
        nbytes = bytes_moe(counts, tokens, hidden, inter, synthetic.DSMOE_ROUTED)
        flops = 2 * int(counts.sum()) * (inter2 * hidden + hidden * inter)
    elif kind == "grouped":
        tokens, proj = dims[0], ("gate_up", "down")[dims[1]]
        n, k = synthetic.DSMOE_SHAPES[proj]
        route = synthetic.moe_routing(tokens, seed=3)
        counts = np.diff(route.offsets)
        off = torch.from_numpy(route.offsets).to(dev)
        e_count = route.experts
        qs = []
        for c in range(2):  # two weight sets of more than L2 each
            q = torch.empty((e_count, n, k), dtype=torch.int8, device=dev)
            sc = torch.empty((e_count, n), dtype=torch.float32, device=dev)
            for e in range(e_count):
                capi.quantize_weight_per_channel_int8(synthetic.weight(n, k, 1000 + e, device=dev), q=q[e], scale=sc[e])
            qs.append((q, sc))
        x = synthetic.activations(route.total_rows, k, 7, device=dev)
        y = torch.empty((route.total_rows, n), dtype=torch.bfloat16, device=dev)
        fns = [lambda q=q, sc=sc: capi.grouped_w8a16_gemm(x, off, q, sc, y=y) for q, sc in qs]
        nbytes, flops = bytes_grouped(counts, n, k), 2 * int(counts.sum()) * n * k
    elif kind == "quant":
        r, k = dims
        copies = max(1, -(-l2 // (2 * r * k)))
        ws = [synthetic.weight(r, k, 1 + c, device=dev) for c in range(copies)]
        q = torch.empty((r, k), dtype=torch.int8, device=dev)
        sc = torch.empty((r,), dtype=torch.float32, device=dev)
        fns = [lambda w=w: capi.quantize_weight_per_channel_int8(w, q=q, scale=sc) for w in ws]
        nbytes, flops = bytes_quant(r, k), 0
    else:
        raise SystemExit(f"unknown kernel {kind}")
    for i in range(args.warmup):
        fns[i % len(fns)]()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        ev[i][0].record()
        fns[i % len(fns)]()
        ev[i][1].record()
    torch.cuda.synchronize()
    times = sorted(a.elapsed_time(b) for a, b in ev)
    med = times[len(times) // 2]
    out = {"single": args.single, "us_median": 1e3 * med, "us_min": 1e3 * times[0],
           "GB/s": nbytes / (med / 1e3) / 1e9, "copies": len(fns)}
    if flops:
        out["TOPS"] = flops / (med / 1e3) / 1e12
    print(json.dumps(out), flush=True)
    return 0


SHAPE_GROUPS = ("decode", "prefill", "fp8", "w4", "grouped", "moe", "fused")


def _graph_us(calls, reps=3):
    """Median over three replays of a graph of `reps` passes over `calls`:
    microseconds per call."""
    for c in calls:
        c()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            for c in calls:
                c()
    g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e3 / reps / len(calls))
    del g
    return statistics.median(times)


def _copies(nbytes):
    """Weight copies a graph pass rotates through: more than L2 in total."""
    return max(2, min(24, int(600e6 // max(1, nbytes)) + 1))


def run_shapes(args, local):
    """Per-shape timings of every path (the tables of the measured results):
    each row is one call, replayed back to back in a CUDA graph over weight
    copies that together exceed L2, so every call streams its weights from
    HBM.  Rates are algorithmic bytes or 2*M*N*K per call time; fractions are
    of the measured copy bandwidth and bf16 peak (FP8 against twice it)."""
    from int8_quantized_linear_gb300 import capi, synthetic
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, _ = load_peaks()
    hbm, bf16 = peaks["hbm_gbs"], peaks["bf16_tflops"]
    groups = SHAPE_GROUPS if args.shapes == "all" else tuple(args.shapes.split(","))
    for g in groups:
        if g not in SHAPE_GROUPS:
            raise SystemExit(f"unknown shape group {g}")

    def row(group, call, shape, m, n, k, us, nbytes=None, flops=None, peak_scale=1.0, **extra):
        out = {"group": group, "call": call, "shape": shape, "M": m, "N": n, "K": k, "us": round(us, 3)}
        if nbytes is not None:
            out["GB/s"] = round(nbytes / us / 1e3, 1)
            out["hbm_frac"] = round(nbytes / us / 1e3 / hbm, 4)
        if flops is not None:
            out["TOPS"] = round(flops / us / 1e6, 1)
            out["tensor_frac"] = round(flops / us / 1e6 / (bf16 * peak_scale), 4)
        out.update(extra)
        print(json.dumps(out), flush=True)

    i8 = {}  # int8 per-channel weights of the Qwen3-4B shapes, shared by the groups that use them

    def int8_weights(name, n, k):
        if name not in i8:
            q, s = capi.quantize_weight_per_channel_int8(synthetic.weight(n, k, 1, device=dev))
            i8[name] = ([q] + [q.clone() for _ in range(_copies(n * k) - 1)], s)
        return i8[name]

    if "decode" in groups:
        for name, (n, k) in synthetic.QWEN3_4B_SHAPES.items():
            ws = [synthetic.weight(n, k, 1 + c, device=dev) for c in range(_copies(2 * n * k))]
            q = torch.empty((n, k), dtype=torch.int8, device=dev)
            s = torch.empty((n,), dtype=torch.float32, device=dev)
            us = _graph_us([lambda w=w: capi.quantize_weight_per_channel_int8(w, q=q, scale=s) for w in ws])
            row("decode", "quantize_weight_per_channel_int8", name, 0, n, k, us, nbytes=bytes_quant(n, k))
            del ws
            qs, s = int8_weights(name, n, k)
            for m in DECODE_MS:
                x = synthetic.activations(m, k, 3, device=dev)
                qx, sx = capi.quantize_act_per_token_int8(x)
                y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
                us = _graph_us([lambda q=q: capi.w8a16_gemm(x, q, s, y=y) for q in qs])
                row("decode", "w8a16_gemm", name, m, n, k, us, nbytes=bytes_w8a16(m, n, k), flops=2 * m * n * k)
                us = _graph_us([lambda q=q: capi.w8a8_gemm(qx, sx, q, s, y=y) for q in qs])
                row("decode", "w8a8_gemm", name, m, n, k, us, nbytes=bytes_w8a8(m, n, k, False),
                    flops=2 * m * n * k)
    if "fused" in groups:
        for name, (n, k) in synthetic.QWEN3_4B_SHAPES.items():
            qs, s = int8_weights(name, n, k)
            for m in DECODE_MS:
                x = synthetic.activations(m, k, 3, device=dev)
                y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
                us1 = _graph_us([lambda q=q: capi.w8a8_linear(x, q, s, y=y, fused=True) for q in qs])
                us2 = _graph_us([lambda q=q: capi.w8a8_linear(x, q, s, y=y) for q in qs])
                row("fused", "w8a8_linear_fused", name, m, n, k, us1, nbytes=bytes_linear_fused(m, n, k, False),
                    w8a8_linear_us=round(us2, 3), w8a8_linear_launches=capi.i8ql_w8a8_linear_launches(m, n, k))
    if "prefill" in groups:
        for name, (n, k) in synthetic.QWEN3_4B_SHAPES.items():
            qs, s = int8_weights(name, n, k)
            bias = synthetic.bias(n, 2, device=dev)
            for m in PREFILL_MS:
                x = synthetic.activations(m, k, 3, device=dev)
                y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
                us = _graph_us([lambda q=q: capi.w8a8_linear(x, q, s, bias=bias, y=y) for q in qs])
                row("prefill", "w8a8_linear", name, m, n, k, us, flops=2 * m * n * k,
                    plan=list(capi.i8ql_w8a8_plan(m, n, k)))
    i8.clear()
    if "fp8" in groups:
        for name, (n, k) in synthetic.QWEN3_4B_SHAPES.items():
            q, s = capi.quantize_weight_per_channel_fp8(synthetic.weight(n, k, 1, device=dev))
            qs = [q] + [q.clone() for _ in range(_copies(n * k) - 1)]
            bias = synthetic.bias(n, 2, device=dev)
            for m in PREFILL_MS:
                x = synthetic.activations(m, k, 3, device=dev)
                y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
                us = _graph_us([lambda q=q: capi.w8a8_fp8_linear(x, q, s, bias=bias, y=y) for q in qs])
                qx, sx = capi.quantize_act_per_token_fp8(x)
                us_g = _graph_us([lambda q=q: capi.w8a8_fp8_gemm(qx, sx, q, s, bias=bias, y=y) for q in qs])
                f = 2 * m * n * k
                row("fp8", "w8a8_fp8_linear", name, m, n, k, us, flops=f, peak_scale=2.0,
                    gemm_us=round(us_g, 3), gemm_TOPS=round(f / us_g / 1e6, 1),
                    plan=list(capi.i8ql_fp8_plan(m, n, k)))
            del qs
    if "w4" in groups:
        for name, (n, k) in synthetic.QWEN3_8B_SHAPES.items():
            ws = [synthetic.weight(n, k, 4 + c, device=dev) for c in range(_copies(2 * n * k))]
            q4 = torch.empty((n, k // 2), dtype=torch.uint8, device=dev)
            s4 = torch.empty((n, k // 128), dtype=torch.bfloat16, device=dev)
            us = _graph_us([lambda w=w: capi.quantize_weight_w4_g128(w, q=q4, scale=s4) for w in ws])
            row("w4", "quantize_weight_w4_g128", name, 0, n, k, us, nbytes=bytes_quant_w4(n, k))
            del ws
            qs = [q4] + [q4.clone() for _ in range(_copies(n * k // 2) - 1)]
            for m in W4_MS:
                x = synthetic.activations(m, k, 5, device=dev)
                y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
                us = _graph_us([lambda q=q: capi.w4a16_gemm(x, q, s4, y=y) for q in qs])
                row("w4", "w4a16_gemm", name, m, n, k, us, nbytes=bytes_w4a16(m, n, k), flops=2 * m * n * k)
            del qs
    if "grouped" in groups or "moe" in groups:
        e_count = synthetic.DSMOE_ROUTED + synthetic.DSMOE_SHARED
        (inter2, hid), (_, inter) = synthetic.DSMOE_SHAPES["gate_up"], synthetic.DSMOE_SHAPES["down"]
        sets = {}
        for pname, (n, k) in synthetic.DSMOE_SHAPES.items():
            sets[pname] = []
            for c in range(3):  # three weight sets, each larger than L2
                q = torch.empty((e_count, n, k), dtype=torch.int8, device=dev)
                s = torch.empty((e_count, n), dtype=torch.float32, device=dev)
                for e in range(e_count):
                    capi.quantize_weight_per_channel_int8(synthetic.weight(n, k, 1000 + e, device=dev),
                                                          q=q[e], scale=s[e])
                sets[pname].append((q, s))
        for tokens in MOE_TOKENS:
            route = synthetic.moe_routing(tokens, seed=3)
            counts = np.diff(route.offsets)
            if "grouped" in groups:
                off = torch.from_numpy(route.offsets).to(dev)
                for pname, (n, k) in synthetic.DSMOE_SHAPES.items():
                    x = synthetic.activations(route.total_rows, k, 7, device=dev)
                    y = torch.empty((route.total_rows, n), dtype=torch.bfloat16, device=dev)
                    us = _graph_us([lambda q=q, s=s: capi.grouped_w8a16_gemm(x, off, q, s, y=y)
                                    for q, s in sets[pname]])
                    row("grouped", "grouped_w8a16_gemm", pname, tokens, n, k, us,
                        nbytes=bytes_grouped(counts, n, k), flops=2 * int(counts.sum()) * n * k,
                        rows=int(counts.sum()), experts_with_rows=int((counts > 0).sum()))
            if "moe" in groups:
                x = synthetic.activations(tokens, hid, 8, device=dev)
                lg = synthetic.gate_logits(tokens, synthetic.DSMOE_ROUTED, 3).to(dev)
                o = torch.empty((tokens, hid), dtype=torch.bfloat16, device=dev)
                us = _graph_us([lambda a=a, b=b: capi.moe_expert_mlp_w8a16(
                    x, lg, synthetic.DSMOE_TOPK, synthetic.DSMOE_SHARED, a[0], a[1], b[0], b[1], out=o)
                    for a, b in zip(sets["gate_up"], sets["down"])])
                rows = int(counts.sum())
                row("moe", "moe_expert_mlp_w8a16", "layer", tokens, hid, inter, us,
                    nbytes=bytes_moe(counts, tokens, hid, inter, synthetic.DSMOE_ROUTED),
                    flops=2 * rows * (inter2 * hid + hid * inter))
    if capi.i8ql_get_device_error() != capi.I8QL_OK:
        raise SystemExit("device error recorded during the shape table")
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["all", *ALL_PARTS], default="all")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of a CUDA graph")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--profile-timed", action="store_true",
                    help="bracket each part's timed region with cudaProfilerStart/Stop, so that "
                         "`ncu --profile-from-start off` lists exactly the timed launches")
    ap.add_argument("--cpu-row-frac", type=float, default=None,
                    help="row fraction of the cpu_baseline sample (default: 1/2 for decode, 1/8 for prefill)")
    ap.add_argument("--ref-row-frac", type=float, default=1 / 8)
    ap.add_argument("--single", default=None,
                    help="time one call: w8a8:M:N:K, linear:M:N:K, w8a16:M:N:K, quant:R:K, "
                         "w4a16:M:N:K, quant_w4:N:K, fp8:M:N:K (the FP8 linear layer), moe:T "
                         "(the DeepSeek-MoE expert MLP) or grouped:T:P (its grouped GEMM, P = 0 "
                         "gate_up, 1 down) (eager, for profiling)")
    ap.add_argument("--shapes", default=None,
                    help="per-shape table instead of the step: comma-separated groups out of "
                         + ",".join(SHAPE_GROUPS) + " (or all); CUDA-graph replays of back-to-back "
                         "calls over weight copies larger than L2, one JSON line per shape")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world, rank, local = dist_env()
    if args.single or args.shapes:
        from int8_quantized_linear_gb300 import build
        build.build()
        return run_single(args, local) if args.single else run_shapes(args, local)
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            dist.init_process_group("gloo")
        else:
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        from int8_quantized_linear_gb300 import build
        if rank == 0 or world == 1:
            build.build()
        barrier(world)
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
