"""Seeded synthetic inputs for the int8 quantized linear layer.

This module only draws inputs. It holds none of the quantization or GEMM
arithmetic, so both the CUDA path and the CPU oracle can be fed from it
without sharing any of the method's code.

Recipe (tensors drawn in fp32 from a seeded ``torch.Generator`` -- on the CPU
for parity cases, on the GPU for the large benchmark buffers -- then cast to
bf16 with round-to-nearest-even):

* Weights ``W [N, K] ~ N(0, 0.02)``; a seeded 0.1 % of the entries are
  multiplied by 30 (isolated outlier weights, the case "Day 6 -- Quantize It
  Yourself", mechanism block 1, question Q1 asks about).
* Activations ``X [M, K] ~ N(0, 1)``; a seeded 0.5 % of the input channels
  (the same channels for every token) are multiplied by 100: the emergent
  outlier feature dimensions of LLM.int8 that the same page describes in
  mechanism block 3.
* The tiny layer: ``W [512, 256]`` with row 7 all zero and one weight x50 in
  rows 100 (k=3) and 300 (k=200); ``X [16, 256]`` with channels 5 and 77
  x100.
* MoE routing for the grouped path (DeepSeek-MoE-16B shape: 64 routed
  experts, top-6, plus 2 shared experts that see every token): softmax over
  seeded N(0,1) gate logits, the six largest probabilities with ties broken
  by the lower expert index, token rows grouped by expert (routed experts
  0..63, then shared experts 64 and 65), and ``offsets`` the exclusive
  prefix sum of the per-expert row counts.  Routing is not part of the
  quantized layer; it only decides which rows each expert sees.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch

__all__ = [
    "QWEN3_4B_SHAPES",
    "QWEN3_4B_EXTRA_SHAPES",
    "QWEN3_8B_SHAPES",
    "DSMOE_SHAPES",
    "weight",
    "activations",
    "bias",
    "outlier_channels",
    "tiny_layer",
    "moe_routing",
    "gate_logits",
    "MoeRouting",
    "bf16_bits",
]

# Output x input shapes of the fused projections (PyTorch Linear layout).
QWEN3_4B_SHAPES = {
    "qkv": (6144, 2560),
    "o": (2560, 2560),
    "gate_up": (19456, 2560),
    "down": (2560, 9728),
}
# The o projection with the input width its attention implies (32 query
# heads x 128 = 4096), next to the stated [2560, 2560]: an extra parity case.
QWEN3_4B_EXTRA_SHAPES = {"o_heads": (2560, 4096)}
QWEN3_8B_SHAPES = {
    "qkv": (6144, 4096),
    "o": (4096, 4096),
    "gate_up": (24576, 4096),
    "down": (4096, 12288),
}
# One expert of DeepSeek-MoE-16B: fused gate/up and down projections.
DSMOE_SHAPES = {"gate_up": (2816, 2048), "down": (2048, 1408)}
DSMOE_ROUTED = 64
DSMOE_SHARED = 2
DSMOE_TOPK = 6

WEIGHT_STD = 0.02
WEIGHT_OUTLIER_FRAC = 1e-3
WEIGHT_OUTLIER_MULT = 30.0
ACT_OUTLIER_FRAC = 5e-3
ACT_OUTLIER_MULT = 100.0


def _gen(seed: int, device: str | torch.device = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def weight(n: int, k: int, seed: int, *, device: str | torch.device = "cpu",
           outlier_frac: float = WEIGHT_OUTLIER_FRAC,
           outlier_mult: float = WEIGHT_OUTLIER_MULT) -> torch.Tensor:
    """bf16 ``[n, k]`` weight ~ N(0, 0.02) with seeded isolated outliers."""
    g = _gen(seed, device)
    w = torch.randn((n, k), generator=g, device=device, dtype=torch.float32)
    w.mul_(WEIGHT_STD)
    n_out = int(round(outlier_frac * n * k))
    if n_out > 0:
        idx = torch.randint(0, n * k, (n_out,), generator=g, device=device)
        w.view(-1)[idx] *= outlier_mult
    return w.to(torch.bfloat16)


def outlier_channels(k: int, seed: int, frac: float = ACT_OUTLIER_FRAC) -> torch.Tensor:
    """The fixed set of outlier hidden dimensions for input width ``k``."""
    g = _gen(seed * 7919 + k)
    count = max(1, int(round(frac * k)))
    return torch.randperm(k, generator=g)[:count].sort().values


def activations(m: int, k: int, seed: int, *, device: str | torch.device = "cpu",
                channels: torch.Tensor | None = None,
                outlier_mult: float = ACT_OUTLIER_MULT) -> torch.Tensor:
    """bf16 ``[m, k]`` tokens ~ N(0, 1) with fixed outlier channels x100."""
    g = _gen(seed, device)
    x = torch.randn((m, k), generator=g, device=device, dtype=torch.float32)
    if channels is None:
        channels = outlier_channels(k, seed)
    if channels.numel() > 0 and m > 0:
        x[:, channels.to(device)] *= outlier_mult
    return x.to(torch.bfloat16)


def bias(n: int, seed: int, *, device: str | torch.device = "cpu") -> torch.Tensor:
    """bf16 ``[n]`` bias ~ N(0, 0.02)."""
    g = _gen(seed, device)
    return (torch.randn((n,), generator=g, device=device) * WEIGHT_STD).to(torch.bfloat16)


def tiny_layer(seed: int = 0):
    """The tiny linear layer: ``(W [512,256], X [16,256])`` in bf16."""
    g = _gen(seed)
    w = torch.randn((512, 256), generator=g) * WEIGHT_STD
    w[7, :] = 0.0
    w[100, 3] *= 50.0
    w[300, 200] *= 50.0
    x = torch.randn((16, 256), generator=g)
    x[:, 5] *= ACT_OUTLIER_MULT
    x[:, 77] *= ACT_OUTLIER_MULT
    return w.to(torch.bfloat16), x.to(torch.bfloat16)


@dataclasses.dataclass
class MoeRouting:
    """Token-to-expert assignment, grouped by expert.

    ``rows[i]`` is the token feeding grouped row ``i``; rows of expert ``e``
    are ``offsets[e] .. offsets[e+1]``; ``topk[t]`` lists token ``t``'s
    routed experts in decreasing probability.
    """

    tokens: int
    experts: int
    topk: np.ndarray        # int64 [T, 6]
    rows: np.ndarray        # int64 [T_total]
    offsets: np.ndarray     # int32 [E + 1]

    @property
    def total_rows(self) -> int:
        return int(self.offsets[-1])


def gate_logits(tokens: int, routed: int, seed: int) -> torch.Tensor:
    """fp32 ``[tokens, routed]`` gate logits ~ N(0, 1), seeded."""
    g = _gen(seed)
    return torch.randn((tokens, routed), generator=g, dtype=torch.float32)


def moe_routing(tokens: int, seed: int, routed: int = DSMOE_ROUTED,
                shared: int = DSMOE_SHARED, topk: int = DSMOE_TOPK) -> MoeRouting:
    """Seeded top-k routing plus shared experts, rows grouped by expert: the
    input recipe of the grouped GEMM's benchmark and parity cases (numpy;
    the oracle's routing of the MoE layer is written independently)."""
    logits = gate_logits(tokens, routed, seed).double().numpy()
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    # Stable sort on -p: among equal probabilities the lower index comes first.
    order = np.argsort(-p, axis=1, kind="stable")[:, :topk].astype(np.int64)
    experts = routed + shared
    members: list[list[int]] = [[] for _ in range(experts)]
    for t in range(tokens):
        for e in order[t]:
            members[int(e)].append(t)
    for s in range(shared):
        members[routed + s] = list(range(tokens))
    counts = np.array([len(mm) for mm in members], dtype=np.int64)
    offsets = np.zeros(experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    rows = np.array([t for mm in members for t in mm], dtype=np.int64)
    return MoeRouting(tokens=tokens, experts=experts, topk=order, rows=rows, offsets=offsets)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a bf16 tensor as a uint16 numpy array."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
