"""Seeded synthetic inputs for the fused NVFP4 MoE layer.

This module only draws random numbers in the shapes and distributions of the
five layer workloads; it holds none of the layer's arithmetic (no
quantisation, routing, GEMM or combine). Both the CPU oracle (through the
tests) and the CUDA path (through the tests and the benchmark) take their
inputs from here, so they always see the same tensors.

Recipe (fixed draw order, everything on the CPU with ``torch.Generator``):

* router logits ``[T, E]`` fp32 ~ N(0, 1); for the skewed workload each
  expert ``e`` (rank ``r = e + 1``) adds ``3 * ln(r**-1.2 / sum_q q**-1.2)``;
* activations ``X [T, H]`` ~ N(0, 1) rounded to bf16; for the W4A4 workload
  each element is independently multiplied by 20 with probability 0.001;
* router weights ``W_router [E, H]`` ~ N(0, 1/H) rounded to bf16, so that
  ``x W_router^T`` has the N(0, 1) logits of the workloads;
* weights per expert ``e`` (routed ``0..E-1``, the shared expert is ``E``)
  and per matrix (gate ``[I, H]``, up ``[I, H]``, down ``[H, I]``) ~
  N(0, 0.02) rounded to bf16, each drawn from its own generator seeded from
  ``(seed, e, matrix)`` so that one expert can be regenerated alone.

Every tensor is returned on the CPU; callers move it where they need it.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import torch

__all__ = ["LayerConfig", "CONFIGS", "make_logits", "make_x", "make_router_weight",
           "make_expert_weight", "make_layer_weights", "weight_seed"]


@dataclass(frozen=True)
class LayerConfig:
    """Sizes of one MoE layer workload.

    T tokens, H hidden, I routed-expert intermediate, I_s shared-expert
    intermediate, E routed experts, k experts per token; ``mode`` is
    ``"w4a16"`` (weight-only NVFP4) or ``"w4a4"`` (NVFP4 weights and
    activations); ``logits`` is ``"normal"`` or ``"zipf"``; ``outliers``
    scales 0.1% of activations by 20.
    """
    name: str
    T: int
    H: int
    I: int
    I_s: int
    E: int
    k: int
    mode: str = "w4a16"
    logits: str = "normal"
    outliers: bool = False
    seed: int = 0

    def with_tokens(self, T: int) -> "LayerConfig":
        return LayerConfig(self.name + f"_T{T}", T, self.H, self.I, self.I_s, self.E,
                           self.k, self.mode, self.logits, self.outliers, self.seed)


#: The five workloads: a tiny case, decode, prefill, skewed routing and W4A4.
CONFIGS = {
    "tiny": LayerConfig("tiny", T=16, H=256, I=128, I_s=128, E=8, k=2),
    "decode": LayerConfig("decode", T=8, H=4096, I=1536, I_s=1536, E=320, k=8),
    "prefill": LayerConfig("prefill", T=4096, H=4096, I=1536, I_s=1536, E=320, k=8),
    "skewed": LayerConfig("skewed", T=2048, H=4096, I=1536, I_s=1536, E=320, k=8,
                          logits="zipf"),
    "w4a4": LayerConfig("w4a4", T=16384, H=7168, I=2048, I_s=2048, E=256, k=8,
                        mode="w4a4", outliers=True),
}

_MATRIX_INDEX = {"gate": 0, "up": 1, "down": 2}


def _gen(seed: int) -> torch.Generator:
    return torch.Generator(device="cpu").manual_seed(seed)


def weight_seed(seed: int, expert: int, matrix: str) -> int:
    """Seed of one weight matrix: distinct for every (seed, expert, matrix)."""
    return 1_000_003 * (seed + 1) + 4 * expert + _MATRIX_INDEX[matrix] + 17


def make_logits(cfg: LayerConfig) -> torch.Tensor:
    """Router logits ``[T, E]`` fp32."""
    g = _gen(cfg.seed * 7919 + 1)
    logits = torch.randn(cfg.T, cfg.E, generator=g, dtype=torch.float32)
    if cfg.logits == "zipf":
        s = 1.2
        z = sum(q ** -s for q in range(1, cfg.E + 1))
        bias = torch.tensor([3.0 * math.log((e + 1) ** -s / z) for e in range(cfg.E)],
                            dtype=torch.float32)
        logits = logits + bias[None, :]
    return logits.contiguous()


def make_x(cfg: LayerConfig, rows: slice | None = None) -> torch.Tensor:
    """Activations ``[T, H]`` bf16 (optionally only ``rows``, same values)."""
    g = _gen(cfg.seed * 7919 + 2)
    x = torch.randn(cfg.T, cfg.H, generator=g, dtype=torch.float32)
    if cfg.outliers:
        g2 = _gen(cfg.seed * 7919 + 3)
        mask = torch.rand(cfg.T, cfg.H, generator=g2) < 0.001
        x = torch.where(mask, x * 20.0, x)
    x = x.to(torch.bfloat16)
    if rows is not None:
        x = x[rows]
    return x.contiguous()


def make_router_weight(cfg: LayerConfig) -> torch.Tensor:
    """Router matrix ``[E, H]`` bf16, entries ~ N(0, 1/H)."""
    g = _gen(cfg.seed * 7919 + 4)
    w = torch.randn(cfg.E, cfg.H, generator=g, dtype=torch.float32) / math.sqrt(cfg.H)
    return w.to(torch.bfloat16).contiguous()


def make_expert_weight(cfg: LayerConfig, expert: int, matrix: str) -> torch.Tensor:
    """One weight matrix, bf16, N x K with K contiguous.

    gate/up are ``[I_e, H]``, down is ``[H, I_e]`` where ``I_e`` is ``I`` for a
    routed expert and ``I_s`` for the shared expert (``expert == E``).
    """
    inter = cfg.I_s if expert == cfg.E else cfg.I
    shape = (inter, cfg.H) if matrix in ("gate", "up") else (cfg.H, inter)
    g = _gen(weight_seed(cfg.seed, expert, matrix))
    w = torch.randn(*shape, generator=g, dtype=torch.float32) * 0.02
    return w.to(torch.bfloat16).contiguous()


def make_layer_weights(cfg: LayerConfig, experts=None, threads: int = 8):
    """Dict ``{expert: (gate, up, down)}`` of bf16 weights, drawn in parallel."""
    if experts is None:
        experts = list(range(cfg.E + 1))

    def one(e):
        return e, tuple(make_expert_weight(cfg, e, m) for m in ("gate", "up", "down"))

    with ThreadPoolExecutor(max(1, threads)) as ex:
        return dict(ex.map(one, experts))
