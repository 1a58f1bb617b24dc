"""Expert parallelism: the layer's experts split into contiguous shards, one
per rank ("Serving Solar Open 2 on DGX Spark", "Adding Expert Parallelism to
b12x": each node holds a contiguous shard of the experts, e.g. experts 0-159
on one node and 160-319 on the other; global expert ids are remapped to
shard-local ones and out-of-shard pairs are filtered out).

Every rank sees all tokens (the same x and router logits), routes them over
all E experts, computes only the pairs routed to its own experts (the shared
expert on rank 0) and produces a partial output; the layer's output is the
sum of the partial outputs over the ranks, one all-reduce. The filtering and
remapping run inside the CUDA library (``moe_layer_desc.expert_offset`` /
``local_experts``); this module holds the host side: which experts a rank
owns and the exchange of the partial outputs.
"""
from __future__ import annotations

import torch


def shard_range(E, world, rank):
    """Experts ``[lo, hi)`` of ``rank`` among ``world`` ranks: contiguous
    shards, the first ``E % world`` ranks one expert larger."""
    if not (0 <= rank < world) or E < 1:
        raise ValueError("need 0 <= rank < world and E >= 1")
    base, extra = divmod(E, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def combine_partials(partial, group=None):
    """Sum of every rank's partial output (bf16 ``[T, H]``): an all-reduce in
    fp32, rounded once to bf16. Returns a new bf16 tensor on the partial's
    device."""
    import torch.distributed as dist
    acc = partial.float()
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    return acc.to(torch.bfloat16)


class ExpertParallelLayer:
    """One rank's shard of an MoE layer: builds an ``Nvfp4MoeLayer`` holding
    experts ``shard_range(E, world, rank)`` (plus the shared expert on rank 0)
    and returns the full layer output (all ranks' partials summed)."""

    def __init__(self, T, H, I, E, k, world, rank, mode=None, I_shared=None, shared=True, device="cuda",
                 group=None):
        from . import binding as B
        from .layer import Nvfp4MoeLayer
        self.lo, self.hi = shard_range(E, world, rank)
        self.group = group
        self.layer = Nvfp4MoeLayer(T, H, I, E, k, mode=B.MOE_W4A16 if mode is None else mode, I_shared=I_shared,
                                   shared=shared and rank == 0, device=device, expert_offset=self.lo,
                                   local_experts=self.hi - self.lo)

    def owns(self, expert):
        return self.lo <= expert < self.hi or (expert == self.layer.E and self.layer.shared)

    def set_expert(self, expert, gate, up, down):
        if self.owns(expert):
            self.layer.set_expert(expert, gate, up, down)

    def forward(self, x, logits, topk_ids=None):
        partial = self.layer.forward(x, logits, topk_ids=topk_ids)
        return combine_partials(partial, self.group)
