"""Device-side setup of one MoE layer through the C ABI.

``Nvfp4MoeLayer`` quantises bf16 weight matrices to NVFP4 with the
library's own quantiser (``moe_nvfp4_quantize``; MXFP4 layers with
``moe_mxfp4_quantize``) or takes pre-quantised
checkpoint matrices (``import_expert``: the stored global scale is converted
with ``moe_import_global_scale``), converts them into the kernels' tile
layout (``moe_nvfp4_prepare_weights``), keeps them resident in device memory
and runs the fused forward (``moe_nvfp4_forward``), optionally with its own
router GEMM (``set_router``) and static W4A4 activation scales
(``set_static_scales``). torch is used only to allocate device memory; every
step of the layer runs in the CUDA library.
"""
from __future__ import annotations

import torch

from . import binding as B


def _empty_bytes(n, device):
    # 256-byte aligned (the caching allocator aligns to 512)
    return torch.empty(max(int(n), 1), dtype=torch.uint8, device=device)


def quantize_bf16(x, device="cuda"):
    """bf16 ``[rows, K]`` on the device -> (packed codes, E4M3 scales, gs tensor)."""
    rows, K = x.shape
    q = torch.empty(rows, K // 2, dtype=torch.uint8, device=device)
    sf = torch.empty(rows, K // 16, dtype=torch.uint8, device=device)
    gs = torch.empty(1, dtype=torch.float32, device=device)
    ws = _empty_bytes(B.moe_quantize_workspace_size(), device)
    B.moe_nvfp4_quantize(x, rows, K, q, sf, gs, ws)
    return q, sf, gs


def quantize_mx(x, device="cuda"):
    """bf16 ``[rows, K]`` on the device -> MXFP4 (packed codes, E8M0 scales)."""
    rows, K = x.shape
    q = torch.empty(rows, K // 2, dtype=torch.uint8, device=device)
    sf = torch.empty(rows, K // 32, dtype=torch.uint8, device=device)
    B.moe_mxfp4_quantize(x, rows, K, q, sf)
    return q, sf


class Nvfp4MoeLayer:
    """NVFP4 weights of E routed experts (+ optional shared expert) on one GPU."""

    def __init__(self, T, H, I, E, k, mode=B.MOE_W4A16, I_shared=None, shared=True, device="cuda",
                 expert_offset=0, local_experts=None):
        """``expert_offset`` / ``local_experts``: expert parallelism, this layer
        holds (and computes) only the experts ``[expert_offset, expert_offset +
        local_experts)`` of the E the router ranks; its output is then the
        shard's partial output (see ``ep``)."""
        self.T, self.H, self.I, self.E, self.k = T, H, I, E, k
        self.I_shared = I if I_shared is None else I_shared
        self.mode = mode
        self.shared = shared
        self.device = device
        self.expert_offset = expert_offset
        self.local_experts = E if local_experts is None else local_experts
        if not (0 <= expert_offset and expert_offset + self.local_experts <= E):
            raise ValueError("expert shard outside [0, E)")
        self.s13 = B.moe_prepare_size(2 * I, H, mode, 1)
        self.s2 = B.moe_prepare_size(H, I, mode, 0)
        self.w13 = _empty_bytes(self.local_experts * self.s13, device)
        self.w2 = _empty_bytes(self.local_experts * self.s2, device)
        if shared:
            self.w13_s = _empty_bytes(B.moe_prepare_size(2 * self.I_shared, H, mode, 1), device)
            self.w2_s = _empty_bytes(B.moe_prepare_size(H, self.I_shared, mode, 0), device)
        else:
            self.w13_s = self.w2_s = None
        self.gs = {}  # (expert, matrix) -> quant-convention global scale (float)
        self.w_router = None
        self.x_gs = self.h_gs = 0.0

    def _slot(self, expert, which):
        if expert == self.E:
            return self.w13_s if which == 13 else self.w2_s
        e = expert - self.expert_offset  # this shard's block of the (global) expert
        if not 0 <= e < self.local_experts:
            raise ValueError(f"expert {expert} is not in this layer's shard")
        if which == 13:
            return self.w13[e * self.s13:(e + 1) * self.s13]
        return self.w2[e * self.s2:(e + 1) * self.s2]

    def set_expert(self, expert, gate, up, down):
        """bf16 gate ``[I, H]``, up ``[I, H]``, down ``[H, I]`` (any device); expert E = shared."""
        dev = self.device
        gate, up, down = (t.to(dev, torch.bfloat16).contiguous() for t in (gate, up, down))
        if self.mode == B.MOE_MXFP4:  # E8M0 scales per 32, no global scale
            (qg, sg), (qu, su), (qd, sd) = (quantize_mx(m, dev) for m in (gate, up, down))
            inter = gate.shape[0]
            B.moe_nvfp4_prepare_weights(torch.cat([qg, qu]), torch.cat([sg, su]), None, 2 * inter, self.H,
                                        self.mode, 1, self._slot(expert, 13))
            B.moe_nvfp4_prepare_weights(qd, sd, None, self.H, inter, self.mode, 0, self._slot(expert, 2))
            return (qg, sg), (qu, su), (qd, sd)
        qg, sg, gg = quantize_bf16(gate, dev)
        qu, su, gu = quantize_bf16(up, dev)
        qd, sd, gd = quantize_bf16(down, dev)
        gsv = torch.cat([gg, gu, gd]).cpu().tolist()
        self.gs[(expert, "gate")], self.gs[(expert, "up")], self.gs[(expert, "down")] = gsv
        inter = gate.shape[0]
        codes13 = torch.cat([qg, qu])
        sf13 = torch.cat([sg, su])
        B.moe_nvfp4_prepare_weights(codes13, sf13, gsv[:2], 2 * inter, self.H, self.mode, 1,
                                    self._slot(expert, 13))
        B.moe_nvfp4_prepare_weights(qd, sd, gsv[2:], self.H, inter, self.mode, 0, self._slot(expert, 2))
        return (qg, sg, gsv[0]), (qu, su, gsv[1]), (qd, sd, gsv[2])

    def import_expert(self, expert, gate, up, down, fmt):
        """Pre-quantised checkpoint matrices of one expert (expert E = shared).

        ``gate``, ``up`` (``[I, H]``) and ``down`` (``[H, I]``) are each a
        triple (packed codes uint8 ``[N, K/2]``, E4M3 scales uint8
        ``[N, K/16]``, stored global scale) with the scale stored in ``fmt``
        (``MOE_SCALE_QUANT``: compressed-tensors; ``MOE_SCALE_DEQUANT``:
        ModelOpt). Returns the three quant-convention global scales.
        """
        dev = self.device
        gs = [B.moe_import_global_scale(m[2], fmt) for m in (gate, up, down)]
        (qg, sg, _), (qu, su, _), (qd, sd, _) = (
            (m[0].to(dev).contiguous(), m[1].to(dev).contiguous(), m[2]) for m in (gate, up, down))
        self.gs[(expert, "gate")], self.gs[(expert, "up")], self.gs[(expert, "down")] = gs
        inter = qg.shape[0]
        B.moe_nvfp4_prepare_weights(torch.cat([qg, qu]), torch.cat([sg, su]), gs[:2], 2 * inter, self.H,
                                    self.mode, 1, self._slot(expert, 13))
        B.moe_nvfp4_prepare_weights(qd, sd, gs[2:], self.H, inter, self.mode, 0, self._slot(expert, 2))
        return gs

    def set_router(self, w_router):
        """bf16 router matrix ``[E, H]``; the forward then computes its own logits."""
        self.w_router = None if w_router is None else w_router.to(self.device, torch.bfloat16).contiguous()

    def set_static_scales(self, x_gs=0.0, h_gs=0.0):
        """W4A4 static global scales (quant convention) for x and h; 0 = dynamic."""
        self.x_gs, self.h_gs = float(x_gs), float(h_gs)

    def desc(self, T=None):
        d = B.MoeLayerDesc()
        d.T = self.T if T is None else T
        d.H, d.I, d.I_shared, d.E, d.k = self.H, self.I, self.I_shared, self.E, self.k
        d.mode = self.mode
        d.w13, d.w2 = self.w13.data_ptr(), self.w2.data_ptr()
        d.w13_shared = self.w13_s.data_ptr() if self.shared else None
        d.w2_shared = self.w2_s.data_ptr() if self.shared else None
        d.w_router = None if self.w_router is None else self.w_router.data_ptr()
        d.x_global_scale, d.h_global_scale = self.x_gs, self.h_gs
        sharded = self.local_experts != self.E
        d.expert_offset = self.expert_offset if sharded else 0
        d.local_experts = self.local_experts if sharded else 0
        return d

    def workspace(self, T=None):
        # the first 256 bytes hold the device status word and must start at zero
        ws = _empty_bytes(B.moe_workspace_size(self.desc(T)), self.device)
        ws[:256].zero_()
        return ws

    def forward(self, x, logits=None, out=None, topk_ids=None, ws=None, stream=None):
        """``logits`` may be None when a router matrix is set."""
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, device=self.device)
        if ws is None:
            ws = self.workspace(T)
        B.moe_nvfp4_forward(self.desc(T), x, logits, out, topk_ids, ws, stream)
        return out
