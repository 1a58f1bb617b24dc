"""Degenerate shapes of the fused forward against the oracle: no shared
expert, a single token, a single expert with top-1, and k = E."""
import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import moe as omoe
from tests.gpu_layers import OracleWeights
from tests.tolerance import check_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _layer(cfg, shared):
    from nvfp4_mixture_experts_moe_gb300 import Nvfp4MoeLayer
    layer = Nvfp4MoeLayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, I_shared=cfg.I_s, shared=shared, device="cuda")
    experts = list(range(cfg.E + (1 if shared else 0)))
    W = si.make_layer_weights(cfg, experts=experts, threads=8)
    for e in experts:
        layer.set_expert(e, *W[e])
    torch.cuda.synchronize()
    return layer


def _check(cfg, shared):
    from nvfp4_mixture_experts_moe_gb300 import binding
    layer = _layer(cfg, shared)
    x = si.make_x(cfg)
    logits = si.make_logits(cfg)
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
    ws = layer.workspace()
    out = layer.forward(x.cuda(), logits.cuda(), topk_ids=ids, ws=ws)
    torch.cuda.synchronize()
    assert binding.moe_get_device_status(ws) == 0
    ow = OracleWeights(cfg)
    experts = [ow(e) for e in range(cfg.E)]
    ref, parts = omoe.layer(x.float().numpy(), logits.numpy(), experts, ow(cfg.E) if shared else None, cfg.k,
                            return_parts=True)
    assert (ids.cpu().numpy() == parts["ids"]).all()
    check_outputs(out.float().cpu().numpy(), ref, what=cfg.name)


@pytest.mark.parametrize("T", [5, 300])
def test_forward_without_shared_expert(T):
    _check(si.LayerConfig(f"noshared{T}", T=T, H=256, I=128, I_s=128, E=8, k=2), shared=False)


def test_forward_single_token():
    _check(si.LayerConfig("one_token", T=1, H=256, I=128, I_s=128, E=8, k=2), shared=True)


def test_forward_one_expert_top1():
    _check(si.LayerConfig("one_expert", T=40, H=256, I=128, I_s=128, E=1, k=1), shared=True)


def test_forward_k_equals_e():
    _check(si.LayerConfig("k_eq_e", T=24, H=256, I=128, I_s=128, E=4, k=4), shared=True)
