"""Failure detection without a GPU fault: with the test hook's wait limit at
one clock cycle every bounded wait inside the GEMM kernels gives up at once.
Each kernel must then record MOE_ERR_TIMEOUT in the workspace status word,
let its copies and tensor-core work drain, free its tensor memory and return,
so that the next forward on the same stream and workspace (default limit)
gives exactly the result of a forward that never timed out."""
import pytest
import torch

import synthetic_inputs as si
from tests.gpu_layers import device_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def B():
    from nvfp4_mixture_experts_moe_gb300 import binding
    return binding


@pytest.fixture(autouse=True)
def default_hooks():
    yield
    for key in (B().MOE_DEBUG_WAIT_LIMIT, B().MOE_DEBUG_EXTRA_ARRIVALS, B().MOE_DEBUG_DISABLE_DECODE_FUSED,
                B().MOE_DEBUG_FP4_TILE):
        B().moe_debug_set(key, 0)


W4A4_SMALL = si.LayerConfig("to_w4a4", T=300, H=512, I=256, I_s=256, E=8, k=2, mode="w4a4")


@pytest.mark.parametrize("cfg,chain,fp4_tile", [
    (W4A4_SMALL, False, 0),                                                                        # 128 x 256 tiles
    (W4A4_SMALL, False, 33),                                                                       # 128 x 128, two CTAs per SM
    (W4A4_SMALL, False, 11),                                                                       # 128 x 128, one CTA per SM
    (si.LayerConfig("to_mx", T=300, H=512, I=256, I_s=256, E=8, k=2, mode="mxfp4"), False, 0),     # kind::mxf4
    (si.LayerConfig("to_w4a16", T=300, H=512, I=256, I_s=256, E=4, k=2), False, 0),                # gemm_tc_f16
    (si.LayerConfig("to_dec", T=8, H=512, I=256, I_s=256, E=16, k=4), True, 0),                    # gemm_small
], ids=["w4a4_tcgen05", "w4a4_tile128_2cta", "w4a4_tile128_1cta", "mxfp4_tcgen05", "w4a16_tcgen05",
        "decode_chain"])
def test_timeout_is_reported_and_the_next_forward_is_exact(cfg, chain, fp4_tile):
    cfg, layer = device_layer(cfg)
    x = si.make_x(cfg).cuda()
    lg = si.make_logits(cfg).cuda()
    B().moe_debug_set(B().MOE_DEBUG_FP4_TILE, fp4_tile)
    if chain:
        B().moe_debug_set(B().MOE_DEBUG_DISABLE_DECODE_FUSED, 1)
    ws = layer.workspace()
    good = layer.forward(x, lg, ws=ws).clone()
    torch.cuda.synchronize()
    assert B().moe_get_device_status(ws) == 0
    B().moe_debug_set(B().MOE_DEBUG_WAIT_LIMIT, 1)
    layer.forward(x, lg, ws=ws)
    torch.cuda.synchronize()
    assert B().moe_get_device_status(ws) == B().MOE_ERR_TIMEOUT
    B().moe_debug_set(B().MOE_DEBUG_WAIT_LIMIT, 0)
    again = layer.forward(x, lg, ws=ws)
    torch.cuda.synchronize()
    assert B().moe_get_device_status(ws) == 0
    assert torch.equal(good, again)
