"""MXFP4 ("vLLM on the NVIDIA DGX Spark", section 6.4 "NVFP4 vs MXFP4": e2m1
elements, one E8M0 power-of-two scale per 32 along K, no global scale)
through the C ABI against the CPU oracle: the quantiser bit for bit, and
whole MXFP4 layers (block-scaled FP4 MMA with UE8M0 scales, kind::mxf4)
within the output bars."""
import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import moe as omoe
from oracle import mxfp4 as omx
from oracle import nvfp4 as onv
from tests.gpu_layers import OracleWeights, device_layer
from tests.tolerance import check_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _quant_gpu(x_bf16):
    from nvfp4_mixture_experts_moe_gb300 import quantize_mx
    q, sf = quantize_mx(x_bf16.cuda())
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy()


@pytest.mark.parametrize("rows,K,scale,outliers", [(16, 256, 1.0, False), (64, 4096, 0.02, False),
                                                   (257, 7168, 1.0, True), (3, 32, 1e-3, False),
                                                   (8, 64, 1e-38, False), (4, 96, 1e37, False)])
def test_mxfp4_quantize_bit_exact(rows, K, scale, outliers):
    g = torch.Generator().manual_seed(rows * K + 5)
    x = torch.randn(rows, K, generator=g) * scale
    if outliers:
        m = torch.rand(rows, K, generator=g) < 0.001
        x = torch.where(m, x * 20, x)
    x = x.to(torch.bfloat16)
    x[0, :32] = 0.0                       # an all-zero block
    if rows > 1:
        x[1, :32] = -0.0                  # all negative zeros: codes 0, smallest scale
        if K > 40:
            x[1, 40] = -0.0               # a -0 inside a non-zero block keeps its sign
    q, sf = _quant_gpu(x)
    rq, rsf = omx.quantize(x.float().numpy())
    assert (sf == rsf).all()
    assert (q == onv.pack(rq)).all()


def test_mxfp4_quantize_ties():
    # values on e2m1 midpoints at a block scale of 1 (block amax 6 -> e = 0)
    vals = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 4
    x = torch.tensor([vals, [-v for v in vals]], dtype=torch.float32).to(torch.bfloat16)
    q, sf = _quant_gpu(x)
    rq, rsf = omx.quantize(x.float().numpy())
    assert (sf == rsf).all() and (q == onv.pack(rq)).all()
    assert (rsf == 127).all()  # the page's format at scale 1: codes are the plain e2m1 roundings


def _run(cfg):
    cfg, layer = device_layer(cfg)
    x = si.make_x(cfg)
    logits = si.make_logits(cfg)
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
    ws = layer.workspace()
    out = layer.forward(x.cuda(), logits.cuda(), topk_ids=ids, ws=ws)
    torch.cuda.synchronize()
    from nvfp4_mixture_experts_moe_gb300 import binding
    assert binding.moe_get_device_status(ws) == 0
    return cfg, layer, x, logits, out.float().cpu().numpy(), ids.cpu().numpy()


SMALL = si.LayerConfig("mx_small", T=64, H=512, I=256, I_s=256, E=8, k=2, mode="mxfp4", outliers=True)
GROUPS = si.LayerConfig("mx_groups", T=300, H=512, I=256, I_s=256, E=24, k=4, mode="mxfp4", logits="zipf")


@pytest.mark.parametrize("cfg", [SMALL, GROUPS], ids=["small", "skewed_groups"])
def test_mxfp4_layer_full_check(cfg):
    cfg, layer, x, logits, out, ids = _run(cfg)
    if cfg is GROUPS or cfg.name == "mx_groups":
        counts = np.bincount(ids.ravel(), minlength=cfg.E)
        assert (counts == 0).any() and counts.max() > 128   # empty groups and multi-tile groups
    experts, shared = OracleWeights(cfg).all()
    ref, parts = omoe.layer(x.float().numpy(), logits.numpy(), experts, shared, cfg.k, mode="mxfp4",
                            return_parts=True)
    assert (ids == parts["ids"]).all()
    check_outputs(out, ref, what=f"mxfp4 {cfg.name}")


def test_mxfp4_layer_is_deterministic_and_not_nvfp4():
    cfg, layer = device_layer(SMALL)
    x = si.make_x(cfg).cuda()
    lg = si.make_logits(cfg).cuda()
    o = [layer.forward(x, lg).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(o[0], t) for t in o[1:])


def test_mxfp4_prepare_refuses_nan_scale_codes():
    from nvfp4_mixture_experts_moe_gb300 import binding as B
    N, K = 128, 256
    codes = torch.zeros(N, K // 2, dtype=torch.uint8, device="cuda")
    sf = torch.full((N, K // 32), 127, dtype=torch.uint8, device="cuda")
    out = torch.empty(B.moe_prepare_size(N, K, B.MOE_MXFP4, 0), dtype=torch.uint8, device="cuda")
    B.moe_nvfp4_prepare_weights(codes, sf, None, N, K, B.MOE_MXFP4, 0, out)
    sf[5, 3] = 0xFF
    with pytest.raises(B.MoeError) as ei:
        B.moe_nvfp4_prepare_weights(codes, sf, None, N, K, B.MOE_MXFP4, 0, out)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG
