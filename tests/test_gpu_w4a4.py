"""W4A4 path (NVFP4 weights and activations, block-scaled FP4 MMA on tcgen05)
against the CPU oracle through the C ABI."""
import os

import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import moe as omoe
from oracle import nvfp4 as onv
from tests.gpu_layers import OracleWeights, device_layer
from tests.tolerance import TOPK_W_ABS, check_outputs

pytestmark = pytest.mark.gpu

SMALL = si.LayerConfig("w4a4_small", T=64, H=512, I=256, I_s=256, E=8, k=2, mode="w4a4", outliers=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


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


def test_w4a4_small_layer_full_check():
    cfg, layer, x, logits, out, ids = _run(SMALL)
    ow = OracleWeights(cfg)
    experts, shared = ow.all()
    ref, parts = omoe.layer(x.float().numpy(), logits.numpy(), experts, shared, cfg.k, mode="w4a4",
                            return_parts=True)
    assert (ids == parts["ids"]).all()
    check_outputs(out, ref, what="w4a4 small")


# skewed routing at a small size: empty groups, groups of several 128-row
# tiles and ragged last tiles through the fused forward's per-tile operand assembly and
# its block-scaled GEMMs
GROUPS = si.LayerConfig("w4a4_groups", T=300, H=512, I=256, I_s=256, E=24, k=4, mode="w4a4", logits="zipf")


def test_w4a4_skewed_groups_full_check():
    cfg, layer, x, logits, out, ids = _run(GROUPS)
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    assert (counts == 0).any() and counts.max() > 128  # the cases this test is for
    ow = OracleWeights(cfg)
    experts, shared = ow.all()
    ref, parts = omoe.layer(x.float().numpy(), logits.numpy(), experts, shared, cfg.k, mode="w4a4",
                            return_parts=True)
    assert (ids == parts["ids"]).all()
    check_outputs(out, ref, what="w4a4 skewed groups")


MX_GROUPS = si.LayerConfig("mx_groups", T=300, H=512, I=256, I_s=256, E=24, k=4, mode="mxfp4", logits="zipf")


@pytest.mark.parametrize("cfg", [GROUPS, MX_GROUPS], ids=["nvfp4", "mxfp4"])
def test_fp4_tile_shapes_agree(cfg):
    """Every tile shape of the block-scaled FP4 GEMMs (one or two CTAs per SM;
    weight rows or the group's rows on the MMA's M side; 128 or 256 weight
    rows per tile, the latter as two N = 128 MMAs or one N = 256) gives the library
    default's bits, on skewed routing with empty groups, groups of several
    128-row tiles and ragged last tiles (the default is checked against the
    oracle above)."""
    from nvfp4_mixture_experts_moe_gb300 import binding as Bd
    cfg, layer = device_layer(cfg)
    x = si.make_x(cfg).cuda()
    lg = si.make_logits(cfg).cuda()
    ws = layer.workspace()
    outs = {}
    try:
        for shape in (0, 11, 12, 13, 14, 15, 21, 22, 23, 24, 25, 31, 32, 33, 34, 35, 41, 42, 43, 44, 45, 51, 52,
                      53, 54, 55):
            Bd.moe_debug_set(Bd.MOE_DEBUG_FP4_TILE, shape)
            outs[shape] = layer.forward(x, lg, ws=ws).clone()
            torch.cuda.synchronize()
            assert Bd.moe_get_device_status(ws) == 0, shape
    finally:
        Bd.moe_debug_set(Bd.MOE_DEBUG_FP4_TILE, 0)
    differ = [shape for shape, o in outs.items() if not torch.equal(o, outs[0])]
    assert not differ, f"tile shapes {differ} differ from the default"


def test_w4a4_small_deterministic():
    cfg, layer = device_layer(SMALL)
    x = si.make_x(cfg).cuda()
    lg = si.make_logits(cfg).cuda()
    o = [layer.forward(x, lg).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(o[0], t) for t in o[1:])


def _fp4_groups(G, N, K, gate_up, seed):
    from nvfp4_mixture_experts_moe_gb300 import binding as Bd, quantize_bf16
    g = torch.Generator().manual_seed(seed)
    size = Bd.moe_prepare_size(N, K, 1, gate_up)
    buf = torch.empty(G * size, dtype=torch.uint8, device="cuda")
    ow = []
    for i in range(G):
        shapes = [(N // 2, K)] * 2 if gate_up else [(N, K)]
        mats = [(torch.randn(*sh, generator=g) * 0.02).to(torch.bfloat16) for sh in shapes]
        qs = [quantize_bf16(m.cuda()) for m in mats]
        Bd.moe_nvfp4_prepare_weights(torch.cat([q[0] for q in qs]), torch.cat([q[1] for q in qs]),
                                     [q[2].item() for q in qs], N, K, 1, gate_up,
                                     buf[i * size:(i + 1) * size])
        ow.append([omoe.QuantWeight.from_dense(m.float().numpy()) for m in mats])
    return buf, ow


@pytest.mark.parametrize("path", ["gather", "tiles", "tiles_in_place"])
@pytest.mark.parametrize("gate_up", [1, 0])
def test_w4a4_grouped_gemm_tile_edges(gate_up, path):
    """The public W4A4 grouped GEMM against the oracle on empty, small,
    ragged and multi-tile groups: without the row count (the kernel that
    gathers rows inside the GEMM), and with it (the forward's tile kernels),
    the codes gathered through the row index or read in place in group order."""
    from nvfp4_mixture_experts_moe_gb300 import binding as Bd, quantize_bf16
    rows = [0, 40, 300, 7, 129, 128, 1]
    G = len(rows)
    N, K = (256, 512) if gate_up else (384, 256)
    buf, ow = _fp4_groups(G, N, K, gate_up, seed=21 + gate_up)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    total = int(off[-1])
    g = torch.Generator().manual_seed(9)
    src = total + 5
    a = torch.randn(src, K, generator=g).to(torch.bfloat16)
    aq, asf, ags = quantize_bf16(a.cuda())
    idx = torch.randperm(src, generator=g)[:total].to(torch.int32)
    rs = torch.rand(total, generator=g) + 0.5
    out = torch.full((total, N // 2 if gate_up else N), float("nan"), dtype=torch.bfloat16, device="cuda")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    offs_d, idx_d, rs_d = torch.from_numpy(off).cuda(), idx.cuda(), rs.cuda()
    args = Bd.MoeGemmArgs(mode=1, gate_up=gate_up, num_groups=G, N=N, K=K)
    args.weights = buf.data_ptr()
    args.group_offsets = offs_d.data_ptr()
    args.a, args.a_sf, args.a_gs = aq.data_ptr(), asf.data_ptr(), ags.data_ptr()
    args.a_row_index = idx_d.data_ptr()
    if path == "tiles_in_place":   # the rows already in group order, no row index
        aq_g, asf_g = aq[idx_d.long()].contiguous(), asf[idx_d.long()].contiguous()
        args.a, args.a_sf, args.a_row_index = aq_g.data_ptr(), asf_g.data_ptr(), None
    args.row_scale = None if gate_up else rs_d.data_ptr()
    args.out = out.data_ptr()
    args.out_amax = amax.data_ptr() if gate_up else None
    if path == "gather":
        ws = torch.zeros(Bd.moe_gemm_workspace_size(G), dtype=torch.uint8, device="cuda")
    else:
        args.rows = total
        ws = torch.zeros(Bd.moe_gemm_workspace_size_rows(G, total, K), dtype=torch.uint8, device="cuda")
    Bd.moe_nvfp4_grouped_gemm(args, ws)
    assert Bd.moe_get_device_status(ws) == 0
    got = out.float().cpu().numpy()
    q, sf, gs = onv.quantize(a.float().numpy())
    assert gs == np.float32(ags.item())
    xa = onv.dequantize(q, sf, gs)[idx.numpy()]
    for gi in range(G):
        r0, r1 = off[gi], off[gi + 1]
        if r1 == r0:
            continue
        if gate_up:
            ref = omoe.gate_up_swiglu(xa[r0:r1], ow[gi][0], ow[gi][1])
        else:
            ref = omoe.down_proj(xa[r0:r1], ow[gi][0]) * rs.numpy()[r0:r1, None]
        check_outputs(got[r0:r1], ref, what=f"group {gi} ({r1 - r0} rows)")
    if gate_up:
        assert amax.item() == float(np.abs(got).max())


def test_w4a4_grouped_gemm_row_count_checked():
    """The public W4A4 grouped GEMM's row count: a larger one than the groups
    hold gives the exact count's bits; a smaller one makes the GEMM record
    MOE_ERR_DEVICE and compute nothing (the code gather stays within the
    workspace)."""
    from nvfp4_mixture_experts_moe_gb300 import binding as Bd, quantize_bf16
    rows = [40, 300, 7, 129]
    G, N, K = len(rows), 256, 512
    buf, _ = _fp4_groups(G, N, K, 1, seed=33)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    total = int(off[-1])
    g = torch.Generator().manual_seed(8)
    a = torch.randn(total + 5, K, generator=g).to(torch.bfloat16)
    aq, asf, ags = quantize_bf16(a.cuda())
    idx = torch.randperm(total + 5, generator=g)[:total].to(torch.int32).cuda()
    offs = torch.from_numpy(off).cuda()

    def run(count):
        out = torch.full((total, N // 2), float("nan"), dtype=torch.bfloat16, device="cuda")
        args = Bd.MoeGemmArgs(mode=1, gate_up=1, num_groups=G, N=N, K=K, rows=count)
        args.weights, args.group_offsets = buf.data_ptr(), offs.data_ptr()
        args.a, args.a_sf, args.a_gs = aq.data_ptr(), asf.data_ptr(), ags.data_ptr()
        args.a_row_index, args.out = idx.data_ptr(), out.data_ptr()
        ws = torch.zeros(Bd.moe_gemm_workspace_size_rows(G, count, K), dtype=torch.uint8, device="cuda")
        Bd.moe_nvfp4_grouped_gemm(args, ws)
        return out, Bd.moe_get_device_status(ws)

    exact, st = run(total)
    assert st == 0
    more, st = run(total + 37)
    assert st == 0 and torch.equal(more, exact)
    _, st = run(total - 1)
    assert st == Bd.MOE_ERR_DEVICE


def test_w4a4_grouped_gemm_many_groups_fall_back():
    """600 groups with N = 384 (not a multiple of 256): the tile kernel's
    shape for that N cannot hold the groups in shared memory, so a call with
    the row count runs the gather kernel, with its exact bits."""
    from nvfp4_mixture_experts_moe_gb300 import binding as Bd, quantize_bf16
    G, N, K = 600, 384, 256
    size = Bd.moe_prepare_size(N, K, 1, 0)
    g = torch.Generator().manual_seed(12)
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    wq, wsf, wgs = quantize_bf16(w.cuda())
    buf = torch.empty(G * size, dtype=torch.uint8, device="cuda")
    Bd.moe_nvfp4_prepare_weights(wq, wsf, [wgs.item()], N, K, 1, 0, buf[:size])
    buf.view(G, size)[1:] = buf[:size]   # every group the same prepared block
    rows = torch.randint(0, 3, (G,), generator=g).tolist()
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    total = int(off[-1])
    a = torch.randn(total, K, generator=g).to(torch.bfloat16)
    aq, asf, ags = quantize_bf16(a.cuda())
    rs = (torch.rand(total, generator=g) + 0.5).cuda()
    offs = torch.from_numpy(off).cuda()

    def run(count):
        out = torch.full((total, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        args = Bd.MoeGemmArgs(mode=1, gate_up=0, num_groups=G, N=N, K=K, rows=count)
        args.weights, args.group_offsets = buf.data_ptr(), offs.data_ptr()
        args.a, args.a_sf, args.a_gs = aq.data_ptr(), asf.data_ptr(), ags.data_ptr()
        args.row_scale, args.out = rs.data_ptr(), out.data_ptr()
        n = Bd.moe_gemm_workspace_size_rows(G, count, K) if count else Bd.moe_gemm_workspace_size(G)
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
        Bd.moe_nvfp4_grouped_gemm(args, ws)
        assert Bd.moe_get_device_status(ws) == 0
        return out

    ref = run(0)
    assert not torch.isnan(ref.float()).any()
    assert torch.equal(run(total), ref)


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "w4a4_full_tokens.npz")


@pytest.mark.slow
def test_w4a4_full_size_against_golden():
    """The W4A4 workload at full size (16384 tokens, hidden 7168, 256 experts
    top-8 + shared): routing exact; X quantisation bit-exact over the whole
    tensor with the oracle's global scale; and 64 tokens spread over the batch
    element by element against the oracle's outputs at the stated bars plus
    the oracle's allowance for FP4 re-quantisation of h. The global scale of
    h depends on all 147,456 rows, so those outputs were computed once by the
    oracle alone (tests/golden/make_w4a4_full.py) and stored with the scales
    and the allowance."""
    ref = np.load(GOLDEN)
    cfg, layer, x, logits, out, ids = _run("w4a4")
    rids, rw = omoe.route(logits.numpy(), cfg.k)
    assert (ids == rids).all()
    toks = ref["tokens"]
    # the stored routing was computed on another machine: ids bit for bit, weights
    # within the routing-weight bar (numpy's exp may differ in the last place)
    assert (rids[toks] == ref["ids"]).all() and np.abs(rw[toks] - ref["w"]).max() <= TOPK_W_ABS
    from nvfp4_mixture_experts_moe_gb300 import quantize_bf16
    q, sf, gs = quantize_bf16(x.cuda())
    xs = x.float().numpy()
    rq, rsf, rgs = onv.quantize(xs)
    assert np.float32(gs.item()) == rgs == ref["gs_x"]
    assert (sf.cpu().numpy() == rsf).all() and (q.cpu().numpy() == onv.pack(rq)).all()
    # the bar plus, per element, how far FP4 re-quantisation of h can move it when
    # h (fp32 on the GPU, float64 in the oracle) rounds the other way to bf16 at
    # elements that lie on a bf16 midpoint straddling an FP4 decision (computed
    # by the oracle alone; tests/golden/make_w4a4_full.py)
    check_outputs(out[toks], ref["out"].astype(np.float64), extra=ref["flip"].astype(np.float64),
                  what="w4a4 full size (64 stored tokens)")
