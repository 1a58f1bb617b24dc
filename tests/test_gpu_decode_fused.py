"""The single-kernel decode path ("micro path": routing, permutation, both
expert GEMMs and the combine in one cooperative launch; "Serving Solar Open 2
on DGX Spark", "The fix") against the multi-kernel path and the oracle.

The two paths share their arithmetic (the same MMA inner loop, accumulation
order, row scales, epilogue operations and combine order), so their outputs
must agree bit for bit; the oracle check of the decode workload itself runs
in test_gpu_parity.py through whichever path the forward takes (this one).
"""
import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import moe as omoe
from tests.gpu_layers import OracleWeights, device_layer
from tests.tolerance import check_outputs

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
    for key in (B().MOE_DEBUG_WAIT_LIMIT, B().MOE_DEBUG_EXTRA_ARRIVALS, B().MOE_DEBUG_DISABLE_DECODE_FUSED):
        B().moe_debug_set(key, 0)


def _both_paths(layer, x, logits, T, k):
    outs = []
    for disable in (0, 1):
        B().moe_debug_set(B().MOE_DEBUG_DISABLE_DECODE_FUSED, disable)
        ids = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        ws = layer.workspace(T)
        launches0 = B().moe_kernel_launches()
        out = layer.forward(x, logits, topk_ids=ids, ws=ws)
        torch.cuda.synchronize()
        launches = B().moe_kernel_launches() - launches0
        assert B().moe_get_device_status(ws) == 0
        outs.append((out.clone(), ids.clone(), launches))
    return outs


@pytest.mark.parametrize("T", [1, 2, 5, 8])
def test_fused_equals_multi_kernel_path(T):
    cfg, layer = device_layer("decode")
    c = cfg.with_tokens(T)
    x = si.make_x(c).cuda()
    logits = si.make_logits(c).cuda()
    (fo, fi, fl), (mo, mi, ml) = _both_paths(layer, x, logits, T, cfg.k)
    assert fl == 1 and ml > 1           # one kernel against the chain
    assert torch.equal(fi, mi)
    assert torch.equal(fo, mo)
    rids, _ = omoe.route(logits.cpu().numpy(), cfg.k)
    assert (fi.cpu().numpy() == rids).all()


def test_fused_tiny_layer_against_oracle():
    cfg, layer = device_layer("tiny", T=8)
    x = si.make_x(cfg)
    logits = si.make_logits(cfg)
    (fo, fi, fl), (mo, _, _) = _both_paths(layer, x.cuda(), logits.cuda(), cfg.T, cfg.k)
    assert fl == 1 and torch.equal(fo, mo)
    experts, shared = OracleWeights(cfg).all()
    ref = omoe.layer(x.float().numpy(), logits.numpy(), experts, shared, cfg.k)
    check_outputs(fo.float().cpu().numpy(), ref, what="tiny T=8, single-kernel decode")


def test_fused_without_shared_expert():
    from nvfp4_mixture_experts_moe_gb300 import Nvfp4MoeLayer
    cfg = si.LayerConfig("noshared_dec", T=6, H=512, I=256, I_s=256, E=16, k=4)
    layer = Nvfp4MoeLayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, shared=False, device="cuda")
    W = si.make_layer_weights(cfg, experts=list(range(cfg.E)))
    for e in range(cfg.E):
        layer.set_expert(e, *W[e])
    x = si.make_x(cfg)
    logits = si.make_logits(cfg)
    (fo, _, fl), (mo, _, _) = _both_paths(layer, x.cuda(), logits.cuda(), cfg.T, cfg.k)
    assert fl == 1 and torch.equal(fo, mo)
    ow = OracleWeights(cfg)
    ref = omoe.layer(x.float().numpy(), logits.numpy(), [ow(e) for e in range(cfg.E)], None, cfg.k)
    check_outputs(fo.float().cpu().numpy(), ref, what="no shared expert, single-kernel decode")


def test_fused_with_router_gemm():
    cfg, layer = device_layer("decode")
    x = si.make_x(cfg).cuda()
    layer.set_router(si.make_router_weight(cfg))
    try:
        (fo, fi, _), (mo, mi, _) = _both_paths(layer, x, None, cfg.T, cfg.k)
    finally:
        layer.set_router(None)
    assert torch.equal(fi, mi) and torch.equal(fo, mo)


def test_fused_is_deterministic():
    cfg, layer = device_layer("decode")
    x = si.make_x(cfg).cuda()
    logits = si.make_logits(cfg).cuda()
    outs = [layer.forward(x, logits).clone() for _ in range(5)]
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_fused_timeout_is_reported_and_recovers():
    """The down phase waits for arrivals that never come: every wait gives up
    after the (shortened) limit, the status word reads MOE_ERR_TIMEOUT, and the
    next forward on the same workspace is correct again."""
    cfg, layer = device_layer("tiny", T=8)
    x = si.make_x(cfg).cuda()
    logits = si.make_logits(cfg).cuda()
    ws = layer.workspace()
    good = layer.forward(x, logits, ws=ws).clone()
    torch.cuda.synchronize()
    assert B().moe_get_device_status(ws) == 0
    B().moe_debug_set(B().MOE_DEBUG_WAIT_LIMIT, 2_000_000)      # ~1 ms
    B().moe_debug_set(B().MOE_DEBUG_EXTRA_ARRIVALS, 1)
    layer.forward(x, logits, ws=ws)
    torch.cuda.synchronize()
    assert B().moe_get_device_status(ws) == B().MOE_ERR_TIMEOUT
    B().moe_debug_set(B().MOE_DEBUG_EXTRA_ARRIVALS, 0)
    B().moe_debug_set(B().MOE_DEBUG_WAIT_LIMIT, 0)
    again = layer.forward(x, logits, ws=ws)
    torch.cuda.synchronize()
    assert B().moe_get_device_status(ws) == 0
    assert torch.equal(good, again)


def test_fused_counters_survive_workspace_reuse():
    """The single-kernel path keeps its counters in a fixed region after the
    workspace header and leaves them zero at the end of every launch. A
    workspace whose bytes past the header start as garbage, then serves a
    multi-kernel (larger T) forward and a standalone permutation (whose
    scratch overlaps the region), still gives the decode call's exact bits."""
    cfg, layer = device_layer("decode")
    x = si.make_x(cfg).cuda()
    logits = si.make_logits(cfg).cuda()
    ref = layer.forward(x, logits).clone()              # fresh workspace
    big = cfg.with_tokens(64)                           # multi-kernel path
    ws = layer.workspace(big.T)
    ws[256:].fill_(0xFF)                                # garbage past the zeroed header
    first = layer.forward(x, logits, ws=ws).clone()     # first use: the region is zeroed
    again = layer.forward(x, logits, ws=ws).clone()     # steady state: counters left zero
    layer.forward(si.make_x(big).cuda(), si.make_logits(big).cuda(), ws=ws)
    after_big = layer.forward(x, logits, ws=ws).clone()
    ids = torch.randint(0, cfg.E, (big.T, cfg.k), dtype=torch.int32, device="cuda")
    counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(big.T * cfg.k, dtype=torch.int32, device="cuda")
    inv = torch.empty_like(perm)
    B().moe_permute(ids, big.T, cfg.k, cfg.E, counts, offsets, perm, inv, ws)
    after_permute = layer.forward(x, logits, ws=ws).clone()
    torch.cuda.synchronize()
    assert B().moe_get_device_status(ws) == 0
    for name, o in (("first", first), ("again", again), ("after_big", after_big), ("after_permute", after_permute)):
        assert torch.equal(o, ref), name


def test_fused_counter_sets_alternate_across_shapes_and_graph_replays():
    """Launches alternate between the workspace's two counter sets (a ticket
    per launch): decode batches of different sizes interleaved on one
    workspace, and one forward captured in a CUDA graph and replayed (every
    replay takes new tickets), each give the bits of a forward on a fresh
    workspace."""
    cfg, layer = device_layer("decode")
    xs = {T: si.make_x(cfg.with_tokens(T)).cuda() for T in (1, 2, 5, 8)}
    ls = {T: si.make_logits(cfg.with_tokens(T)).cuda() for T in (1, 2, 5, 8)}
    ref = {T: layer.forward(xs[T], ls[T]).clone() for T in xs}   # fresh workspaces
    ws = layer.workspace(8)
    for T in (8, 2, 8, 5, 8, 1, 8, 8, 2):
        got = layer.forward(xs[T], ls[T], ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(got, ref[T]), T
    out = torch.empty_like(ref[8])
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        layer.forward(xs[8], ls[8], out=out, ws=ws)      # warm-up on the capture stream
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        layer.forward(xs[8], ls[8], out=out, ws=ws, stream=stream)
    for _ in range(5):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref[8])
    assert B().moe_get_device_status(ws) == 0
