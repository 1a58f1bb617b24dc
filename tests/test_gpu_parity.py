"""CUDA path against the CPU oracle, through the C ABI, on seeded inputs.

Integer results (routing ids, counts, offsets, permutation, NVFP4 codes and
scales, global scales) must match bit for bit; float results within the
bars of tests/tolerance.py.
"""
import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import moe as omoe
from oracle import nvfp4 as onv
from tests.gpu_layers import OracleWeights, device_layer
from tests.tolerance import TOPK_W_ABS, check_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def B():
    from nvfp4_mixture_experts_moe_gb300 import binding
    return binding


def route_gpu(logits, k):
    T, E = logits.shape
    ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    B().moe_route_topk(logits.cuda(), T, E, k, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T,E,k,kind", [
    (16, 8, 2, "normal"), (8, 320, 8, "normal"), (4096, 320, 8, "normal"), (2048, 320, 8, "zipf"),
    (16384, 256, 8, "normal"), (5, 1024, 32, "normal"), (3, 7, 7, "normal"), (33, 40, 1, "ties")])
def test_route_topk(T, E, k, kind):
    g = torch.Generator().manual_seed(T * 31 + E)
    if kind == "ties":
        logits = torch.randint(-2, 3, (T, E), generator=g).float()
        logits[0, :] = 0.0
        logits[0, ::2] = -0.0
    else:
        cfg = si.LayerConfig("r", T=T, H=16, I=16, I_s=16, E=E, k=k, logits=kind)
        logits = si.make_logits(cfg)
    ids, w = route_gpu(logits, k)
    rids, rw = omoe.route(logits.numpy(), k)
    assert (ids == rids).all()
    assert np.abs(w - rw).max() <= TOPK_W_ABS


@pytest.mark.parametrize("T,k,E", [(16, 2, 8), (8, 8, 320), (4096, 8, 320), (2048, 8, 320),
                                   (16384, 8, 256), (1, 1, 1), (7, 3, 1024), (0, 8, 320)])
def test_permute(T, k, E):
    g = torch.Generator().manual_seed(T + 7 * E)
    if E == 320 and T == 2048:
        cfg = si.LayerConfig("z", T=T, H=16, I=16, I_s=16, E=E, k=k, logits="zipf")
        ids_cpu = torch.from_numpy(omoe.route(si.make_logits(cfg).numpy(), k)[0])
    else:
        ids_cpu = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    P = T * k
    ids = ids_cpu.cuda()
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(max(P, 1), dtype=torch.int32, device="cuda")
    inv = torch.empty(max(P, 1), dtype=torch.int32, device="cuda")
    ws = torch.zeros(B().moe_permute_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    B().moe_permute(ids, T, k, E, counts, offsets, perm, inv, ws)
    assert B().moe_get_device_status(ws) == 0
    rc, ro, rp, ri = omoe.permute(ids_cpu.numpy(), E)
    assert (counts.cpu().numpy() == rc).all()
    assert (offsets.cpu().numpy() == ro).all()
    assert (perm.cpu().numpy()[:P] == rp).all()
    assert (inv.cpu().numpy()[:P] == ri).all()


def test_permute_flags_out_of_range_ids():
    ids = torch.tensor([[0, 1], [9, 2]], dtype=torch.int32, device="cuda")
    counts = torch.empty(4, dtype=torch.int32, device="cuda")
    offsets = torch.empty(5, dtype=torch.int32, device="cuda")
    perm = torch.empty(4, dtype=torch.int32, device="cuda")
    inv = torch.empty(4, dtype=torch.int32, device="cuda")
    ws = torch.zeros(B().moe_permute_workspace_size(2, 2, 4), dtype=torch.uint8, device="cuda")
    B().moe_permute(ids, 2, 2, 4, counts, offsets, perm, inv, ws)
    assert B().moe_get_device_status(ws) == B().MOE_ERR_DEVICE
    assert B().moe_get_device_status(ws) == 0      # cleared by the read
    assert counts.cpu().tolist() == [1, 1, 1, 0]
    assert inv.cpu().tolist()[2] == -1


def quant_gpu(x_bf16):
    from nvfp4_mixture_experts_moe_gb300 import quantize_bf16
    q, sf, gs = quantize_bf16(x_bf16.cuda())
    torch.cuda.synchronize()
    return q.cpu().numpy(), sf.cpu().numpy(), np.float32(gs.item())


@pytest.mark.parametrize("rows,K,scale,outliers", [(16, 256, 1.0, False), (64, 4096, 0.02, False),
                                                   (257, 7168, 1.0, True), (3, 16, 1e-3, False)])
def test_quantize_bit_exact(rows, K, scale, outliers):
    g = torch.Generator().manual_seed(rows * K)
    x = torch.randn(rows, K, generator=g) * scale
    if outliers:
        m = torch.rand(rows, K, generator=g) < 0.001
        x = torch.where(m, x * 20, x)
    x = x.to(torch.bfloat16)
    q, sf, gs = quant_gpu(x)
    rq, rsf, rgs = onv.quantize(x.float().numpy())
    assert gs == rgs
    assert (sf == rsf).all()
    assert (q == onv.pack(rq)).all()


def test_quantize_ties_and_edges():
    # values constructed to land exactly on e2m1 and e4m3 rounding midpoints
    vals = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -5.0, 0.0, -0.0, 4.0, 3.0, 1.0, 0.5]
    x = torch.tensor([vals, [v * 0.37 for v in vals], [1e-30] * 16, [0.0] * 16], dtype=torch.float32)
    x[0, 7] = 6.0  # block amax 6 -> gs/sf chosen by the quantiser
    x = x.to(torch.bfloat16)
    q, sf, gs = quant_gpu(x)
    rq, rsf, rgs = onv.quantize(x.float().numpy())
    assert gs == rgs and (sf == rsf).all() and (q == onv.pack(rq)).all()
    z = torch.zeros(2, 32, dtype=torch.bfloat16)
    q, sf, gs = quant_gpu(z)
    assert gs == 1.0 and (q == 0).all() and (sf == 0).all()


def run_forward(name, T=None):
    cfg, layer = device_layer(name, T)
    x = si.make_x(cfg)
    logits = si.make_logits(cfg)
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
    ws = layer.workspace()
    out = layer.forward(x.cuda(), logits.cuda(), topk_ids=ids, ws=ws)
    torch.cuda.synchronize()
    from nvfp4_mixture_experts_moe_gb300 import binding
    assert binding.moe_get_device_status(ws) == 0
    return cfg, layer, x, logits, out.float().cpu().numpy(), ids.cpu().numpy()


def test_forward_tiny_full_check():
    cfg, layer, x, logits, out, ids = run_forward("tiny")
    ow = OracleWeights(cfg)
    experts, shared = ow.all()
    ref, parts = omoe.layer(x.float().numpy(), logits.numpy(), experts, shared, cfg.k, return_parts=True)
    assert (ids == parts["ids"]).all()
    check_outputs(out, ref, what="tiny")


def test_forward_tiny_is_deterministic():
    cfg, layer = device_layer("tiny")
    x = si.make_x(cfg).cuda()
    logits = si.make_logits(cfg).cuda()
    outs = [layer.forward(x, logits).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], o) for o in outs[1:])


@pytest.mark.parametrize("cfg", [
    si.LayerConfig("mid4", T=300, H=512, I=256, I_s=256, E=4, k=2),     # groups ~150 rows: tensor-core path
    si.LayerConfig("mid16", T=300, H=256, I=128, I_s=128, E=16, k=2),   # groups ~37 rows: both paths
    si.LayerConfig("midz", T=160, H=256, I=192, I_s=192, E=24, k=4, logits="zipf"),  # skewed, empty groups
])
def test_forward_mid_full_check(cfg):
    cfg, layer, x, logits, out, ids = run_forward(cfg)
    ow = OracleWeights(cfg)
    experts, shared = ow.all()
    ref, parts = omoe.layer(x.float().numpy(), logits.numpy(), experts, shared, cfg.k, return_parts=True)
    assert (ids == parts["ids"]).all()
    check_outputs(out, ref, what=cfg.name)


def test_forward_group_sizes_cover_tile_shapes():
    # top-1 routing forced by the logits: groups of 33..128 rows give every
    # 16-row residue of the 128-row token tiles of the large-group GEMMs;
    # 129..513 rows the 256-row tiles (two 128-row boxes, one box for a short
    # tail, exact multiples)
    sizes = [33, 40, 70, 90, 100, 128, 129, 200, 256, 300, 513]
    cfg = si.LayerConfig("groups11", T=sum(sizes), H=256, I=128, I_s=128, E=len(sizes), k=1)
    _, layer = device_layer(cfg)
    rng = np.random.default_rng(7)
    expert_of = rng.permutation(np.repeat(np.arange(len(sizes)), sizes))
    logits = torch.from_numpy(rng.standard_normal((cfg.T, cfg.E)).astype(np.float32))
    logits[torch.arange(cfg.T), torch.from_numpy(expert_of)] += 10.0
    x = si.make_x(cfg)
    ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
    ws = layer.workspace()
    out = layer.forward(x.cuda(), logits.cuda(), topk_ids=ids, ws=ws)
    torch.cuda.synchronize()
    from nvfp4_mixture_experts_moe_gb300 import binding
    assert binding.moe_get_device_status(ws) == 0
    assert (ids.cpu().numpy()[:, 0] == expert_of).all()
    experts, shared = OracleWeights(cfg).all()
    ref = omoe.layer(x.float().numpy(), logits.numpy(), experts, shared, cfg.k)
    check_outputs(out.float().cpu().numpy(), ref, what="groups11")
    narrow = _forward_narrow_tiles(layer, x.cuda(), logits.cuda(), ws)
    assert torch.equal(narrow, out), "128-row tiles differ from the default tiles"


def test_forward_decode_full_check():
    cfg, layer, x, logits, out, ids = run_forward("decode")
    ow = OracleWeights(cfg)
    rids, rw = omoe.route(logits.numpy(), cfg.k)
    assert (ids == rids).all()
    ref = omoe.token_outputs_w4a16(x.float().numpy(), rids, rw, ow, ow(cfg.E))
    check_outputs(out, ref, what="decode")


def _forward_narrow_tiles(layer, x, logits, ws):
    """The forward with every large group in 128-row tiles (the W4A16 GEMMs'
    other tile shape)."""
    from nvfp4_mixture_experts_moe_gb300 import binding as Bd
    try:
        Bd.moe_debug_set(Bd.MOE_DEBUG_F16_TILE, 1)
        out = layer.forward(x, logits, ws=ws).clone()
        torch.cuda.synchronize()
        assert Bd.moe_get_device_status(ws) == 0
    finally:
        Bd.moe_debug_set(Bd.MOE_DEBUG_F16_TILE, 0)
    return out


def test_grouped_gemm_row_count_checked():
    """The public W4A16 grouped GEMM's row count: a larger one than the
    groups hold gives the exact count's bits (rows past the groups are
    neither read nor computed); a smaller one makes the large-group GEMM
    record MOE_ERR_DEVICE and compute nothing."""
    from nvfp4_mixture_experts_moe_gb300 import binding as Bd
    rows = [40, 300, 7, 129]
    G, N, K = len(rows), 256, 512
    buf, _ = _prepared_groups(G, N, K, 1, seed=31)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    total = int(off[-1])
    g = torch.Generator().manual_seed(6)
    a = torch.randn(total + 3, K, generator=g).to(torch.bfloat16).cuda()
    idx = torch.randperm(total + 3, generator=g)[:total].to(torch.int32).cuda()
    offs = torch.from_numpy(off).cuda()

    def run(count):
        out = torch.full((total, N // 2), float("nan"), dtype=torch.bfloat16, device="cuda")
        args = Bd.MoeGemmArgs(mode=0, gate_up=1, num_groups=G, N=N, K=K, rows=count)
        args.weights, args.group_offsets = buf.data_ptr(), offs.data_ptr()
        args.a, args.a_row_index, args.out = a.data_ptr(), idx.data_ptr(), out.data_ptr()
        ws = torch.zeros(Bd.moe_gemm_workspace_size_rows(G, count, K), dtype=torch.uint8, device="cuda")
        Bd.moe_nvfp4_grouped_gemm(args, ws)
        return out, Bd.moe_get_device_status(ws)

    exact, st = run(total)
    assert st == 0
    more, st = run(total + 37)
    assert st == 0 and torch.equal(more, exact)
    _, st = run(total - 1)
    assert st == Bd.MOE_ERR_DEVICE


_SHARED_WEIGHTS = {}


def _oracle_weights(cfg):
    """One OracleWeights per set of layer weights: the prefill and skewed
    workloads share their layer (same seed and shapes), so the oracle quantises
    its 321 experts once for both."""
    key = (cfg.seed, cfg.H, cfg.I, cfg.I_s, cfg.E)
    if key not in _SHARED_WEIGHTS:
        _SHARED_WEIGHTS.clear()
        _SHARED_WEIGHTS[key] = OracleWeights(cfg)
    return _SHARED_WEIGHTS[key]


@pytest.mark.parametrize("name", ["prefill", "skewed"])
def test_forward_large_full_check(name):
    """Every output of the prefill (4096 tokens) and skewed (2048 tokens,
    Zipf-biased routing with empty groups) workloads against the oracle's
    whole layer: every 128-row tile and ragged tail of every expert group."""
    cfg, layer, x, logits, out, ids = run_forward(name)
    rids, rw = omoe.route(logits.numpy(), cfg.k)
    assert (ids == rids).all()
    counts = np.bincount(rids.ravel(), minlength=cfg.E)
    if name == "skewed":
        assert (counts == 0).any() and counts.max() > 512
    ow = _oracle_weights(cfg)
    ow.prefetch(list(range(cfg.E + 1)))
    experts, shared = ow.all()
    ref = omoe.layer(x.float().numpy(), logits.numpy(), experts, shared, cfg.k)
    check_outputs(out, ref, what=f"{name} (all {cfg.T} tokens)")
    # the checked bits again from the 128-row tiles alone and from repeated
    # launches of the default tiles (a race between a stage's readers and its
    # refill shows as a few wrong weight rows in some launches)
    from nvfp4_mixture_experts_moe_gb300 import binding as Bd
    xd, ld = x.cuda(), logits.cuda()
    ws = layer.workspace()
    runs = [_forward_narrow_tiles(layer, xd, ld, ws)]
    runs += [layer.forward(xd, ld, ws=ws).clone() for _ in range(4)]
    torch.cuda.synchronize()
    assert Bd.moe_get_device_status(ws) == 0
    differ = [i for i, r in enumerate(runs) if not np.array_equal(r.float().cpu().numpy(), out)]
    assert not differ, f"runs {differ} (0: 128-row tiles, 1..4: repeats) differ from the checked output"


def _prepared_groups(G, N, K, gate_up, seed):
    """G prepared NVFP4 matrices (device) + the oracle's QuantWeights of the same bf16 values."""
    from nvfp4_mixture_experts_moe_gb300 import binding as Bd, quantize_bf16
    g = torch.Generator().manual_seed(seed)
    size = Bd.moe_prepare_size(N, K, 0, gate_up)
    buf = torch.empty(G * size, dtype=torch.uint8, device="cuda")
    oracle_w = []
    for i in range(G):
        if gate_up:
            mats = [(torch.randn(N // 2, K, generator=g) * 0.02).to(torch.bfloat16) for _ in range(2)]
        else:
            mats = [(torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)]
        qs = [quantize_bf16(m.cuda()) for m in mats]
        codes = torch.cat([q[0] for q in qs])
        sfs = torch.cat([q[1] for q in qs])
        gss = [q[2].item() for q in qs]
        Bd.moe_nvfp4_prepare_weights(codes, sfs, gss, N, K, 0, gate_up, buf[i * size:(i + 1) * size])
        oracle_w.append([omoe.QuantWeight.from_dense(m.float().numpy()) for m in mats])
    return buf, oracle_w


@pytest.mark.parametrize("f16_copy", [False, True], ids=["direct", "f16_copy"])
@pytest.mark.parametrize("gate_up", [1, 0])
def test_grouped_gemm_entry_tile_edges(gate_up, f16_copy):
    """The public grouped GEMM against the oracle on empty, small, ragged and
    multi-tile groups, both without the row count (the kernel that reads the
    bf16 rows directly) and with it and room for the f16 copy (the forward's
    128-row and 256-row tile kernels)."""
    from nvfp4_mixture_experts_moe_gb300 import binding as Bd
    rows = [0, 40, 300, 7, 129, 33, 1, 256]
    G = len(rows)
    N, K = (256, 512) if gate_up else (384, 256)
    buf, ow = _prepared_groups(G, N, K, gate_up, seed=11 + gate_up)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    total = int(off[-1])
    g = torch.Generator().manual_seed(5)
    src_rows = total + 3
    a = torch.randn(src_rows, K, generator=g).to(torch.bfloat16)
    idx = torch.randperm(src_rows, generator=g)[:total].to(torch.int32)
    rs = torch.rand(total, generator=g) + 0.5
    out_cols = N // 2 if gate_up else N
    out = torch.full((total, out_cols), float("nan"), dtype=torch.bfloat16, device="cuda")
    args = Bd.MoeGemmArgs(mode=0, gate_up=gate_up, num_groups=G, N=N, K=K)
    offs_d = torch.from_numpy(off).cuda()
    a_d, idx_d, rs_d = a.cuda(), idx.cuda(), rs.cuda()
    args.weights = buf.data_ptr()
    args.group_offsets = offs_d.data_ptr()
    args.a = a_d.data_ptr()
    args.a_row_index = idx_d.data_ptr()
    args.row_scale = None if gate_up else rs_d.data_ptr()
    args.out = out.data_ptr()
    if f16_copy:
        args.rows = total
        ws = torch.zeros(Bd.moe_gemm_workspace_size_rows(G, total, K), dtype=torch.uint8, device="cuda")
    else:
        ws = torch.zeros(Bd.moe_gemm_workspace_size(G), dtype=torch.uint8, device="cuda")
    Bd.moe_nvfp4_grouped_gemm(args, ws)
    assert Bd.moe_get_device_status(ws) == 0
    got = out.float().cpu().numpy()
    xa = a.float().numpy()[idx.numpy()]
    for gi in range(G):
        r0, r1 = off[gi], off[gi + 1]
        if r1 == r0:
            continue
        if gate_up:
            ref = omoe.gate_up_swiglu(xa[r0:r1], ow[gi][0], ow[gi][1])
        else:
            ref = omoe.down_proj(xa[r0:r1], ow[gi][0]) * rs.numpy()[r0:r1, None]
        check_outputs(got[r0:r1], ref, what=f"group {gi} ({r1 - r0} rows)")
