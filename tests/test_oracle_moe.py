"""Pins of the oracle's routing, permutation and layer to facts outside itself:
brute force, invariants, library routines (torch.matmul, torch silu) and a
dense reformulation of the layer that never permutes."""
import itertools

import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import moe, nvfp4


def test_route_brute_force_tiny():
    rng = np.random.default_rng(0)
    for T, E, k in [(5, 4, 1), (7, 6, 3), (3, 8, 8), (9, 16, 4)]:
        logits = rng.integers(-3, 4, size=(T, E)).astype(np.float32)  # many exact ties
        ids, w = moe.route(logits, k)
        for t in range(T):
            brute = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
            assert ids[t].tolist() == brute
            ex = np.exp(logits[t].astype(np.float64) - logits[t].max())
            ref = ex[brute] / ex[brute].sum()
            assert np.abs(w[t] - ref).max() <= 1e-7
        assert np.abs(w.astype(np.float64).sum(axis=1) - 1).max() <= 1e-6


def test_route_ties_and_signed_zero():
    logits = np.array([[0.0, -0.0, 0.0, -1.0, 0.0]], dtype=np.float32)
    ids, w = moe.route(logits, 3)
    assert ids.tolist() == [[0, 1, 2]]
    assert np.allclose(w, 1 / 3)
    logits = np.array([[1.0, 2.0, 2.0, 2.0]], dtype=np.float32)
    ids, _ = moe.route(logits, 2)
    assert ids.tolist() == [[1, 2]]


def test_route_k_equals_e_is_full_rank_order():
    logits = np.array([[0.3, -1.0, 2.0, 0.3, 5.0]], dtype=np.float32)
    ids, w = moe.route(logits, 5)
    assert ids.tolist() == [[4, 2, 0, 3, 1]]
    p = torch.softmax(torch.tensor(logits, dtype=torch.float64), dim=1).numpy()
    assert np.abs(w[0] - p[0, ids[0]]).max() <= 1e-7


def test_silu_matches_torch():
    z = np.linspace(-30, 30, 10001)
    ref = torch.nn.functional.silu(torch.tensor(z, dtype=torch.float64)).numpy()
    assert np.abs(moe.silu(z) - ref).max() <= 1e-12


def test_permute_invariants_and_stability():
    rng = np.random.default_rng(1)
    for T, E, k in [(1, 1, 1), (16, 8, 2), (50, 7, 3), (33, 40, 5)]:
        ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
        counts, offsets, perm, inv = moe.permute(ids, E)
        P = T * k
        assert counts.sum() == P
        assert offsets[0] == 0 and offsets[-1] == P
        assert (np.diff(offsets) == counts).all()
        assert (inv[perm] == np.arange(P)).all() and (perm[inv] == np.arange(P)).all()
        flat = ids.reshape(-1)
        ref = sorted(range(P), key=lambda p: (flat[p], p))   # Python's stable sort
        assert perm.tolist() == ref
        for e in range(E):
            assert (flat[perm[offsets[e]:offsets[e + 1]]] == e).all()


def test_permute_empty_and_out_of_range():
    counts, offsets, perm, inv = moe.permute(np.zeros((0, 4), dtype=np.int32), 5)
    assert counts.sum() == 0 and offsets.tolist() == [0] * 6 and perm.size == 0
    with pytest.raises(ValueError):
        moe.permute(np.array([[0, 5]]), 5)


def _tiny_layer(cfg):
    W = si.make_layer_weights(cfg)
    qw = {e: tuple(moe.QuantWeight.from_dense(m.float().numpy()) for m in W[e]) for e in W}
    x = si.make_x(cfg).float().numpy()
    logits = si.make_logits(cfg).numpy()
    return x, logits, [qw[e] for e in range(cfg.E)], qw[cfg.E]


def _ffn_torch(x, trip, hq=None):
    g, u, d = (torch.tensor(m.dequantize()) for m in trip)
    xt = torch.tensor(x, dtype=torch.float64)
    h = torch.nn.functional.silu(torch.matmul(xt, g.T)) * torch.matmul(xt, u.T)
    return h.numpy(), d.numpy()


def test_layer_matches_dense_formulation_w4a16():
    cfg = si.CONFIGS["tiny"]
    x, logits, experts, shared = _tiny_layer(cfg)
    out = moe.layer(x, logits, experts, shared, cfg.k)
    ids, w = moe.route(logits, cfg.k)
    R = np.zeros((cfg.T, cfg.E))
    for t in range(cfg.T):
        for j in range(cfg.k):
            R[t, ids[t, j]] += w[t, j]
    dense = np.zeros_like(out)
    for e in range(cfg.E):
        h, d = _ffn_torch(x, experts[e])
        dense += R[:, e:e + 1] * (torch.tensor(h) @ torch.tensor(d).T).numpy()
    h, d = _ffn_torch(x, shared)
    dense += (torch.tensor(h) @ torch.tensor(d).T).numpy()
    assert np.abs(out - dense).max() <= 1e-12 * max(1.0, np.abs(dense).max())


def test_layer_matches_dense_formulation_w4a4():
    cfg = si.CONFIGS["tiny"]
    x, logits, experts, shared = _tiny_layer(cfg)
    out, parts = moe.layer(x, logits, experts, shared, cfg.k, mode="w4a4", return_parts=True)
    ids, w = moe.route(logits, cfg.k)
    xq, xsf, xgs = nvfp4.quantize(x.astype(np.float32))
    xd = nvfp4.dequantize(xq, xsf, xgs)
    # h of every routed (token, expert) pair and of the shared rows; one global
    # scale over all of them; each row quantises on its own given that scale.
    rows = {}
    for t in range(cfg.T):
        for j in range(cfg.k):
            rows[(t, int(ids[t, j]))] = _ffn_torch(xd[t:t + 1], experts[ids[t, j]])[0][0]
    hs_shared = _ffn_torch(xd, shared)[0]
    allh = np.concatenate([np.stack(list(rows.values())), hs_shared])
    hb = torch.tensor(allh, dtype=torch.float32).to(torch.bfloat16).float().numpy()
    amax = np.abs(hb).max()
    gs = np.float32(2688.0) / np.float32(amax)
    assert gs == parts["hgs"]
    dense = np.zeros_like(out)
    for i, ((t, e), h) in enumerate(rows.items()):
        q, sf, _ = nvfp4.quantize(np.concatenate([hb[i:i + 1], [[amax] + [0] * (hb.shape[1] - 1)]]))
        hd = nvfp4.dequantize(q[:1], sf[:1], gs)
        d = torch.tensor(experts[e][2].dequantize())
        wt = w[t, list(ids[t]).index(e)]
        dense[t] += wt * (torch.tensor(hd) @ d.T).numpy()[0]
    for t in range(cfg.T):
        i = len(rows) + t
        q, sf, _ = nvfp4.quantize(np.concatenate([hb[i:i + 1], [[amax] + [0] * (hb.shape[1] - 1)]]))
        hd = nvfp4.dequantize(q[:1], sf[:1], gs)
        dense[t] += (torch.tensor(hd) @ torch.tensor(shared[2].dequantize()).T).numpy()[0]
    assert np.abs(out - dense).max() <= 1e-12 * max(1.0, np.abs(dense).max())


def test_identical_experts_invariant():
    cfg = si.LayerConfig("same", T=12, H=64, I=32, I_s=48, E=6, k=3)
    W = si.make_layer_weights(cfg, experts=[0, cfg.E])
    e0 = tuple(moe.QuantWeight.from_dense(m.float().numpy()) for m in W[0])
    sh = tuple(moe.QuantWeight.from_dense(m.float().numpy()) for m in W[cfg.E])
    x = si.make_x(cfg).float().numpy()
    for trial in range(3):
        logits = np.random.default_rng(trial).standard_normal((cfg.T, cfg.E)).astype(np.float32)
        out = moe.layer(x, logits, [e0] * cfg.E, sh, cfg.k)
        h, d = _ffn_torch(x, e0)
        hs, ds = _ffn_torch(x, sh)
        ref = h @ d.T + hs @ ds.T
        # routing weights sum to 1 (to fp32 rounding), so the mixture is the expert
        assert np.abs(out - ref).max() <= 1e-6 * max(1.0, np.abs(ref).max())


def test_one_expert_reduces_to_dense_ffn():
    cfg = si.LayerConfig("one", T=10, H=128, I=64, I_s=64, E=1, k=1)
    W = si.make_layer_weights(cfg, experts=[0])
    e0 = tuple(moe.QuantWeight.from_dense(m.float().numpy()) for m in W[0])
    x = si.make_x(cfg).float().numpy()
    logits = si.make_logits(cfg).numpy()
    out = moe.layer(x, logits, [e0], None, 1)
    g, u, d = (torch.tensor(m.dequantize()) for m in e0)
    xt = torch.tensor(x, dtype=torch.float64)
    ref = torch.matmul(torch.nn.functional.silu(xt @ g.T) * (xt @ u.T), d.T).numpy()
    assert np.abs(out - ref).max() <= 1e-12 * np.abs(ref).max()


def test_token_outputs_match_layer():
    cfg = si.CONFIGS["tiny"]
    x, logits, experts, shared = _tiny_layer(cfg)
    out = moe.layer(x, logits, experts, shared, cfg.k)
    ids, w = moe.route(logits, cfg.k)
    sel = [0, 5, 15]
    got = moe.token_outputs_w4a16(x[sel], ids[sel], w[sel], lambda e: experts[e], shared)
    assert np.abs(got - out[sel]).max() <= 1e-12


def test_brute_force_gemm_tiny():
    # plain Python loops over a few outputs of the tiny layer
    cfg = si.CONFIGS["tiny"]
    x, logits, experts, shared = _tiny_layer(cfg)
    out = moe.layer(x, logits, experts, shared, cfg.k)
    ids, w = moe.route(logits, cfg.k)
    t = 3

    def ffn_point(trip, xt, f):
        g, u, d = trip
        wg, wu, wd = g.dequantize(), u.dequantize(), d.dequantize()
        acc = 0.0
        for i in range(wg.shape[0]):
            gi = sum(float(xt[c]) * float(wg[i, c]) for c in range(len(xt)))
            ui = sum(float(xt[c]) * float(wu[i, c]) for c in range(len(xt)))
            acc += gi / (1.0 + np.exp(-gi)) * ui * float(wd[f, i])
        return acc

    for f in (0, 77, 255):
        ref = sum(float(w[t, j]) * ffn_point(experts[ids[t, j]], x[t], f) for j in range(cfg.k))
        ref += ffn_point(shared, x[t], f)
        assert abs(out[t, f] - ref) <= 1e-12


def test_w4a4_golden_script_equals_layer():
    """The full-size W4A4 golden values come from tests/golden/make_w4a4_full.py,
    which computes a few tokens' outputs from the batch-wide global scales
    instead of running oracle.moe.layer on all 16384 tokens at once; on a small
    W4A4 layer the two must agree to float64 rounding, with the same scales."""
    import importlib.util
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "make_w4a4_full.py")
    spec = importlib.util.spec_from_file_location("make_w4a4_full", path)
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    cfg = si.LayerConfig("w4a4_pin", T=64, H=512, I=256, I_s=256, E=8, k=2, mode="w4a4", outliers=True)
    toks = np.array([0, 5, 17, 40, 63])
    out, gs_x, amax_h, gs_h, ids, w, flip = mk.golden_rows(cfg, toks, threads=4, log=lambda m: None)
    assert flip.shape == out.shape and (flip >= 0).all()
    W = {e: tuple(moe.QuantWeight.from_dense(si.make_expert_weight(cfg, e, m).float().numpy())
                  for m in ("gate", "up", "down")) for e in range(cfg.E + 1)}
    ref, parts = moe.layer(si.make_x(cfg).float().numpy(), si.make_logits(cfg).numpy(),
                           [W[e] for e in range(cfg.E)], W[cfg.E], cfg.k, mode="w4a4", return_parts=True)
    assert gs_x == parts["xgs"] and gs_h == parts["hgs"]
    assert amax_h == np.float32(np.max(np.abs(parts["h_bf16"])))
    assert np.abs(out - ref[toks]).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_layer_matches_dense_formulation_mxfp4():
    """MXFP4 layer ("vLLM on the NVIDIA DGX Spark", section 6.4): every expert
    on every token weighted by the routing matrix, with x quantised once and
    each h row quantised on its own (no global scale), against the grouped
    layer."""
    from oracle import mxfp4
    cfg = si.LayerConfig("tiny_mx", T=16, H=256, I=128, I_s=128, E=8, k=2, mode="mxfp4")
    W = si.make_layer_weights(cfg)
    trips = {e: tuple(moe.QuantWeightMX.from_dense(m.float().numpy()) for m in W[e]) for e in W}
    x = si.make_x(cfg).float().numpy().astype(np.float64)
    logits = si.make_logits(cfg).numpy()
    experts, shared = [trips[e] for e in range(cfg.E)], trips[cfg.E]
    out = moe.layer(x, logits, experts, shared, cfg.k, mode="mxfp4")
    ids, w = moe.route(logits, cfg.k)
    xd = mxfp4.dequantize(*mxfp4.quantize(x.astype(np.float32)))

    def ffn(rows, trip):
        g, u, d = (torch.tensor(m.dequantize()) for m in trip)
        xt = torch.tensor(rows)
        h = torch.nn.functional.silu(xt @ g.T) * (xt @ u.T)
        hb = h.to(torch.float32).to(torch.bfloat16).float().numpy()
        hd = mxfp4.dequantize(*mxfp4.quantize(hb))
        return (torch.tensor(hd) @ d.T).numpy()

    dense = np.zeros_like(out)
    for t in range(cfg.T):
        for j in range(cfg.k):
            dense[t] += w[t, j] * ffn(xd[t:t + 1], experts[ids[t, j]])[0]
        dense[t] += ffn(xd[t:t + 1], shared)[0]
    assert np.abs(out - dense).max() <= 1e-12 * max(1.0, np.abs(dense).max())
    # and MXFP4 is not NVFP4: the same layer through the W4A4 path differs
    nv = {e: tuple(moe.QuantWeight.from_dense(m.float().numpy()) for m in W[e]) for e in W}
    out_nv = moe.layer(x, logits, [nv[e] for e in range(cfg.E)], nv[cfg.E], cfg.k, mode="w4a4")
    assert np.abs(out - out_nv).max() > 1e-3


@pytest.mark.parametrize("mode", ["w4a16", "mxfp4"])
def test_expert_shards_sum_to_the_layer(mode):
    """Expert parallelism: contiguous shards of the experts, each computing
    only its own pairs (the shared expert on one shard), add up to the whole
    layer. Modes without a per-tensor activation scale only (with dynamic
    W4A4 scales every shard quantises h with its own scale)."""
    cfg = si.LayerConfig("shards", T=24, H=256, I=128, I_s=128, E=10, k=3, mode=mode)
    W = si.make_layer_weights(cfg)
    kind = moe.QuantWeightMX if mode == "mxfp4" else moe.QuantWeight
    trips = {e: tuple(kind.from_dense(m.float().numpy()) for m in W[e]) for e in W}
    x = si.make_x(cfg).float().numpy().astype(np.float64)
    logits = si.make_logits(cfg).numpy()
    experts, shared = [trips[e] for e in range(cfg.E)], trips[cfg.E]
    full = moe.layer(x, logits, experts, shared, cfg.k, mode=mode)
    bounds = [0, 3, 7, 10]  # uneven shards
    parts = [moe.layer(x, logits, experts, shared if i == 0 else None, cfg.k, mode=mode,
                       experts_range=(bounds[i], bounds[i + 1])) for i in range(3)]
    assert np.abs(sum(parts) - full).max() <= 1e-12 * max(1.0, np.abs(full).max())
    # a shard without experts and without the shared expert contributes nothing
    empty = moe.layer(x, logits, experts, None, cfg.k, mode=mode, experts_range=(4, 4))
    assert not empty.any()


def test_requant_flip_bound_pins():
    """The W4A4 flip allowance: zero when no element of h can round to another
    bf16 value; exactly one dequantised step times |Wd column| for one element
    put on a bf16 midpoint whose two neighbours quantise differently."""
    rng = np.random.default_rng(3)
    H, I = 8, 32
    down_abs = np.abs(rng.standard_normal((H, I)))
    gs = np.float32(1.0)
    # bf16 values are a half ulp away from every midpoint: a window below
    # that never reaches another bf16 value
    h = moe.bf16_round(rng.standard_normal((1, I))).astype(np.float64)[0]
    assert not moe.requant_flip_bound(h, gs, down_abs, 1e-6 * np.abs(h)).any()
    # block 0 with amax 6 -> scale 1 (at gs = 1): e2m1 decides 2.5 between 2 and 3;
    # 2.5 is a bf16 value, so put h midway between 2.5 and its bf16 neighbour 2.515625
    h = np.zeros(I)
    h[0] = 6.0
    h[5] = 0.5 * (2.5 + 2.515625)
    got = moe.requant_flip_bound(h, gs, down_abs, 1e-6)
    d0 = nvfp4.dequantize(*nvfp4.quantize(np.array([[6.0, 0, 0, 0, 0, 2.5] + [0] * 10], np.float32), gs=gs)[:2], gs)
    d1 = nvfp4.dequantize(*nvfp4.quantize(np.array([[6.0, 0, 0, 0, 0, 2.515625] + [0] * 10], np.float32), gs=gs)[:2],
                          gs)
    step = np.abs(d1 - d0)[0]
    assert step[5] == 1.0 and step.sum() == 1.0        # 2.5 -> code of 2, 2.515625 -> code of 3
    assert np.array_equal(got, down_abs[:, 5] * 1.0)
    # a wide window on the block's maximum reaches another block scale: every
    # element of the block may move, and the bound covers the recomputed block
    h = np.zeros(I)
    h[:16] = moe.bf16_round(np.linspace(0.3, 5.9, 16)).astype(np.float64)
    win = np.zeros(I)
    win[15] = 0.2                                      # 5.90625 may be anything in [5.70625, 6.10625]
    got = moe.requant_flip_bound(h, gs, down_abs, win)
    base = nvfp4.dequantize(*nvfp4.quantize(h[None, :16].astype(np.float32), gs=gs)[:2], gs)[0]
    alt = h[:16].copy()
    alt[15] = 5.75                                     # in the window: 5.75 / 6 -> E4M3 scale 0.9375, not 1
    moved = np.abs(nvfp4.dequantize(*nvfp4.quantize(alt[None].astype(np.float32), gs=gs)[:2], gs)[0] - base)
    assert (moved[:15] > 0).any()                      # another block scale moves the other elements
    assert np.all(got >= down_abs[:, :16] @ moved - 1e-12)


def test_gate_up_window_contains_fp32_errors():
    """The fp32 window of h is zero for zero rows and contains the actual
    error of float32 evaluations of h in several summation orders (forward,
    reversed, blocked by 64 with a float32 accumulator across blocks)."""
    rng = np.random.default_rng(11)
    K, I = 1024, 64
    g = moe.QuantWeight.from_dense((rng.standard_normal((I, K)) * 0.02).astype(np.float32))
    u = moe.QuantWeight.from_dense((rng.standard_normal((I, K)) * 0.02).astype(np.float32))
    assert not moe.gate_up_window(np.zeros((2, K)), g, u).any()
    x = moe.bf16_round(rng.standard_normal((4, K)) * np.where(rng.random((4, K)) < 0.01, 20.0, 1.0)).astype(np.float64)
    exact = moe.gate_up_swiglu(x, g, u)
    win = moe.gate_up_window(x, g, u)
    gd, ud = g.dequantize().astype(np.float32), u.dequantize().astype(np.float32)
    x32 = x.astype(np.float32)

    def h32(order):
        gg = np.zeros((4, I), np.float32)
        uu = np.zeros((4, I), np.float32)
        if order == "blocked":
            for k0 in range(0, K, 64):
                gg = gg + (x32[:, k0:k0 + 64] @ gd[:, k0:k0 + 64].T).astype(np.float32)
                uu = uu + (x32[:, k0:k0 + 64] @ ud[:, k0:k0 + 64].T).astype(np.float32)
        else:
            ks = range(K) if order == "forward" else range(K - 1, -1, -1)
            for kk in ks:
                gg = gg + x32[:, kk:kk + 1] * gd[None, :, kk]
                uu = uu + x32[:, kk:kk + 1] * ud[None, :, kk]
        sg = (gg / (np.float32(1) + np.exp(-gg))).astype(np.float32)
        return (sg * uu).astype(np.float64)

    for order in ("forward", "reversed", "blocked"):
        err = np.abs(h32(order) - exact)
        assert np.all(err <= win), (order, float(np.max(err - win)))
    # and the window is not vacuous: well below |h| for most elements
    assert np.median(win / np.maximum(np.abs(exact), 1e-30)) < 2.0 ** -8


