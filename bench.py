#!/usr/bin/env python
"""Benchmark of the fused NVFP4 MoE layer on GB300.

One step = one full pass of the layer (route, permute, [quantise x], gate/up
GEMM + SwiGLU, [quantise h], down GEMM + routing weight, combine) over one
batch of seeded synthetic input, through the C ABI ``moe_nvfp4_forward``.
The default workload is the decode-shaped layer (8 tokens, hidden 4096,
expert intermediate 1536, 320 routed experts top-8 + 1 shared, W4A16).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
    python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Prints one JSON line (rank 0). With N > 1 (torchrun) every rank runs an
independent replica of the same workload (the layer does not shard here:
replicas only) and ``value`` is the sum over ranks. On one GPU the line also
carries ``configs``: the same measurement (step time, tokens/s, roofline of
the dominant kernel, layer roofline, end-to-end number, CPU baseline) for
every other workload (tiny, prefill, skewed, W4A4), run in the same process
after the headline; ``--only`` skips them.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and % of roofline (HBM GB/s decode, FP4/BF16 TFLOP/s prefill)"
L2_BYTES = 129 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="decode")
    ap.add_argument("--batches", type=int, default=4, help="distinct input batches rotated over steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=2)
    ap.add_argument("--tokens", type=int, default=None, help="override T (a smaller case, e.g. for ncu)")
    ap.add_argument("--experts", type=int, default=None, help="override E (a smaller case, e.g. for ncu)")
    ap.add_argument("--only", action="store_true", help="measure the chosen workload only (no 'configs' key)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sus": p.get("bf16_tflops_sustained"),
                "source": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sus": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
class ClockSampler:
    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if self.bus_id:
            mine = [r for r in rows if r[1].lower().endswith(self.bus_id[-12:])]
            rows = mine or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
def algorithmic(cfg, ids_list):
    """Per-step algorithmic bytes/FLOPs averaged over the batches' routings."""
    import numpy as np
    w13 = 2 * cfg.I * cfg.H * 9 // 16     # packed e2m1 + one E4M3 per 16
    w2 = cfg.H * cfg.I * 9 // 16
    rows = cfg.T * cfg.k + cfg.T
    touched = [len(np.unique(ids)) + 1 for ids in ids_list]  # + shared expert
    t = statistics.mean(touched)
    act = 2 if cfg.mode == "w4a16" else 2  # bf16 x in, bf16 out
    gemm1_bytes = t * w13 + cfg.T * cfg.H * act + rows * cfg.I * 2
    layer_bytes = t * (w13 + w2) + cfg.T * cfg.H * 2 + cfg.T * cfg.E * 4 + cfg.T * cfg.H * 2
    gemm1_flops = rows * 2 * (2 * cfg.I) * cfg.H
    layer_flops = rows * 6 * cfg.H * cfg.I
    return {"touched_experts": t, "gemm1_bytes": gemm1_bytes, "layer_bytes": layer_bytes,
            "gemm1_flops": gemm1_flops, "layer_flops": layer_flops, "w13_bytes": w13, "w2_bytes": w2}


def ncu_traffic(workload_key):
    """DRAM bytes per launch of the reported kernel from the committed ncu
    summary (profiles/ncu_traffic.json), or None when there is none for this
    workload or the kernel's sources changed since the capture."""
    import hashlib
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "ncu_traffic.json")
    try:
        rec = json.load(open(path))[workload_key]
        h = hashlib.sha256()
        root = os.path.dirname(path)
        for f in rec["sources"]:
            h.update(open(os.path.join(root, "..", f), "rb").read())
        return rec["bytes"] if h.hexdigest() == rec["sources_sha256"] else None
    except (OSError, KeyError, ValueError):
        return None


def max_over_ranks(v, dist, device):
    """The largest of every rank's ``v`` (the job's step time is its slowest
    rank's); identity without a process group."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(v)
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, ms_per_step):
    """Whole-job throughput: every rank processes its own batch of tokens."""
    return tokens_per_rank * world / (ms_per_step / 1e3)


def config_dict(cfg, nb, flush):
    return {"workload": f"{cfg.name}: T={cfg.T} H={cfg.H} I={cfg.I} I_shared={cfg.I_s} E={cfg.E} k={cfg.k} "
                        f"{cfg.mode.upper()} +1 shared expert",
            "T": cfg.T, "H": cfg.H, "I": cfg.I, "E": cfg.E, "k": cfg.k, "mode": cfg.mode,
            "batches": nb, "l2": flush, "weights": "seeded N(0,0.02) bf16 -> NVFP4 (g16, E4M3, fp32 gs)"}


# ---------------------------------------------------------------------------
def oracle_prepare(cfg, x, logits, n_rows, pool_threads=8):
    """The (token, expert) rows of one batch in order (each token's routed
    slots by rank, then its shared-expert row), the first ``n_rows`` of them,
    and the oracle's NVFP4 weights of the experts they touch (quantised by the
    oracle, untimed)."""
    from concurrent.futures import ThreadPoolExecutor

    import synthetic_inputs as si
    from oracle import moe as omoe

    ids, w = omoe.route(logits.numpy(), cfg.k)
    plan = []
    for t in range(cfg.T):
        for j in range(cfg.k):
            plan.append((t, int(ids[t, j]), float(w[t, j])))
        plan.append((t, cfg.E, 1.0))
    plan = plan[:n_rows]

    def prep(e):
        mats = [si.make_expert_weight(cfg, e, m) for m in ("gate", "up", "down")]
        return e, tuple(omoe.QuantWeight.from_dense(m.float().numpy()) for m in mats)

    with ThreadPoolExecutor(pool_threads) as ex:
        qw = dict(ex.map(prep, sorted({e for _, e, _ in plan})))
    return plan, qw, x.float().numpy()


def oracle_rows(plan, qw, xs, out):
    """Runs the oracle (float64) on the given rows, accumulating into ``out``.
    Returns (wall seconds, process CPU seconds)."""
    from oracle import moe as omoe
    c0, t0 = time.process_time(), time.perf_counter()
    for t, e, wt in plan:
        g, u, d = qw[e]
        out[t] += wt * omoe.down_proj(omoe.gate_up_swiglu(xs[t:t + 1], g, u), d)[0]
    return time.perf_counter() - t0, time.process_time() - c0


def oracle_rows_w4a4(plan, qw, xs, gs_x, out):
    """W4A4 rows through the oracle: x quantised with the tensor's global
    scale, h rounded to bf16 and quantised (one global scale over the sampled
    rows), down GEMM. Returns (wall seconds, process CPU seconds)."""
    import numpy as np
    from oracle import moe as omoe
    from oracle import nvfp4 as onv
    c0, t0 = time.process_time(), time.perf_counter()
    hs = []
    for t, e, wt in plan:
        g, u, d = qw[e]
        xq, xsf, _ = onv.quantize(xs[t:t + 1], gs=gs_x)
        hs.append(omoe.bf16_round(omoe.gate_up_swiglu(onv.dequantize(xq, xsf, gs_x), g, u)))
    gs_h = onv.global_scale(np.float32(max(float(np.abs(h).max()) for h in hs)))
    for (t, e, wt), h in zip(plan, hs):
        hq, hsf, _ = onv.quantize(h.astype(np.float32), gs=gs_h)
        out[t] += wt * omoe.down_proj(onv.dequantize(hq, hsf, gs_h), qw[e][2])[0]
    return time.perf_counter() - t0, time.process_time() - c0


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np

    import synthetic_inputs as si
    cfg = workload(args)
    x = si.make_x(cfg)
    logits = si.make_logits(cfg)
    rows_per_token = cfg.k + 1
    all_rows = cfg.T * rows_per_token
    steps = args.warmup + args.steps
    plan, qw, xs = oracle_prepare(cfg, x, logits, min(all_rows, max(steps, rows_per_token)), pool_threads=16)
    out = np.zeros((cfg.T, cfg.H))
    est, _ = oracle_rows(plan[:1], qw, xs, out)
    # whole tokens per step if that keeps the run short, else one row per step
    per_step = rows_per_token if steps * est * rows_per_token < 150 else 1
    if per_step > 1:
        plan, qw, xs = oracle_prepare(cfg, x, logits, all_rows, pool_threads=16)
    wall = cpu = 0.0
    rows = 0
    for i in range(steps):
        sel = [plan[(i * per_step + r) % len(plan)] for r in range(per_step)]
        w_, c_ = oracle_rows(sel, qw, xs, out)
        if i >= args.warmup:
            wall += w_
            cpu += c_
            rows += len(sel)
    tokens = rows / rows_per_token
    value = tokens / wall
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(cfg, 1, "n/a (CPU)"),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": round(cpu / wall, 2),
                             "kind": "oracle",
                             "sample": f"{per_step} (token, expert) row(s) per step of the {cfg.name} batch "
                                       f"({rows} rows = {tokens:.2f} tokens timed); oracle weights "
                                       f"quantised untimed"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def workload(args):
    import synthetic_inputs as si
    cfg = si.CONFIGS[args.config]
    if args.tokens is not None or args.experts is not None:
        T = cfg.T if args.tokens is None else args.tokens
        E = cfg.E if args.experts is None else args.experts
        cfg = si.LayerConfig(f"{cfg.name}_T{T}_E{E}", T, cfg.H, cfg.I, cfg.I_s, E, cfg.k, cfg.mode, cfg.logits,
                             cfg.outliers, cfg.seed)
    return cfg


def build_layer(cfg, dev):
    """A device layer with every expert of the workload prepared (seeded weights)."""
    import torch

    import synthetic_inputs as si
    from nvfp4_mixture_experts_moe_gb300 import MOE_MXFP4, MOE_W4A4, MOE_W4A16, Nvfp4MoeLayer
    mode = {"w4a4": MOE_W4A4, "mxfp4": MOE_MXFP4}.get(cfg.mode, MOE_W4A16)
    layer = Nvfp4MoeLayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, mode=mode, I_shared=cfg.I_s, device=dev)
    for e0 in range(0, cfg.E + 1, 32):
        W = si.make_layer_weights(cfg, experts=list(range(e0, min(cfg.E + 1, e0 + 32))), threads=16)
        for e, mats in W.items():
            layer.set_expert(e, *mats)
        del W
    torch.cuda.synchronize()
    return layer


def decode_fused(cfg):
    """The forward runs this workload as the single-kernel decode path."""
    return cfg.mode == "w4a16" and cfg.T <= 8


def cpu_baseline(cfg, x0, l0, n_tokens):
    """The float64 oracle on the first ``n_tokens`` tokens of a batch, timed on
    the host cores (weights quantised by the oracle beforehand, untimed)."""
    import numpy as np
    from oracle import nvfp4 as onv
    n_rows = min(cfg.T, n_tokens) * (cfg.k + 1)
    plan, qw, xs = oracle_prepare(cfg, x0, l0, n_rows, pool_threads=16)
    if cfg.mode == "w4a4":
        wall, cpu = oracle_rows_w4a4(plan, qw, xs, onv.global_scale(np.float32(np.abs(xs).max())),
                                     np.zeros((cfg.T, cfg.H)))
        how = ("x rows quantised with the tensor's global scale, h of the sampled rows with the "
               "sample's own global scale")
    else:
        wall, cpu = oracle_rows(plan, qw, xs, np.zeros((cfg.T, cfg.H)))
        how = "W4A16"
    rows = len(plan)
    return {"value": rows / (cfg.k + 1) / wall, "unit": "tokens/s", "cores": round(cpu / wall, 2),
            "kind": "oracle",
            "sample": f"first {rows} (token, expert) rows = {rows / (cfg.k + 1):.0f} token(s) of batch 0 through "
                      f"the float64 oracle ({how}); weights prepared untimed"}


def measure(cfg, layer, args, dev, dist, world, rank, headline):
    """Times the forward on ``cfg`` (K steps after W warm-up steps, L2 flushed
    between steps) and returns the fields of a result line. ``headline`` adds
    the clock record, CUDA-graph replay and the router GEMM."""
    import numpy as np
    import torch

    import synthetic_inputs as si
    from nvfp4_mixture_experts_moe_gb300 import binding as B

    nb = max(1, args.batches)
    batches = []
    for b in range(nb):
        c = si.LayerConfig(cfg.name, cfg.T, cfg.H, cfg.I, cfg.I_s, cfg.E, cfg.k, cfg.mode, cfg.logits,
                           cfg.outliers, seed=cfg.seed + 1000 * b + rank)
        batches.append((si.make_x(c).to(dev), si.make_logits(c).to(dev)))
    ids_list = [__import__("oracle").moe.route(lg.cpu().numpy(), cfg.k)[0] for _, lg in batches]
    alg = algorithmic(cfg, ids_list)

    ws = layer.workspace(cfg.T)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    desc = layer.desc(cfg.T)

    def step(i, stage_events=None):
        x, lg = batches[i % nb]
        if stage_events is not None:
            B.moe_set_stage_events(stage_events)
        B.moe_nvfp4_forward(desc, x, lg, out, None, ws, stream)

    for i in range(args.warmup):
        flush.zero_()
        step(i)
    torch.cuda.synchronize()
    if B.moe_get_device_status(ws) != 0:
        raise RuntimeError(f"{cfg.name}: device status set during warm-up")

    K = args.steps
    # Pass 1 (the measurement): K steps, one event pair per step, nothing else
    # inside the forward. Pass 2: the same K steps with the library recording
    # an event between every stage, for the per-kernel durations.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(B.MOE_STAGE_COUNT)] for _ in range(K)]
    for e in [x for pair in ev for x in pair] + [x for row in sev for x in row]:
        e.record(stream)  # torch creates the underlying CUDA events on first record
    torch.cuda.synchronize()
    sampler = None
    if headline:
        props = torch.cuda.get_device_properties(dev)
        bus = getattr(props, "pci_bus_id", None)
        sampler = ClockSampler(bus if isinstance(bus, str) else None)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
        time.sleep(0.2)
    launches0 = B.moe_kernel_launches()
    t0 = time.perf_counter()
    for i in range(K):
        flush.zero_()  # L2 flush between steps, outside the timed events
        ev[i][0].record(stream)
        step(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    launches = B.moe_kernel_launches() - launches0
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    step_ms = [a.elapsed_time(b) for a, b in ev]
    for i in range(K):
        flush.zero_()
        step(i, sev[i])
    torch.cuda.synchronize()
    stage_ms = [[e[s].elapsed_time(e[s + 1]) for e in sev] for s in range(B.MOE_STAGE_COUNT - 1)]
    staged_step_ms = statistics.mean(e[0].elapsed_time(e[-1]) for e in sev)
    ms = max_over_ranks(statistics.mean(step_ms), dist, dev)
    if B.moe_get_device_status(ws) != 0:
        raise RuntimeError(f"{cfg.name}: device status set during the timed steps")
    value = job_tokens_per_s(cfg.T, world, ms)

    # end to end: pinned host inputs copied in (x and the logits packed in one
    # pinned buffer, one copy), result read back, every step
    xb = batches[0][0].numel() * batches[0][0].element_size()
    lb = batches[0][1].numel() * batches[0][1].element_size()
    loff = (xb + 255) // 256 * 256
    hbuf = []
    for bx, bl in batches:
        hb = torch.empty(loff + lb, dtype=torch.uint8).pin_memory()
        hb[:xb].view(bx.dtype).view(bx.shape).copy_(bx.cpu())
        hb[loff:].view(bl.dtype).view(bl.shape).copy_(bl.cpu())
        hbuf.append(hb)
    hout = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16).pin_memory()
    dbuf = torch.empty(loff + lb, dtype=torch.uint8, device=dev)
    dx = dbuf[:xb].view(batches[0][0].dtype).view(batches[0][0].shape)
    dl = dbuf[loff:].view(batches[0][1].dtype).view(batches[0][1].shape)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(args.warmup + K):
        flush.zero_()
        if i >= args.warmup:
            e2e_ev[i - args.warmup][0].record(stream)
        dbuf.copy_(hbuf[i % nb], non_blocking=True)
        B.moe_nvfp4_forward(desc, dx, dl, out, None, ws, stream)
        hout.copy_(out, non_blocking=True)
        if i >= args.warmup:
            e2e_ev[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    if not torch.equal(hout.to(dev), out):
        raise RuntimeError(f"{cfg.name}: end-to-end output differs from the device output")
    e2e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in e2e_ev), dist, dev)
    h2d = loff + lb
    d2h = hout.numel() * hout.element_size()

    pk = peaks()
    per_stage = {name: statistics.mean(stage_ms[i]) for i, name in enumerate(B.STAGES)}
    if decode_fused(cfg):
        # one kernel is the whole layer: its roofline is the layer's bytes
        k_ms = per_stage["route"]
        bound, unit, peak = "hbm", "GB/s", pk["hbm"]
        achieved = alg["layer_bytes"] / (k_ms / 1e3) / 1e9
        kernel = "decode_fused_kernel (whole layer: route, permute, gate/up GEMM + SwiGLU, down GEMM, combine)"
        traffic = ncu_traffic(cfg.name)
        per_unit = "touched experts x (W13 + W2 NVFP4 bytes) + x in + out + logits"
    else:
        k_ms = per_stage["gemm1_gate_up_swiglu"]
        kernel = "gemm1 (gate/up grouped GEMM + SwiGLU epilogue)"
        if cfg.mode == "w4a16" and cfg.T <= 64:
            bound, unit, peak = "hbm", "GB/s", pk["hbm"]
            achieved = alg["gemm1_bytes"] / (k_ms / 1e3) / 1e9
            per_unit = "touched experts x W13 NVFP4 bytes + x rows in + h out"
        else:
            bound, unit = "tensor", "TFLOP/s"
            achieved = alg["gemm1_flops"] / (k_ms / 1e3) / 1e12
            peak = pk["bf16"] * (6.0 if cfg.mode == "w4a4" else 1.0)
            per_unit = "rows x 2 x 2I x H FLOPs"
        traffic = ncu_traffic(cfg.name)
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": traffic, "kernel": kernel, "kernel_ms": k_ms, "per_launch": per_unit,
                "peak_source": pk["source"] + (" (fp4 = 6 x measured bf16, the nominal ratio)"
                                               if cfg.mode == "w4a4" and bound == "tensor" else "")}
    layer_time_hbm = alg["layer_bytes"] / (pk["hbm"] * 1e9)
    tc_peak = pk["bf16"] * (6.0 if cfg.mode == "w4a4" else 1.0)
    layer_time_tc = alg["layer_flops"] / (tc_peak * 1e12)
    layer_roof_ms = 1e3 * max(layer_time_hbm, layer_time_tc)
    res = {"ms_per_step": ms, "value": value, "unit": "tokens/s",
           "config": config_dict(cfg, nb, "flushed: 258 MB write between timed steps"),
           "roofline": roofline,
           "layer_roofline": {"roofline_ms": layer_roof_ms, "frac": layer_roof_ms / ms,
                              "bound": "hbm" if layer_time_hbm >= layer_time_tc else "tensor",
                              "bytes": alg["layer_bytes"], "flops": alg["layer_flops"],
                              "touched_experts": alg["touched_experts"]},
           "stages_ms": per_stage,
           "stages_note": ("single-kernel decode path: 'route' is the whole fused kernel"
                           if decode_fused(cfg) else
                           "per-stage CUDA events recorded by the library in a second pass of the same K steps")
                          + f" (that pass: {staged_step_ms:.4f} ms/step, stages serialised)",
           "e2e": {"value": job_tokens_per_s(cfg.T, world, e2e_ms), "unit": "tokens/s", "ms_per_step": e2e_ms,
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
           "gpu_launches": int(launches), "host_wall_s": t1 - t0}
    if clocks is not None:
        res["clocks"] = clocks
    if headline:
        res["graph_replay"] = graph_replay(desc, batches, out, ws, flush, stream, args, dist, dev, world, cfg)
        res["router_gemm"] = router_gemm(cfg, layer, batches, out, flush, stream, args, dev, pk)
    if cfg.T > 64 and cfg.mode in ("w4a16", "w4a4") and layer.shared:
        res["public_grouped_gemm"] = public_grouped_gemm(cfg, layer, batches, flush, stream, args, dev, pk)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_tok = {"tiny": 16, "w4a4": 1}.get(cfg.name, args.cpu_sample_tokens)
        res["cpu_baseline"] = cpu_baseline(cfg, batches[0][0].cpu(), batches[0][1].cpu(), n_tok)
    return res


def graph_replay(desc, batches, out, ws, flush, stream, args, dist, dev, world, cfg):
    """The same forward captured once as a CUDA graph and replayed (batch 0's
    inputs, L2 flushed between replays outside the graph)."""
    import torch

    from nvfp4_mixture_experts_moe_gb300 import binding as B
    K = args.steps
    try:
        gx, gl = batches[0]
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                B.moe_nvfp4_forward(desc, gx, gl, out, None, ws, torch.cuda.current_stream())
        torch.cuda.synchronize()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(args.warmup + K):
            flush.zero_()
            if i >= args.warmup:
                gev[i - args.warmup][0].record(stream)
            g.replay()
            if i >= args.warmup:
                gev[i - args.warmup][1].record(stream)
        torch.cuda.synchronize()
        g_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in gev), dist, dev)
        if B.moe_get_device_status(ws) != 0:
            raise RuntimeError("device status set during graph replay")
        return {"ms_per_step": g_ms, "value": job_tokens_per_s(cfg.T, world, g_ms), "unit": "tokens/s",
                "note": "moe_nvfp4_forward captured once in a CUDA graph, replayed K times"}
    except RuntimeError as exc:  # capture not possible here: report why
        return {"error": str(exc).splitlines()[0][:200]}


def router_gemm(cfg, layer, batches, out, flush, stream, args, dev, pk):
    """The router GEMM ahead of the top-k (logits = x W_router^T) on this
    workload's shapes: alone, and inside the forward (which then takes x
    only). The measured step takes the logits as an input."""
    import torch

    import synthetic_inputs as si
    from nvfp4_mixture_experts_moe_gb300 import binding as B
    K, nb = args.steps, len(batches)
    w_router = si.make_router_weight(cfg).to(dev)
    rlog = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev)
    rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    layer.set_router(w_router)
    desc_r = layer.desc(cfg.T)
    layer.set_router(None)
    ws_r = torch.empty(B.moe_workspace_size(desc_r), dtype=torch.uint8, device=dev)
    ws_r[:256].zero_()
    for i in range(args.warmup + K):
        flush.zero_()
        if i >= args.warmup:
            rev[i - args.warmup][0].record(stream)
        B.moe_router_gemm(batches[i % nb][0], w_router, cfg.T, cfg.H, cfg.E, rlog, stream)
        if i >= args.warmup:
            rev[i - args.warmup][1].record(stream)
    for i in range(args.warmup + K):
        flush.zero_()
        if i >= args.warmup:
            fev[i - args.warmup][0].record(stream)
        B.moe_nvfp4_forward(desc_r, batches[i % nb][0], None, out, None, ws_r, stream)
        if i >= args.warmup:
            fev[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    if B.moe_get_device_status(ws_r) != 0:
        raise RuntimeError("device status set in the forward with the router GEMM")
    r_ms = statistics.mean(a.elapsed_time(b) for a, b in rev)
    fr_ms = statistics.mean(a.elapsed_time(b) for a, b in fev)
    r_bytes = cfg.E * cfg.H * 2 + cfg.T * cfg.H * 2 + cfg.T * cfg.E * 4
    r_flops = 2 * cfg.T * cfg.H * cfg.E
    if cfg.T <= 16:
        r_roof = {"bound": "hbm", "unit": "GB/s", "achieved": r_bytes / (r_ms / 1e3) / 1e9, "peak": pk["hbm"],
                  "kernel": "router_gemv_kernel"}
    else:
        r_roof = {"bound": "tensor", "unit": "TFLOP/s", "achieved": r_flops / (r_ms / 1e3) / 1e12,
                  "peak": pk["bf16"], "kernel": "router_tc_kernel (tcgen05 kind::f16, bf16)"}
    r_roof["frac"] = r_roof["achieved"] / r_roof["peak"]
    return dict(ms=r_ms, bytes=r_bytes, flops=r_flops, **r_roof, forward_with_router_ms=fr_ms,
                note="logits = x W_router^T (bf16 [E, H] router, seeded N(0, 1/H)); timed alone and inside "
                     "moe_nvfp4_forward (x only), L2 flushed between launches")


def public_grouped_gemm(cfg, layer, batches, flush, stream, args, dev, pk):
    """The public grouped GEMM entry point (moe_nvfp4_grouped_gemm) on this
    workload's gate/up GEMM: the same routed and shared rows, the activations
    row-major with a row index (W4A4: quantised by moe_nvfp4_quantize), timed
    alone with L2 flushed between launches. The forward runs its own GEMM
    kernels on activations it has put in group order."""
    import torch

    from nvfp4_mixture_experts_moe_gb300 import binding as B
    K, k, T, E = args.steps, cfg.k, cfg.T, cfg.E
    x, logits = batches[0]
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    B.moe_route_topk(logits, T, E, k, ids, w, stream)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    inv = torch.empty(T * k, dtype=torch.int32, device=dev)
    pws = torch.zeros(B.moe_permute_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    B.moe_permute(ids, T, k, E, counts, offsets, perm, inv, pws, stream)
    torch.cuda.synchronize()
    # groups: the E routed experts, then the shared expert's T rows
    offs = torch.cat([offsets, torch.tensor([T * k + T], dtype=torch.int32, device=dev)])
    row_tok = torch.cat([(perm.long() // k).to(torch.int32), torch.arange(T, dtype=torch.int32, device=dev)])
    rows = T * k + T
    h = torch.empty(rows, cfg.I, dtype=torch.bfloat16, device=dev)
    w4a4 = cfg.mode == "w4a4"
    args_g = B.MoeGemmArgs(mode=1 if w4a4 else 0, gate_up=1, num_groups=E + 1, N=2 * cfg.I, K=cfg.H)
    args_g.weights = layer.w13.data_ptr()
    args_g.last_weights = layer.w13_s.data_ptr()
    args_g.group_offsets = offs.data_ptr()
    args_g.a_row_index = row_tok.data_ptr()
    args_g.out = h.data_ptr()
    args_g.rows = rows   # the row count and room for the copies select the forward's kernels
    if w4a4:
        from nvfp4_mixture_experts_moe_gb300 import quantize_bf16
        q, sf, gs = quantize_bf16(x)
        keep = (q, sf, gs)
        args_g.a, args_g.a_sf, args_g.a_gs = q.data_ptr(), sf.data_ptr(), gs.data_ptr()
    else:
        keep = (x,)
        args_g.a = x.data_ptr()
    gws = torch.zeros(B.moe_gemm_workspace_size_rows(E + 1, rows, cfg.H), dtype=torch.uint8, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(args.warmup + K):
        flush.zero_()
        if i >= args.warmup:
            ev[i - args.warmup][0].record(stream)
        B.moe_nvfp4_grouped_gemm(args_g, gws, stream)
        if i >= args.warmup:
            ev[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    del keep
    if B.moe_get_device_status(gws) != 0:
        raise RuntimeError("device status set in the public grouped GEMM")
    g_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    flops = rows * 2 * (2 * cfg.I) * cfg.H
    peak = pk["bf16"] * (6.0 if w4a4 else 1.0)
    achieved = flops / (g_ms / 1e3) / 1e12
    return {"ms": g_ms, "flops": flops, "achieved": achieved, "unit": "TFLOP/s", "peak": peak,
            "frac": achieved / peak,
            "kernel": "tile_gather_kernel + gemm_tc_fp4_wide_kernel" if w4a4 else
                      "rows_to_f16_kernel + gemm_small_kernel + gemm_tc_f16_kernel (128- and 256-row tiles)",
            "note": "moe_nvfp4_grouped_gemm, gate/up + SwiGLU, the workload's routed and shared rows, "
                    "activations row-major with a row index (row count given: the copy of the rows into "
                    "group order is made inside the call and timed); L2 flushed between launches"}


def run_ours(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import synthetic_inputs as si

    cfg = workload(args)
    t_setup = time.perf_counter()
    layer = build_layer(cfg, dev)
    setup_s = time.perf_counter() - t_setup
    res = measure(cfg, layer, args, dev, dist, world, rank, headline=True)
    line = {"metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp4xf16" if cfg.mode == "w4a16" else "fp4",
            "data": "synthetic"}
    line.update({k: v for k, v in res.items() if k not in ("value", "ms_per_step", "unit")})
    line["setup_s"] = setup_s

    # every other workload in the same process (one GPU only): its own step
    # time, roofline, end-to-end number and CPU baseline
    if world == 1 and not args.only and args.tokens is None and args.experts is None:
        configs = {}
        same_layer = (cfg.H, cfg.I, cfg.I_s, cfg.E, cfg.k, cfg.mode, cfg.seed)
        for name, c in si.CONFIGS.items():
            if name == cfg.name:
                continue
            if (c.H, c.I, c.I_s, c.E, c.k, c.mode, c.seed) != same_layer:
                del layer
                torch.cuda.empty_cache()
                t_setup = time.perf_counter()
                layer = build_layer(c, dev)
                same_layer = (c.H, c.I, c.I_s, c.E, c.k, c.mode, c.seed)
                setup = time.perf_counter() - t_setup
            else:
                setup = 0.0
            r = measure(c, layer, args, dev, None, 1, 0, headline=False)
            r["setup_s"] = setup
            configs[name] = r
        line["configs"] = configs

    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
