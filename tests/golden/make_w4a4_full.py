"""Writes ``w4a4_full_tokens.npz``: oracle outputs of the full-size W4A4 workload.

The W4A4 workload (16384 tokens, hidden 7168, expert intermediate 2048, 256
routed experts top-8 + 1 shared expert, activations with 0.1% outliers x20)
quantises the SwiGLU output ``h`` of *all* 147,456 grouped rows with one
dynamic global scale, so no single token's output can be computed without
first running the gate/up GEMM and SwiGLU over every row. This script does
that once, on the CPU, with the oracle only (``oracle/`` and the seeded
generators in ``synthetic_inputs``; nothing from the CUDA path), and stores:

* ``gs_x``: the dynamic global scale of X (2688 / amax over the whole tensor);
* ``amax_h``, ``gs_h``: the amax of the bf16-rounded h over all rows and its
  global scale;
* ``tokens``: 64 token indices spread over the batch, with their routing
  (``ids``, ``w``) and their float64 layer outputs ``out`` stored as float32;
* ``flip``: per output element of those tokens, how far FP4 re-quantisation
  of h can move it when h is computed in fp32 (``oracle.moe.requant_flip_bound``
  with the window ``oracle.moe.gate_up_window``, the fp32 summation bound of
  the gate/up GEMM): a GPU computes h in another summation order, so an h
  element lying within that window of a bf16 rounding midpoint may round the
  other way, and where the bf16 values quantise to different FP4 codes (or
  block scales) the token's whole output row moves by the FP4 steps times
  the down-projection column.

Given ``gs_x`` and ``gs_h`` every token's output depends on that token alone,
so the stored rows are exactly the rows of ``oracle.moe.layer(..., mode="w4a4")``
for these tokens: X is quantised with ``gs_x`` and dequantised; each of the
token's k routed experts and the shared expert computes h, h is rounded to
bf16, quantised with ``gs_h`` (the oracle quantiser with a given scale, whose
equality with the dynamic path at the same scale is pinned by the oracle
tests), dequantised and multiplied by the down matrix; the routed rows are
weighted by the renormalised router probabilities and summed in slot order,
then the shared expert's row is added.

Run from the repository root (about 10 minutes on 8 cores, ~20 GB of RAM):

    python tests/golden/make_w4a4_full.py
"""
from __future__ import annotations

import os
import sys
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synthetic_inputs as si  # noqa: E402
from oracle import moe as omoe  # noqa: E402
from oracle import nvfp4 as onv  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "w4a4_full_tokens.npz")
N_TOKENS = 64


def sample_tokens(T, n):
    """n token indices spread over [0, T): the two ends plus a seeded draw."""
    rng = np.random.default_rng(20260)
    mid = rng.choice(np.arange(1, T - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, T - 1], mid])).astype(np.int64)


def golden_rows(cfg, tokens, threads=8, log=print):
    """Oracle outputs ``[len(tokens), H]`` (float64) of the W4A4 layer ``cfg``
    for the given tokens, with the scales: returns (out, gs_x, amax_h, gs_h,
    ids, w, flip) where ids/w are the whole batch's routing and flip the
    re-quantisation allowance of the tokens' outputs."""
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    t0 = time.time()
    x = si.make_x(cfg).float().numpy()
    logits = si.make_logits(cfg).numpy()
    ids, w = omoe.route(logits, k)
    counts, offsets, perm, inv_perm = omoe.permute(ids, E)
    xq, xsf, gs_x = onv.quantize(x)
    x_deq = onv.dequantize(xq, xsf, gs_x)
    del xq, xsf
    want = set(int(t) for t in tokens)
    log(f"inputs, route, X quantised: {time.time() - t0:.0f} s; gs_x = {gs_x!r}")

    def expert(e):
        mats = [si.make_expert_weight(cfg, e, m).float().numpy() for m in ("gate", "up", "down")]
        gq, uq, dq = (omoe.QuantWeight.from_dense(m) for m in mats)
        toks = np.arange(T) if e == E else perm[offsets[e]:offsets[e + 1]] // k
        amax = 0.0
        sampled = {}
        for c0 in range(0, len(toks), 2048):  # bounded memory for the shared expert's 16384 rows
            tk = toks[c0:c0 + 2048]
            h_exact = omoe.gate_up_swiglu(x_deq[tk], gq, uq)
            h = omoe.bf16_round(h_exact)
            if h.size:
                amax = max(amax, float(np.max(np.abs(h))))
            pick = [i for i, t in enumerate(tk) if int(t) in want]
            if pick:
                win = omoe.gate_up_window(x_deq[tk[pick]], gq, uq)
                for n, i in enumerate(pick):
                    sampled[int(tk[i])] = (h[i].copy(), h_exact[i].copy(), win[n])
        return e, amax, sampled, (dq if sampled else None)

    amax_h = 0.0
    h_rows = {}        # (token, expert) -> (bf16-rounded h row, float64 h row, fp32 window)
    downs = {}
    done = 0
    with ThreadPoolExecutor(threads) as ex:
        for e, amax, sampled, dq in ex.map(expert, range(E + 1)):
            amax_h = max(amax_h, amax)
            for t, h in sampled.items():
                h_rows[(t, e)] = h
            if dq is not None:
                downs[e] = dq
            done += 1
            if done % 16 == 0:
                log(f"  {done}/{E + 1} experts, {time.time() - t0:.0f} s")
    gs_h = onv.global_scale(np.float32(amax_h))
    log(f"gate/up + SwiGLU over all rows: {time.time() - t0:.0f} s; amax_h = {amax_h!r}, gs_h = {gs_h!r}")

    def y_of(t, e):
        h = h_rows[(t, e)][0][None, :].astype(np.float32)
        hq, hsf, _ = onv.quantize(h, gs=gs_h)
        return omoe.down_proj(onv.dequantize(hq, hsf, gs_h), downs[e])[0]

    down_abs = {}

    def flip_of(t, e):
        if e not in down_abs:
            down_abs[e] = np.abs(downs[e].dequantize())
        return omoe.requant_flip_bound(h_rows[(t, e)][1], gs_h, down_abs[e], h_rows[(t, e)][2])

    out = np.zeros((len(tokens), H), dtype=np.float64)
    flip = np.zeros((len(tokens), H), dtype=np.float64)
    for i, t in enumerate(tokens):
        for j in range(k):
            out[i] += np.float64(w[t, j]) * y_of(int(t), int(ids[t, j]))
            flip[i] += np.float64(w[t, j]) * flip_of(int(t), int(ids[t, j]))
        out[i] += y_of(int(t), E)
        flip[i] += flip_of(int(t), E)
    return out, gs_x, np.float32(amax_h), gs_h, ids, w, flip


def main(threads=8):
    cfg = si.CONFIGS["w4a4"]
    t0 = time.time()
    tokens = sample_tokens(cfg.T, N_TOKENS)
    out, gs_x, amax_h, gs_h, ids, w, flip = golden_rows(cfg, tokens, threads,
                                                        log=lambda m: print(m, flush=True))
    np.savez_compressed(OUT, tokens=tokens, out=out.astype(np.float32), ids=ids[tokens], w=w[tokens],
                        gs_x=np.float32(gs_x), amax_h=np.float32(amax_h), gs_h=np.float32(gs_h),
                        flip=flip.astype(np.float32))
    print(f"wrote {OUT} ({os.path.getsize(OUT)} bytes) in {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main()
