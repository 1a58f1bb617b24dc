"""The fused NVFP4 MoE layer, step by step, in float64 on the CPU.

Test infrastructure only (see the package docstring for who may import it).

Steps follow "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide",
section 7.1 (router -> quantise/dispatch -> permute, experts, unpermute ->
combine) and section 4.3 (dispatch, two GEMMs with SwiGLU between them, top-k
weight reduction; BF16 input quantised to FP4 on the W4A4 path), with one
shared expert that every token uses ("Serving Solar Open 2 on DGX Spark",
"Solar Open 2 in brief").

Readings adopted where the pages are silent:

* the router's logits are an input; softmax over all routed experts, top-k by
  logit (ties to the lower expert index), weights renormalised over the k;
* the shared expert's output is added with weight 1 and no gate;
* each expert's gate, up and down matrices carry their own global scale;
* ``h = silu(g) * u`` with ``silu(z) = z / (1 + exp(-z))``;
* W4A4: X is quantised with one global scale over the whole ``[T, H]``
  tensor; h is rounded to bf16 (the activation precision) and quantised with
  one global scale over all rows (routed pairs and shared rows together).
"""
from __future__ import annotations

import numpy as np

from . import mxfp4, nvfp4

F32 = np.float32


def bf16_round(x):
    """float -> nearest bf16 value (ties to even), returned as float32.

    bf16 keeps the top 16 bits of an fp32; rounding adds half of the dropped
    part with the tie going to an even kept part. Pinned by: torch's bf16
    conversion (tests).
    """
    f = np.asarray(x, dtype=np.float64).astype(F32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) >> 16 << 16
    out = u.astype(np.uint32).view(F32)
    return np.where(np.isnan(f), f, out)


def route(logits, k):
    """Router: softmax over experts, top-k, renormalised weights.

    ``logits`` ``[T, E]`` fp32 -> ``(ids [T, k] int32, w [T, k] fp32)``. The k
    slots are ordered by rank: higher logit first, equal logits (including
    -0 and +0) by lower expert index. The weights are the softmax
    probabilities of the chosen experts divided by their sum, computed in
    float64 and stored as fp32.
    Pinned by: brute-force selection on tiny inputs; weights summing to 1;
    constructed ties; k = E returning every expert in rank order.
    """
    logits = np.asarray(logits, dtype=F32)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    l64 = logits.astype(np.float64)
    p = np.exp(l64 - l64.max(axis=1, keepdims=True))
    p = p / p.sum(axis=1, keepdims=True)
    # Stable sort on the negated logit keeps ascending expert order among ties.
    order = np.argsort(-l64, axis=1, kind="stable")
    ids = order[:, :k]
    pk = np.take_along_axis(p, ids, axis=1)
    w = pk / pk.sum(axis=1, keepdims=True)
    return ids.astype(np.int32), w.astype(F32)


def permute(ids, E):
    """Group the T*k (token, slot) pairs by expert with a stable counting sort.

    Pair ``p = t*k + j`` goes to expert ``ids[t, j]``. Returns
    ``counts [E]``, ``offsets [E+1]`` (exclusive prefix sum, ``offsets[E] =
    T*k``), ``perm [T*k]`` (sorted position -> pair) and ``inv_perm [T*k]``
    (pair -> sorted position). Inside an expert's group pairs keep ascending
    ``p``. The shared expert's rows follow at ``T*k .. T*k + T - 1`` in token
    order and are not listed.
    Pinned by: inv_perm(perm) = identity, counts summing to T*k, offsets as
    the exclusive scan, and stability against Python's sorted().
    """
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    P = ids.size
    if P and (ids.min() < 0 or ids.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.zeros(E, dtype=np.int64)
    for e in ids:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    cursor = offsets[:-1].copy()
    perm = np.empty(P, dtype=np.int64)
    inv_perm = np.empty(P, dtype=np.int64)
    for p in range(P):
        e = ids[p]
        perm[cursor[e]] = p
        inv_perm[p] = cursor[e]
        cursor[e] += 1
    return (counts.astype(np.int32), offsets.astype(np.int32),
            perm.astype(np.int32), inv_perm.astype(np.int32))


def silu(z):
    """SiLU, ``z / (1 + exp(-z))``, float64. Pinned by: torch's silu (tests)."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


class QuantWeight:
    """One NVFP4 weight matrix ``[N, K]``: unpacked codes, E4M3 scales, gs."""

    def __init__(self, codes, sf, gs):
        self.codes = np.asarray(codes, dtype=np.uint8)
        self.sf = np.asarray(sf, dtype=np.uint8)
        self.gs = F32(gs)

    @classmethod
    def from_dense(cls, w):
        return cls(*nvfp4.quantize(np.asarray(w, dtype=F32)))

    def dequantize(self):
        return nvfp4.dequantize(self.codes, self.sf, self.gs)


class QuantWeightMX:
    """One MXFP4 weight matrix ``[N, K]``: unpacked e2m1 codes and E8M0 scale
    codes (one per 32 along K); no per-tensor global scale ("vLLM on the
    NVIDIA DGX Spark", section 6.4 "NVFP4 vs MXFP4")."""

    def __init__(self, codes, sc):
        self.codes = np.asarray(codes, dtype=np.uint8)
        self.sc = np.asarray(sc, dtype=np.uint8)

    @classmethod
    def from_dense(cls, w):
        return cls(*mxfp4.quantize(np.asarray(w, dtype=F32)))

    def dequantize(self):
        return mxfp4.dequantize(self.codes, self.sc)


def gate_up_swiglu(x_rows, gate, up):
    """First GEMM pair and SwiGLU on a block of rows: ``h = silu(x Wg^T) * (x Wu^T)``.

    ``x_rows`` are float64 rows already in the GEMM's input precision (bf16
    values on W4A16, dequantised NVFP4 on W4A4); ``gate``/``up`` are
    ``QuantWeight``. Returns ``h`` float64.
    Pinned by: the dense one-expert reduction against torch.matmul and
    torch's silu; brute force on tiny sizes (tests).
    """
    g = x_rows @ gate.dequantize().T
    u = x_rows @ up.dequantize().T
    return silu(g) * u


def down_proj(h_rows, down):
    """Second GEMM: ``y = h Wd^T`` in float64."""
    return h_rows @ down.dequantize().T


def router_logits(x, w_router):
    """Router GEMM: ``logits = x W_router^T`` in float64.

    ``x`` ``[T, H]`` and ``w_router`` ``[E, H]`` hold bf16 values (exact in
    float64). The pages name the router as the step ahead of top-k ("vLLM on
    the NVIDIA DGX Spark", section 7.1, [Router]); the router matrix stays in
    16-bit, outside the NVFP4 expert weights.
    Pinned by: exact rational dot products (fractions) on tiny sizes; one-hot
    router rows that pick out a scaled column of x exactly (tests).
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w_router, dtype=np.float64)
    return x @ w.T


def layer(x, logits, experts, shared, k, mode="w4a16", return_parts=False, x_gs=None, h_gs=None,
          experts_range=None):
    """The whole layer for ``T`` tokens, float64.

    ``x`` ``[T, H]`` (bf16 values), ``logits`` ``[T, E]`` fp32, ``experts`` a
    list of E ``(gate, up, down)`` QuantWeight triples, ``shared`` one triple
    or None. Returns ``out [T, H]`` float64 (and a dict of intermediates when
    ``return_parts``):

        out[t] = sum_j w[t, j] * y[(t, j)] + y_shared[t]

    W4A16: ``x`` enters the GEMMs as is. W4A4: ``x`` is quantised (one global
    scale) and dequantised first; ``h`` is rounded to bf16, quantised over all
    rows with one global scale, and dequantised before the down GEMM. The two
    W4A4 global scales are dynamic (from the tensors' amax) unless ``x_gs`` /
    ``h_gs`` give static calibrated ones (quant convention). MXFP4 (the
    experts are ``QuantWeightMX``): as W4A4 with MXFP4 for x and h (E8M0
    scales per 32, no global scale).
    ``experts_range=(lo, hi)`` computes one shard of expert parallelism
    ("Serving Solar Open 2 on DGX Spark", "Adding Expert Parallelism to b12x":
    each node holds a contiguous shard of the experts and filters out the
    pairs of other shards): the router still ranks all E experts, only the
    pairs routed to experts lo..hi-1 are computed (W4A4: the global scale of h
    is taken over those rows and the shared rows), and the result is that
    shard's partial output (plus the shared expert when ``shared`` is given).
    Pinned by: a dense formulation (every expert on every token, weighted by a
    T x E routing matrix) on tiny sizes, the identical-experts invariant, the
    one-expert dense reduction, (static scales) the dynamic result when the
    static scales equal the dynamic ones, and (shards) the shards' partial
    outputs summing to the whole layer (tests).
    """
    x = np.asarray(x, dtype=np.float64)
    T, H = x.shape
    E = len(experts)
    ids, w = route(logits, k)
    counts, offsets, perm, inv_perm = permute(ids, E)
    parts = {"ids": ids, "w": w, "counts": counts, "offsets": offsets,
             "perm": perm, "inv_perm": inv_perm}
    if mode == "w4a4":
        xq, xsf, xgs = nvfp4.quantize(x.astype(F32), gs=x_gs)
        parts.update(xq=xq, xsf=xsf, xgs=xgs)
        x_in = nvfp4.dequantize(xq, xsf, xgs)
    elif mode == "mxfp4":
        xq, xsc = mxfp4.quantize(x.astype(F32))
        parts.update(xq=xq, xsc=xsc)
        x_in = mxfp4.dequantize(xq, xsc)
    elif mode == "w4a16":
        x_in = x
    else:
        raise ValueError(mode)
    lo, hi = (0, E) if experts_range is None else experts_range
    if not 0 <= lo <= hi <= E:
        raise ValueError("expert range outside [0, E]")
    # Rows in the order the layer lays them out: routed pairs grouped by
    # expert (sorted order; this shard's experts only), then the shared
    # expert's rows in token order.
    groups = [(experts[e], perm[offsets[e]:offsets[e + 1]] // k) for e in range(lo, hi)]
    E_local = hi - lo
    if shared is not None:
        groups.append((shared, np.arange(T)))
    hs = [gate_up_swiglu(x_in[toks], gate, up) for (gate, up, _), toks in groups]
    if mode == "w4a4":
        sizes = [h.shape[0] for h in hs]
        allh = np.concatenate(hs, axis=0)
        allh_bf = bf16_round(allh)
        hq, hsf, hgs = nvfp4.quantize(allh_bf, gs=h_gs)
        parts.update(h_bf16=allh_bf, hq=hq, hsf=hsf, hgs=hgs)
        hs = np.split(nvfp4.dequantize(hq, hsf, hgs), np.cumsum(sizes)[:-1], axis=0)
    if mode == "mxfp4":
        # h rounded to bf16, then every row quantised on its own (block scales
        # per 32; MXFP4 has no per-tensor scale)
        q = [mxfp4.quantize(bf16_round(h)) if h.shape[0] else (h, None) for h in hs]
        hs = [mxfp4.dequantize(c, sc) if sc is not None else h for (c, sc), h in zip(q, hs)]
    ys = [down_proj(h, trip[2]) for h, (trip, _) in zip(hs, groups)]
    y_routed = np.concatenate(ys[:E_local], axis=0) if E_local else np.zeros((0, H))
    out = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            if lo <= ids[t, j] < hi:
                out[t] += np.float64(w[t, j]) * y_routed[inv_perm[t * k + j] - offsets[lo]]
    if shared is not None:
        out += ys[E_local]
    parts.update(h=hs, y_routed=y_routed)
    if return_parts:
        return out, parts
    return out


#: Lipschitz constant of silu: max |silu'(z)| = 1.0998 (at z = 2.40)
SILU_LIP = 1.1


def gate_up_window(x_rows, gate, up):
    """Bound on how far an fp32 computation of ``h = silu(g) * u`` can lie
    from the float64 ``h`` of ``gate_up_swiglu`` (same inputs), per element.

    A dot product of K terms summed in fp32 in any order, with r roundings on
    the path of every term, is within ``r * 2**-24 * sum |terms|`` of the exact
    sum (the standard recursive-summation bound, first order). Reading taken
    for a block-scaled tensor-core GEMM that accumulates one 64-wide K block
    at a time into an fp32 accumulator: at most 6 roundings inside a block
    (a pairwise tree over 64 products) and one per block added, plus 2 for the
    global-scale product, so ``r = K / 64 + 8``. Then, with ``dg``, ``du``
    the bounds of g and u and silu 1.1-Lipschitz,
    ``|h' - h| <= 1.1 dg (|u| + du) + |silu(g)| du`` plus ``2**-20`` relative
    for evaluating silu and the product in fp32 (exp, a division, two
    multiplies, each a few ulps).

    ``x_rows`` float64 ``[n, K]`` (the GEMM's input values), ``gate``/``up``
    ``QuantWeight``. Returns float64 ``[n, I]``.
    Pinned by: zero for zero rows; it contains the actual error of float32
    evaluations of h in several summation orders (tests).
    """
    x = np.abs(np.asarray(x_rows, dtype=np.float64))
    K = x.shape[1]
    r = K / 64.0 + 8.0
    gd, ud = gate.dequantize(), up.dequantize()
    xr = np.asarray(x_rows, dtype=np.float64)
    g, u = xr @ gd.T, xr @ ud.T
    dg = r * 2.0 ** -24 * (x @ np.abs(gd).T)
    du = r * 2.0 ** -24 * (x @ np.abs(ud).T)
    sg = np.abs(silu(g))
    w = SILU_LIP * dg * (np.abs(u) + du) + sg * du
    return w + 2.0 ** -20 * (sg + SILU_LIP * dg) * (np.abs(u) + du)


def _bf16_values_between(lo, hi):
    """All bf16 values v with lo <= v <= hi (lo, hi bf16 values, lo <= hi)."""
    def key(v):  # monotone integer key of a bf16 value (sign-magnitude -> ordered)
        b = int(np.float32(v).view(np.uint32)) >> 16
        return -(b & 0x7FFF) if b & 0x8000 else b
    def val(k):
        b = (0x8000 | -k) if k < 0 else k
        return float(np.uint32(b << 16).view(np.float32))
    return [val(k) for k in range(key(lo), key(hi) + 1)]


def requant_flip_bound(h_exact, gs, down_abs, window):
    """How much FP4 re-quantisation of h can move one row's down projection
    when h is known only to within ``window`` (absolute, per element, e.g.
    ``gate_up_window``) of ``h_exact``.

    The layer rounds h to bf16 and quantises it (W4A4). A computation of h
    within the window rounds to some bf16 value between ``bf16(h - window)``
    and ``bf16(h + window)``. For every element where that is not just
    ``bf16(h)``, the element's block is quantised with each other such value
    (up to 8 of them; beyond that the two ends) and the rest of the row as the
    oracle has it (global scale ``gs``); the largest absolute change of each
    dequantised block element is added up over the ambiguous elements.
    ``down_abs`` is ``|Wd|``, the element-wise absolute value of the
    dequantised down matrix ``[H, I]``. Returns ``down_abs @ changes`` (the
    largest change of each output element of this row, by the triangle
    inequality, counting the flips one at a time), float64 ``[H]``.
    Pinned by: zero when no element can round to another bf16 value; an
    element put on a midpoint that straddles an e2m1 decision gives exactly
    one step times |Wd column| (tests).
    """
    h = np.asarray(h_exact, dtype=np.float64).reshape(-1)
    win = np.broadcast_to(np.asarray(window, dtype=np.float64).reshape(-1), h.shape)
    b0 = bf16_round(h).astype(np.float64)
    lo = bf16_round(h - win).astype(np.float64)
    hi = bf16_round(h + win).astype(np.float64)
    amb = np.nonzero((lo != b0) | (hi != b0))[0]
    diff = np.zeros_like(h)
    if amb.size:
        base = nvfp4.dequantize(*nvfp4.quantize(b0[None, :].astype(F32), gs=gs)[:2], gs)[0]
        rows, owner = [], []
        for i in amb:
            vals = _bf16_values_between(lo[i], hi[i])
            if len(vals) > 9:
                vals = [vals[0], vals[-1]]
            s0 = 16 * (i // 16)
            for v in vals:
                if v == b0[i]:
                    continue
                blk = b0[s0:s0 + 16].copy()
                blk[i - s0] = v
                rows.append(blk)
                owner.append(i)
        if rows:
            alt = np.stack(rows).astype(F32)
            q = nvfp4.quantize(alt, gs=gs)
            d = nvfp4.dequantize(q[0], q[1], gs)
            owner = np.asarray(owner)
            starts = 16 * (owner // 16)
            delta = np.abs(d - base[starts[:, None] + np.arange(16)[None, :]])
            # largest change per ambiguous element over its alternatives
            best = {}
            for r_, i in enumerate(owner):
                best[i] = delta[r_] if i not in best else np.maximum(best[i], delta[r_])
            for i, dl in best.items():
                s0 = 16 * (i // 16)
                diff[s0:s0 + 16] += dl
    return down_abs @ diff


def token_outputs_w4a16(x_tokens, ids, w, expert_weights, shared):
    """W4A16 outputs of a few tokens, one at a time, from their routing.

    ``x_tokens`` ``[n, H]``, ``ids``/``w`` ``[n, k]`` from ``route``;
    ``expert_weights(e)`` returns expert e's ``(gate, up, down)`` triple.
    ``out[t] = sum_j w[t, j] * expert_{ids[t, j]}(x_t) + shared(x_t)``. Used to
    check sampled tokens of workloads too large for ``layer``.
    """
    x_tokens = np.asarray(x_tokens, dtype=np.float64)
    out = np.zeros_like(x_tokens)
    for t in range(x_tokens.shape[0]):
        xt = x_tokens[t:t + 1]
        for j in range(ids.shape[1]):
            g, u, d = expert_weights(int(ids[t, j]))
            out[t] += np.float64(w[t, j]) * down_proj(gate_up_swiglu(xt, g, u), d)[0]
        if shared is not None:
            g, u, d = shared
            out[t] += down_proj(gate_up_swiglu(xt, g, u), d)[0]
    return out
