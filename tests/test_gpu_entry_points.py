"""The standalone entry points of the C ABI that the fused forward also runs
internally (SwiGLU, combine, the quantiser's amax) against the CPU oracle.

"vLLM on the NVIDIA DGX Spark: A Complete Technical Guide", section 4.3
(SwiGLU between the two expert GEMMs; top-k weight reduction) and section 7.1
([Combine]).
"""
import numpy as np
import pytest
import torch

from oracle import moe as omoe
from oracle import nvfp4 as onv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def B():
    from nvfp4_mixture_experts_moe_gb300 import binding
    return binding


@pytest.mark.parametrize("rows,I", [(1, 64), (37, 128), (300, 1536)])
def test_swiglu_matches_oracle(rows, I):
    g = torch.Generator().manual_seed(rows * 7 + I)
    gu = torch.randn(rows, 2 * I, generator=g) * 3.0
    gu[0, 0], gu[0, I] = -40.0, 2.0   # exp overflow side of silu: the result is -0 or tiny
    h = torch.empty(rows, I, dtype=torch.bfloat16, device="cuda")
    B().moe_swiglu(gu.cuda(), rows, I, h)
    torch.cuda.synchronize()
    gn = gu.numpy().astype(np.float64)
    ref = omoe.silu(gn[:, :I]) * gn[:, I:]
    got = h.float().cpu().numpy()
    # bf16 rounding of the result (at most half an ulp, 2^-8 |ref|) plus the
    # fp32 evaluation with the hardware exp and fast division (~1e-6 relative)
    bar = (2.0 ** -8 + 1e-5) * np.abs(ref) + 1e-30
    assert np.all(np.abs(got - ref) <= bar), float(np.max(np.abs(got - ref) - bar))


def _combine_case(T, k, H, shared, weighted, seed):
    g = torch.Generator().manual_seed(seed)
    E = max(2 * k, 8)
    ids = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32) if T < 4096 \
        else torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    _, _, _, inv = omoe.permute(ids.numpy(), E)
    y = (torch.randn(T * k, H, generator=g) * 2.0).to(torch.bfloat16)
    ys = torch.randn(T, H, generator=g) * 2.0 if shared else None
    w = torch.rand(T, k, generator=g) + 0.1 if weighted else None
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    B().moe_combine(y.cuda(), torch.from_numpy(inv).cuda(), None if w is None else w.cuda(),
                    None if ys is None else ys.cuda(), T, k, H, out)
    torch.cuda.synchronize()
    yn = y.float().numpy().astype(np.float64)
    wn = np.ones((T, k)) if w is None else w.numpy().astype(np.float64)
    terms = yn[inv.reshape(T, k)] * wn[:, :, None]                  # [T, k, H]
    ref = terms.sum(axis=1)
    mag = np.abs(terms).sum(axis=1)
    if shared:
        ysn = ys.numpy().astype(np.float64)
        ref = ref + ysn
        mag = mag + np.abs(ysn)
    got = out.float().cpu().numpy()
    # bf16 output rounding plus the fp32 sum of k+1 terms (fixed order)
    bar = 2.0 ** -8 * np.abs(ref) + (k + 2) * 2.0 ** -24 * mag + 1e-30
    assert np.all(np.abs(got - ref) <= bar), float(np.max(np.abs(got - ref) - bar))
    return out


@pytest.mark.parametrize("T,k,H,shared,weighted", [
    (5, 2, 64, 1, True), (64, 8, 4096, 1, False), (3, 1, 8, 0, True), (17, 4, 7168, 0, False)])
def test_combine_matches_oracle(T, k, H, shared, weighted):
    _combine_case(T, k, H, shared, weighted, seed=T * 131 + H)


def test_combine_more_tokens_than_grid_y():
    """65,536 tokens: more than the 65,535 blocks a grid's y dimension holds."""
    out = _combine_case(65536, 2, 64, 1, True, seed=3)
    assert out.shape[0] == 65536


def test_combine_is_deterministic():
    a = _combine_case(64, 8, 4096, 1, True, seed=9)
    b = _combine_case(64, 8, 4096, 1, True, seed=9)
    assert torch.equal(a, b)


def test_quantize_amax_ignores_nan():
    """A NaN activation is outside the contract, but it must not become the
    tensor's amax (an infinite amax would make the global scale 0 and zero
    every code): the global scale is the one of the finite values."""
    from nvfp4_mixture_experts_moe_gb300 import quantize_bf16
    g = torch.Generator().manual_seed(4)
    x = torch.randn(4, 256, generator=g).to(torch.bfloat16)
    x[1, 7] = float("nan")
    q, sf, gs = quantize_bf16(x.cuda())
    torch.cuda.synchronize()
    xf = x.float().numpy()
    finite_amax = np.float32(np.nanmax(np.abs(xf)))
    assert np.float32(gs.item()) == onv.global_scale(finite_amax)
    # every block without the NaN quantises exactly as the oracle's
    clean = xf.copy()
    clean[1, 7] = 0.0
    rq, rsf, rgs = onv.quantize(clean, gs=onv.global_scale(finite_amax))
    got_sf = sf.cpu().numpy()
    got_q = onv.unpack(q.cpu().numpy())
    mask = np.ones(got_sf.shape, dtype=bool)
    mask[1, 0] = False
    assert (got_sf[mask] == rsf[mask]).all()
    assert (got_q.reshape(4, 16, 16)[mask] == rq.reshape(4, 16, 16)[mask]).all()
