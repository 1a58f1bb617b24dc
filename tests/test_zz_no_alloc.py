"""moe_permute_noalloc (the permutation for callers that cannot allocate device
memory per call: its scratch is a fixed array inside the library) must give
exactly what moe_permute gives with a caller workspace, call after call, even
though every call reuses the same scratch. This file is collected last."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _run(fn_noalloc, ids, T, k, E):
    from nvfp4_mixture_experts_moe_gb300 import binding as B
    P = T * k
    outs = []
    for noalloc in (False, True):
        counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
        offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
        perm = torch.full((max(P, 1),), -7, dtype=torch.int32, device="cuda")
        inv = torch.full((max(P, 1),), -7, dtype=torch.int32, device="cuda")
        if noalloc:
            status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
            B.moe_permute_noalloc(ids, T, k, E, counts, offsets, perm, inv, status)
            torch.cuda.synchronize()
            st = int(status.item())
        else:
            ws = torch.zeros(B.moe_permute_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
            B.moe_permute(ids, T, k, E, counts, offsets, perm, inv, ws)
            st = B.moe_get_device_status(ws)
        outs.append((st, counts.cpu(), offsets.cpu(), perm.cpu()[:P], inv.cpu()[:P]))
    return outs


@pytest.mark.parametrize("T,k,E", [(4096, 8, 320), (16384, 8, 256), (8, 8, 320)])
def test_noalloc_matches_workspace_version_two_calls(T, k, E):
    for call in range(2):  # second call runs on the scratch the first one left behind
        g = torch.Generator().manual_seed(100 * call + T + E)
        ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
        if call == 1:
            ids[:, 0] = 3  # a different histogram from the first call
        ref, got = _run(True, ids.cuda(), T, k, E)
        assert got[0] == ref[0] == 0
        for a, b in zip(ref[1:], got[1:]):
            assert torch.equal(a, b)


def test_noalloc_reports_bad_ids_and_recovers():
    from nvfp4_mixture_experts_moe_gb300 import binding as B
    bad = torch.tensor([[0, 1], [9, 2]], dtype=torch.int32, device="cuda")
    ref, got = _run(True, bad, 2, 2, 4)
    assert got[0] == B.MOE_ERR_DEVICE == ref[0]
    assert torch.equal(ref[4], got[4])
    good = torch.tensor([[0, 1], [3, 2]], dtype=torch.int32, device="cuda")
    ref, got = _run(True, good, 2, 2, 4)
    assert got[0] == 0  # the status word from the previous call was cleared


def test_noalloc_rejects_oversized_problems():
    from nvfp4_mixture_experts_moe_gb300 import binding as B
    T, k, E = 65536, 8, 1024   # histogram of 128 chunks x 1024 experts > 64 KiB
    dummy = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MoeError) as ei:
        B.moe_permute_noalloc(dummy, T, k, E, dummy, dummy, dummy, dummy)
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("T,k,E", [(4096, 8, 320), (8, 8, 320), (2048, 8, 320)])
def test_noalloc_matches_oracle_two_calls(T, k, E):
    """Bit for bit against the oracle's stable counting sort, on two calls in a
    row (the second reuses the scratch the first one left behind)."""
    from nvfp4_mixture_experts_moe_gb300 import binding as B
    from oracle import moe as omoe
    P = T * k
    for call in range(2):
        g = torch.Generator().manual_seed(7 * call + T)
        ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
        if call == 1:
            ids[: T // 2, 1] = E - 1  # a skewed histogram on the second call
        counts = torch.empty(E, dtype=torch.int32, device="cuda")
        offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        perm = torch.empty(P, dtype=torch.int32, device="cuda")
        inv = torch.empty(P, dtype=torch.int32, device="cuda")
        status = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        B.moe_permute_noalloc(ids.cuda(), T, k, E, counts, offsets, perm, inv, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        rc, ro, rp, ri = omoe.permute(ids.numpy(), E)
        assert (counts.cpu().numpy() == rc).all()
        assert (offsets.cpu().numpy() == ro).all()
        assert (perm.cpu().numpy() == rp).all()
        assert (inv.cpu().numpy() == ri).all()
