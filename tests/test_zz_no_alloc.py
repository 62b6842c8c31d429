"""moe_dispatch_noalloc, the dispatch entry point for callers that cannot allocate device
memory (their memory belongs to another allocator, or they only receive tensor pointers):
through the C ABI it must give exactly the outputs of moe_dispatch, on consecutive calls
that share the library's built-in scratch array.  Kept in a file of its own that pytest
collects last."""

import pytest
import torch

from top_routing_grouped_gemm_gb300 import moe, synth

pytestmark = pytest.mark.gpu


def _routing(cfg, seed):
    g = torch.Generator().manual_seed(seed)
    L = torch.randn((cfg.T, cfg.E), generator=g)
    if cfg.zipf_bias:
        L = L + synth.zipf_bias(cfg.E)
    return torch.topk(L, cfg.k, dim=1).indices.to(torch.int32)


def _outputs(p, device="cuda"):
    N = p.T * p.k
    return dict(counts=torch.empty(p.E, dtype=torch.int32, device=device),
                offsets=torch.empty(p.E + 1, dtype=torch.int32, device=device),
                slot_row=torch.empty(N, dtype=torch.int32, device=device),
                row_slot=torch.empty(N, dtype=torch.int32, device=device),
                n_kept_dropped=torch.empty(2, dtype=torch.int32, device=device),
                x_perm=torch.zeros((N, p.d), dtype=torch.bfloat16, device=device),
                status=torch.zeros(1, dtype=torch.int32, device=device))


def _dispatch(p, idx, x, noalloc, maps_only=False):
    o = _outputs(p)
    x_perm = None if maps_only else o["x_perm"]
    x = None if maps_only else x
    if noalloc:
        moe.moe_dispatch_noalloc(p, idx, x, o["counts"], o["offsets"], o["slot_row"],
                                 o["row_slot"], o["n_kept_dropped"], x_perm, o["status"])
    else:
        ws = torch.empty(moe.moe_dispatch_workspace_size(p), dtype=torch.uint8, device="cuda")
        moe.moe_dispatch(p, idx, x, o["counts"], o["offsets"], o["slot_row"], o["row_slot"],
                         o["n_kept_dropped"], x_perm, ws, o["status"])
    torch.cuda.synchronize()
    return o


def test_noalloc_dispatch_matches_workspace_dispatch_on_consecutive_calls():
    cases = [synth.config("c3", T=4096), synth.config("c2")]  # capacity drops, then dropless
    for n, cfg in enumerate(cases):
        p = moe.problem_of(cfg)
        idx = _routing(cfg, seed=n).cuda()
        x = synth.make_inputs(cfg, "cuda", seed=n, weights=False)["x"]
        ref = _dispatch(p, idx, x, noalloc=False)
        got = _dispatch(p, idx, x, noalloc=True)
        n_kept = int(ref["n_kept_dropped"][0].item())
        assert int(got["status"].item()) == 0
        for key in ("counts", "offsets", "slot_row", "row_slot", "n_kept_dropped"):
            assert torch.equal(got[key], ref[key]), (cfg.name, key)
        assert torch.equal(got["x_perm"][:n_kept], ref["x_perm"][:n_kept]), cfg.name
        if cfg.cap_den:
            assert int(ref["n_kept_dropped"][1].item()) > 0


def test_noalloc_dispatch_index_maps_only_matches_workspace_dispatch():
    """x and x_perm both NULL: only the index maps (the mode the fused-permute expert GEMM
    uses), on two consecutive calls."""
    for n, cfg in enumerate([synth.config("c3", T=2048), synth.config("c2", T=1024)]):
        p = moe.problem_of(cfg)
        idx = _routing(cfg, seed=10 + n).cuda()
        ref = _dispatch(p, idx, None, noalloc=False, maps_only=True)
        got = _dispatch(p, idx, None, noalloc=True, maps_only=True)
        assert int(got["status"].item()) == 0
        for key in ("counts", "offsets", "slot_row", "row_slot", "n_kept_dropped"):
            assert torch.equal(got[key], ref[key]), (cfg.name, key)


def test_noalloc_dispatch_rejects_problems_beyond_its_scratch():
    p = moe.Problem(T=1 << 20, d=64, E=1024, k=8, F=64)  # needs far more than 8 MiB
    o = _outputs(moe.Problem(T=8, d=64, E=8, k=2, F=64))
    with pytest.raises(moe.MoEError) as err:
        moe.moe_dispatch_noalloc(p, o["slot_row"], o["x_perm"], o["counts"], o["offsets"],
                                 o["slot_row"], o["row_slot"], o["n_kept_dropped"], o["x_perm"])
    assert err.value.status == 3  # MOE_ERR_WORKSPACE, nothing enqueued
