"""GPU parity of moe_route_fused_topk (softmax and top-k folded into the router GEMM's
epilogue, per-tile candidate lists merged by a light kernel) against moe_route and the fp64
oracle: identical logits and selection, gates and probability sums equal up to fp32
summation order.  Covers exact ties across expert tiles (duplicated router rows), a router
bias, tiles with fewer than 16 valid experts, E not a multiple of the tile width, and k = E."""

import numpy as np
import pytest
import torch

import oracle
from top_routing_grouped_gemm_gb300 import moe
from parity_util import RTOL_LOGITS, f64, relerr

pytestmark = pytest.mark.gpu


def _route(fn, p, x, w, bias):
    T, E, k = p.T, p.E, p.k
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    part = torch.empty((moe.moe_route_num_partials(p), E), dtype=torch.float32, device="cuda")
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.moe_route_workspace_size(p), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn(p, x, w, bias, idx, gate, part, logits, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return idx, gate, part, logits


def _inputs(T, d, E, seed, dup=False, bias=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, d, generator=g).to(torch.bfloat16)
    w = torch.randn(E, d, generator=g) * 0.02
    if dup:
        # experts e and e + E/2 (different expert tiles) share their router rows, and a block
        # of experts has all-zero rows: exact ties, resolved by the lower expert index
        half = E // 2
        w[half:2 * half] = w[:half]
        w[E // 3:E // 3 + 40] = 0.0
    b = None
    if bias:
        q = torch.arange(1, E + 1, dtype=torch.float64)
        wq = q ** -1.1
        b = (1.5 * torch.log(wq / wq.sum())).float()
    return x.cuda(), w.cuda(), (b.cuda() if b is not None else None)


@pytest.mark.parametrize("T, d, E, k, dup, bias", [
    (512, 256, 896, 16, False, False),
    (512, 256, 896, 16, True, False),
    (300, 192, 896, 16, False, True),
    (257, 128, 1000, 16, True, False),     # 128-wide tiles, the last one partly empty
    (200, 64, 10, 4, False, False),        # one tile with fewer than 16 experts
    (130, 64, 16, 16, True, True),         # k = E
    (64, 128, 300, 7, False, True),
])
def test_fused_topk_matches_route(T, d, E, k, dup, bias):
    p = moe.Problem(T, d, E, k, 64)
    x, w, b = _inputs(T, d, E, seed=T + E + k, dup=dup, bias=bias)
    i1, g1, p1, L1 = _route(moe.moe_route, p, x, w, b)
    i2, g2, p2, L2 = _route(moe.moe_route_fused_topk, p, x, w, b)
    assert torch.equal(L1, L2)
    assert torch.equal(i1, i2)
    L64 = f64(L1)
    assert relerr(L64, oracle.router_logits(f64(x), f64(w), f64(b) if b is not None else None)) \
        <= RTOL_LOGITS
    ref = oracle.topk_select(L64, k)
    assert np.array_equal(i2.cpu().numpy(), ref)
    prob = oracle.softmax(L64)
    assert relerr(f64(g2), oracle.renormalised_gates(prob, ref)) <= 1e-5
    assert relerr(f64(g2), f64(g1)) <= 1e-6
    assert relerr(f64(p2).sum(axis=0), prob.sum(axis=0)) <= 1e-5


def test_fused_topk_rejects_k_above_16():
    p = moe.Problem(64, 64, 64, 17, 64)
    x, w, b = _inputs(64, 64, 64, seed=3)
    with pytest.raises(moe.MoEError):
        _route(moe.moe_route_fused_topk, p, x, w, b)
