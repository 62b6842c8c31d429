"""GPU parity of the LoRA backward (gradient of <dy, y> with routing fixed, base weights and
router frozen) against the fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

import oracle
from top_routing_grouped_gemm_gb300 import moe, synth
from parity_util import RTOL_FP, f64, lora64, oracle_experts_backward, relerr, to_dev

pytestmark = pytest.mark.gpu

GRADS = ("A_g", "B_g", "A_u", "B_u", "A_d", "B_d")


def run_fwd_bwd(cfg, inp):
    p = moe.problem_of(cfg)
    buf = moe.LayerBuffers(p, "cuda", train=True)
    moe.layer_forward(buf, inp["x"], inp["w_router"], inp.get("bias"), inp["w_gate"],
                      inp["w_up"], inp["w_down"], inp.get("lora"))
    moe.layer_backward(buf, inp["dy"], inp["x"], inp["w_router"], inp["w_gate"], inp["w_up"],
                       inp["w_down"], inp.get("lora"))
    torch.cuda.synchronize()
    assert int(buf.dev_status.item()) == 0
    return p, buf


def small_cfg(**kw):
    base = dict(name="small_bwd", T=300, d=192, E=6, k=2, F=192, r=16, alpha=32.0,
                backward=True)
    base.update(kw)
    return synth.MoEConfig(**base)


@pytest.mark.parametrize("cfg", [
    small_cfg(),
    small_cfg(T=777, d=320, E=9, k=3, F=448, r=24, alpha=48.0, cap_num=1, cap_den=1),
    small_cfg(T=260, d=256, E=40, k=4, F=128, r=8, alpha=16.0, cap_num=3, cap_den=4,
              zipf_bias=True),
    small_cfg(r=0, alpha=0.0),
    small_cfg(T=50, d=128, E=16, k=4, F=64, r=16, alpha=32.0, cap_num=0, cap_den=1),
    small_cfg(T=1, d=128, E=8, k=2, F=64, r=8, alpha=16.0),
    small_cfg(T=300, d=256, E=12, k=3, F=192, r=64, alpha=128.0),
    # 129..256 rows per expert: the dx GEMM on 256-row tiles
    small_cfg(T=400, d=192, E=4, k=2, F=192),
    small_cfg(T=500, d=320, E=5, k=2, F=256, r=8, alpha=16.0, cap_num=5, cap_den=4),
    # over 1024 rows per expert: the dh and dx GEMMs on CTA pairs
    small_cfg(T=2600, d=192, E=4, k=2, F=192),
], ids=["small", "ragged_capacity", "many_experts_some_empty", "no_lora", "capacity_zero",
        "one_token", "lora_r64", "two_tile_groups", "two_tile_groups_ragged_capacity",
        "big_groups"])
def test_backward_whole(cfg):
    inp = synth.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    p, buf = run_fwd_bwd(cfg, dev)
    L_gpu = f64(buf.logits)
    X, Wr = f64(inp["x"]), f64(inp["w_router"])
    Wg, Wu, Wd = f64(inp["w_gate"]), f64(inp["w_up"]), f64(inp["w_down"])
    lora = lora64(inp.get("lora"))
    fwd = oracle.moe_forward(X, None, Wg, Wu, Wd, p.k, p.cap_num, p.cap_den, lora=lora,
                             s=p.lora_scale, logits=L_gpu)
    # the router's gradient path uses W_r: give the oracle the fp32 router weights
    bwd = oracle.moe_backward(fwd, X, f64(inp["dy"]), Wr, Wg, Wu, Wd, lora, p.lora_scale)
    n = fwd["disp"]["n_kept"]
    assert relerr(f64(buf.dz_perm[:n]), bwd["dO"]) <= RTOL_FP
    assert relerr(f64(buf.dgate), bwd["dgate"]) <= RTOL_FP
    assert relerr(f64(buf.dx_perm[:n]), bwd["dx_perm"]) <= RTOL_FP
    assert relerr(f64(buf.dx), bwd["dx"]) <= RTOL_FP
    if p.r:
        for nm in GRADS:
            assert relerr(f64(buf.grads["d" + nm]), bwd["d" + nm]) <= RTOL_FP, nm
        # experts that received no rows get exactly zero gradients
        empty = np.where(np.diff(fwd["disp"]["offsets"]) == 0)[0]
        for e in empty:
            for nm in GRADS:
                assert float(buf.grads["d" + nm][e].abs().max()) == 0.0


def test_gate_gradient_from_dh_matches_combine_backward():
    """The gate gradients the expert backward forms from its dh product (<dh, h> / g) against
    the combine backward's <dy, y_perm> / g on the same step (two roundings apart)."""
    cfg = small_cfg(T=300, cap_num=5, cap_den=4)
    inp = synth.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    p, buf = run_fwd_bwd(cfg, dev)
    dg_ref = torch.empty_like(buf.dgate)
    dz = torch.empty_like(buf.dz_perm)
    moe.moe_combine_bwd(p, dev["dy"], buf.y_perm, buf.slot_row, buf.topk_gate, dz, dg_ref)
    torch.cuda.synchronize()
    assert torch.equal(dz, buf.dz_perm)
    assert relerr(f64(buf.dgate), f64(dg_ref)) <= RTOL_FP
    dropped = buf.slot_row < 0
    assert bool((buf.dgate[dropped.view(buf.dgate.shape)] == 0).all())


def test_fused_dispatch_route_backward_is_bit_exact():
    cfg = small_cfg(T=257, cap_num=5, cap_den=4)
    inp = synth.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    p, buf = run_fwd_bwd(cfg, dev)
    dx2 = torch.empty_like(buf.dx)
    moe.moe_dispatch_bwd(p, buf.dx_perm, buf.slot_row, dx2)
    moe.moe_route_bwd(p, buf.topk_idx, buf.topk_gate, buf.dgate, dev["w_router"], dx2)
    torch.cuda.synchronize()
    assert torch.equal(buf.dx, dx2)


def test_backward_gate_and_expert_paths_separately():
    cfg = small_cfg(T=200, cap_num=5, cap_den=4)
    inp = synth.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    p, buf = run_fwd_bwd(cfg, dev)
    X = f64(inp["x"])
    lora = lora64(inp.get("lora"))
    fwd = oracle.moe_forward(X, None, f64(inp["w_gate"]), f64(inp["w_up"]), f64(inp["w_down"]),
                             p.k, p.cap_num, p.cap_den, lora=lora, s=p.lora_scale,
                             logits=f64(buf.logits))
    bwd = oracle.moe_backward(fwd, X, f64(inp["dy"]), f64(inp["w_router"]), f64(inp["w_gate"]),
                              f64(inp["w_up"]), f64(inp["w_down"]), lora, p.lora_scale)
    # expert path alone: dispatch backward into a fresh buffer
    dx_e = torch.empty_like(buf.dx)
    moe.moe_dispatch_bwd(p, buf.dx_perm, buf.slot_row, dx_e)
    torch.cuda.synchronize()
    assert relerr(f64(dx_e), bwd["dx_expert"]) <= RTOL_FP
    assert relerr(f64(buf.dx) - f64(dx_e), bwd["dx_gate"]) <= RTOL_FP


def test_full_c5_sampled():
    """c5 at full size: the LoRA gradients and dx_perm rows of 32 experts (all their rows),
    and dgate and dx of 64 tokens (each token's 16 expert slots plus the gate path through
    the renormalised softmax), against the oracle."""
    cfg = synth.config("c5")
    inp = synth.make_inputs(cfg, "cuda")
    p, buf = run_fwd_bwd(cfg, inp)
    k, s = p.k, p.lora_scale
    L_gpu = f64(buf.logits)
    idx = oracle.topk_select(L_gpu, k)
    assert np.array_equal(idx, buf.topk_idx.cpu().numpy())
    prob = oracle.softmax(L_gpu)
    gates = oracle.renormalised_gates(prob, idx)
    D = oracle.dispatch(idx, p.E, None)
    assert np.array_equal(buf.slot_row.cpu().numpy(), D["slot_row"])
    offs = D["offsets"]
    rng = np.random.default_rng(5)
    # LoRA gradients of 32 experts (all their rows)
    experts = sorted(set([0, p.E - 1] + list(rng.choice(np.arange(1, p.E - 1), 30, replace=False))))
    assert len(experts) >= 32
    for e in experts:
        lo, hi = int(offs[e]), int(offs[e + 1])
        rows = D["row_slot"][lo:hi]
        tok = torch.from_numpy(rows // k).cuda()
        Xe = f64(inp["x"][tok])
        dOe = gates.reshape(-1)[rows][:, None] * f64(inp["dy"][tok])
        Le = lora64(inp["lora"], e)
        dX, ge = oracle.expert_backward(Xe, dOe, f64(inp["w_gate"][e]), f64(inp["w_up"][e]),
                                        f64(inp["w_down"][e]), Le, s)
        assert relerr(f64(buf.dx_perm[lo:hi]), dX) <= RTOL_FP, e
        for nm in GRADS:
            assert relerr(f64(buf.grads["d" + nm][e]), ge[nm]) <= RTOL_FP, (e, nm)
    # dgate and dx of 64 tokens: each expert's slots evaluated together
    tokens = sorted(set([0, p.T - 1] + list(rng.choice(np.arange(1, p.T - 1), 62, replace=False))))
    assert len(tokens) >= 64
    x64 = np.zeros((p.T, p.d))
    dy64 = np.zeros((p.T, p.d))
    tt = torch.tensor(tokens).cuda()
    x64[tokens] = f64(inp["x"][tt])
    dy64[tokens] = f64(inp["dy"][tt])
    by_expert = {}
    for t in tokens:
        for j in range(k):
            by_expert.setdefault(int(idx[t, j]), []).append((t, j))
    o, dXs = oracle_experts_backward(inp, p, by_expert, gates, x64, dy64)
    Wr = f64(inp["w_router"])
    dg = np.array([[float(dy64[t] @ o[(t, j)]) for j in range(k)] for t in tokens])
    dx_ref = np.array([sum(dXs[(t, j)] for j in range(k)) for t in tokens])
    dl = oracle.route_backward(prob[tokens], idx[tokens], gates[tokens], dg,
                               np.ones((len(tokens), k)))
    dx_ref = dx_ref + dl @ Wr
    assert relerr(f64(buf.dgate[tt]), dg) <= RTOL_FP
    assert relerr(f64(buf.dx[tt]), dx_ref) <= RTOL_FP
    for n, t in enumerate(tokens[:8]):
        assert relerr(f64(buf.dx[t:t + 1]), dx_ref[n:n + 1]) <= RTOL_FP, t
