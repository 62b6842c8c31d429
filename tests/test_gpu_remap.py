"""GPU parity of overflow remapping ("Adapting Ultra-Large MoE Models ...", section 3.3:
excess tokens remapped instead of dropped) against the oracle's rule, through the C ABI:
the alternatives and the remapped index maps bit-exact (the oracle orders the GPU's fp32
logits), the layer output and the LoRA backward within 5e-3."""

import numpy as np
import pytest
import torch

import oracle
from top_routing_grouped_gemm_gb300 import moe, synth
from parity_util import (RTOL_FP, DeviceExperts, f64, lora64, relerr, to_dev)

pytestmark = pytest.mark.gpu


def run_remap(cfg, dev, R, gather=False, train=False):
    p = moe.problem_of(cfg)
    buf = moe.LayerBuffers(p, "cuda", train=train, remap_rounds=R)
    moe.layer_forward(buf, dev["x"], dev["w_router"], dev.get("bias"), dev["w_gate"],
                      dev["w_up"], dev["w_down"], dev.get("lora"), gather=gather)
    if train:
        moe.layer_backward(buf, dev["dy"], dev["x"], dev["w_router"], dev["w_gate"],
                           dev["w_up"], dev["w_down"], dev.get("lora"))
    torch.cuda.synchronize()
    assert int(buf.dev_status.item()) == 0
    return p, buf


def check_maps(p, buf, R):
    L = f64(buf.logits)
    order = oracle.topk_select(L, (R + 1) * p.k)
    assert np.array_equal(buf.topk_idx.cpu().numpy(), order[:, :p.k])
    assert np.array_equal(buf.alt_idx.cpu().numpy(), order[:, p.k:])
    C = oracle.capacity(p.T, p.k, p.E, p.cap_num, p.cap_den)
    D = oracle.dispatch_remap(order, p.k, p.E, C, R)
    assert np.array_equal(buf.counts.cpu().numpy(), D["counts"])
    assert np.array_equal(buf.offsets.cpu().numpy(), D["offsets"])
    assert np.array_equal(buf.slot_row.cpu().numpy(), D["slot_row"])
    assert np.array_equal(buf.slot_expert.cpu().numpy(), D["slot_expert"])
    rs = buf.row_slot.cpu().numpy()
    assert np.array_equal(rs[:D["n_kept"]], D["row_slot"]) and (rs[D["n_kept"]:] == -1).all()
    assert buf.n_kept_dropped.cpu().tolist() == [D["n_kept"], D["n_dropped"]]
    return L, D


def small_cfg(**kw):
    base = dict(name="remap", T=400, d=128, E=12, k=2, F=128, cap_num=1, cap_den=2,
                zipf_bias=True)
    base.update(kw)
    return synth.MoEConfig(**base)


CASES = [
    (small_cfg(), 1),
    (small_cfg(), 3),
    (small_cfg(T=777, d=192, E=16, k=4, F=192, r=16, alpha=32.0, cap_num=3, cap_den=4), 2),
    (small_cfg(T=300, E=64, k=16, cap_num=1, cap_den=1), 1),
    (small_cfg(T=50, E=8, k=4, cap_num=0, cap_den=1), 1),      # capacity 0: all dropped
    (small_cfg(T=200, E=8, k=2, cap_num=0, cap_den=0), 3),     # unlimited: pass 0 only
]


@pytest.mark.parametrize("cfg, R", CASES, ids=["R1", "R3", "lora_R2", "k16_R1",
                                               "capacity_zero", "unlimited"])
def test_remap_layer_whole(cfg, R):
    inp = synth.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    p, buf = run_remap(cfg, dev, R)
    L, D = check_maps(p, buf, R)
    ref = oracle.moe_forward(f64(inp["x"]), None, f64(inp["w_gate"]), f64(inp["w_up"]),
                             f64(inp["w_down"]), p.k, p.cap_num, p.cap_den,
                             lora=lora64(inp.get("lora")), s=p.lora_scale, logits=L,
                             remap_rounds=R)
    n = D["n_kept"]
    if n:
        assert relerr(f64(buf.h[:n]), ref["h"]) <= RTOL_FP
    assert relerr(f64(buf.y), ref["y"]) <= RTOL_FP or np.abs(ref["y"]).max() == 0
    assert abs(float(buf.aux.item()) - ref["aux"]) <= 1e-5 * abs(ref["aux"])
    if p.cap_den and p.cap_num:
        assert D["n_dropped"] < oracle.dispatch(oracle.topk_select(L, p.k), p.E,
                                                oracle.capacity(p.T, p.k, p.E, p.cap_num,
                                                                p.cap_den))["n_dropped"]


def test_remap_zero_rounds_equals_plain_dispatch():
    cfg = small_cfg(T=500)
    dev = to_dev(synth.make_inputs(cfg, "cpu"))
    p = moe.problem_of(cfg)
    a = moe.LayerBuffers(p, "cuda")
    moe.layer_forward(a, dev["x"], dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"],
                      dev["w_down"], gather=False)
    ws = torch.empty(moe.moe_dispatch_remap_workspace_size(p, 0), dtype=torch.uint8,
                     device="cuda")
    b = {n: torch.empty_like(getattr(a, n)) for n in ("counts", "offsets", "slot_row",
                                                       "row_slot", "n_kept_dropped", "x_perm")}
    moe.moe_dispatch_remap(p, a.topk_idx, None, 0, dev["x"], b["counts"], b["offsets"],
                           b["slot_row"], b["row_slot"], None, b["n_kept_dropped"], b["x_perm"],
                           ws, a.dev_status)
    torch.cuda.synchronize()
    n = int(a.n_kept_dropped[0].item())
    for name in ("counts", "offsets", "slot_row", "row_slot", "n_kept_dropped"):
        assert torch.equal(b[name], getattr(a, name)), name
    assert torch.equal(b["x_perm"][:n], a.x_perm[:n])


def test_remap_fused_gather_matches_permuted_path():
    cfg = small_cfg(T=600, E=16, k=4, F=192, d=192)
    dev = to_dev(synth.make_inputs(cfg, "cpu"))
    _, a = run_remap(cfg, dev, 2, gather=False)
    _, b = run_remap(cfg, dev, 2, gather=True)
    assert torch.equal(a.slot_row, b.slot_row) and torch.equal(a.y, b.y)


def test_remap_backward_whole():
    cfg = small_cfg(T=300, d=128, E=12, k=3, F=128, r=8, alpha=16.0, backward=True)
    inp = synth.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    R = 2
    p, buf = run_remap(cfg, dev, R, train=True)
    L, D = check_maps(p, buf, R)
    X = f64(inp["x"])
    Wg, Wu, Wd = f64(inp["w_gate"]), f64(inp["w_up"]), f64(inp["w_down"])
    lora = lora64(inp["lora"])
    fwd = oracle.moe_forward(X, None, Wg, Wu, Wd, p.k, p.cap_num, p.cap_den, lora=lora,
                             s=p.lora_scale, logits=L, remap_rounds=R)
    bwd = oracle.moe_backward(fwd, X, f64(inp["dy"]), f64(inp["w_router"]), Wg, Wu, Wd, lora,
                              p.lora_scale)
    assert relerr(f64(buf.dgate), bwd["dgate"]) <= RTOL_FP
    assert relerr(f64(buf.dx), bwd["dx"]) <= RTOL_FP
    for nm in ("A_g", "B_g", "A_u", "B_u", "A_d", "B_d"):
        assert relerr(f64(buf.grads["d" + nm]), bwd["d" + nm]) <= RTOL_FP, nm


def test_remap_full_c3():
    """c3 at full size with one remap round (k = 16, so each slot has one alternative): the
    maps bit-exact against the oracle rule on the GPU's logits, y on every token."""
    cfg = synth.config("c3")
    inp = synth.make_inputs(cfg, "cuda")
    p, buf = run_remap(cfg, inp, 1, gather=False)
    L, D = check_maps(p, buf, 1)
    plain = oracle.dispatch(oracle.topk_select(L, p.k), p.E, 366)
    assert D["n_dropped"] < plain["n_dropped"]
    ref = oracle.moe_forward(f64(inp["x"]), None, DeviceExperts(inp["w_gate"]),
                             DeviceExperts(inp["w_up"]), DeviceExperts(inp["w_down"]), p.k,
                             p.cap_num, p.cap_den, logits=L, remap_rounds=1)
    assert relerr(f64(buf.y), ref["y"]) <= RTOL_FP
