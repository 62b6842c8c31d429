"""GPU parity of the forward path (route, dispatch, experts, combine, aux) against the fp64
oracle, through the C ABI, on the seeded workloads and on edge cases."""

import numpy as np
import pytest
import torch

import oracle
from top_routing_grouped_gemm_gb300 import moe, synth
from parity_util import (RTOL_FP, RTOL_LOGITS, DeviceExperts, ExpertCache, f64, lora64,
                         oracle_tokens, relerr, run_forward, to_dev)

pytestmark = pytest.mark.gpu


def check_routing(buf, p, inp, full_logits_check=True):
    """Logits to fp32 accuracy; selection, order, gates and probabilities on the GPU's logits."""
    L_gpu = f64(buf.logits)
    if full_logits_check:
        L64 = oracle.router_logits(f64(inp["x"]), f64(inp["w_router"]), f64(inp.get("bias")))
        assert relerr(L_gpu, L64) <= RTOL_LOGITS
    idx = buf.topk_idx.cpu().numpy()
    idx_ref = oracle.topk_select(L_gpu, p.k)
    assert np.array_equal(idx, idx_ref)
    prob = oracle.softmax(L_gpu)
    g_ref = oracle.renormalised_gates(prob, idx_ref)
    assert relerr(f64(buf.topk_gate), g_ref) <= 1e-5
    P_gpu = f64(buf.partials).sum(axis=0) / p.T
    assert relerr(P_gpu, prob.mean(axis=0)) <= 1e-5
    return L_gpu, idx_ref, g_ref, prob


def check_dispatch(buf, p, idx, x=None):
    C = oracle.capacity(p.T, p.k, p.E, p.cap_num, p.cap_den)
    D = oracle.dispatch(idx, p.E, C)
    assert np.array_equal(buf.counts.cpu().numpy(), D["counts"])
    assert np.array_equal(buf.offsets.cpu().numpy(), D["offsets"])
    assert np.array_equal(buf.slot_row.cpu().numpy(), D["slot_row"])
    rs = buf.row_slot.cpu().numpy()
    assert np.array_equal(rs[:D["n_kept"]], D["row_slot"])
    assert (rs[D["n_kept"]:] == -1).all()
    assert buf.n_kept_dropped.cpu().tolist() == [D["n_kept"], D["n_dropped"]]
    if x is not None:
        rows = torch.from_numpy(D["row_slot"] // p.k).to(x.device)
        assert torch.equal(buf.x_perm[:D["n_kept"]], x[rows])
    return D


def small_cfg(**kw):
    base = dict(name="small", T=300, d=192, E=6, k=2, F=192)
    base.update(kw)
    return synth.MoEConfig(**base)


# ----------------------------------------------------------------------------- whole-problem

@pytest.mark.parametrize("cfg", [
    synth.config("c1"),
    small_cfg(),
    small_cfg(cap_num=5, cap_den=4, zipf_bias=True),
    small_cfg(r=16, alpha=32.0),
    small_cfg(T=777, d=320, E=9, k=3, F=448, r=24, alpha=48.0, cap_num=1, cap_den=1),
    small_cfg(T=129, d=64, E=1, k=1, F=64),
    small_cfg(T=1, d=128, E=8, k=2, F=64),
    small_cfg(T=50, d=64, E=16, k=4, F=64, cap_num=0, cap_den=1),
    small_cfg(T=200, d=128, E=1024, k=32, F=64),
    small_cfg(T=64, d=128, E=32, k=32, F=128),
    small_cfg(T=300, d=256, E=12, k=3, F=192, r=64, alpha=128.0),
    small_cfg(T=300, d=256, E=12, k=3, F=192, r=8, alpha=16.0, cap_num=1, cap_den=2),
    small_cfg(T=40, d=192, E=500, k=8, F=128, zipf_bias=True),
    # groups of over 1024 rows on average: the expert GEMMs run on CTA pairs
    small_cfg(T=2600, d=192, E=4, k=2, F=192),
    small_cfg(T=2200, d=256, E=2, k=1, F=320, r=16, alpha=32.0),
    small_cfg(T=3000, d=128, E=4, k=2, F=128, cap_num=3, cap_den=4, zipf_bias=True),
    # 129..256 rows per expert: the gate/up GEMM on CTA pairs
    small_cfg(T=400, d=192, E=4, k=2, F=192),
    small_cfg(T=500, d=320, E=5, k=2, F=256, r=16, alpha=32.0, cap_num=5, cap_den=4),
], ids=["c1", "small", "small_capacity_bias", "small_lora", "ragged_lora_capacity", "single_expert",
        "one_token", "capacity_zero", "max_experts_k32", "k_equals_E", "lora_r64", "lora_r8_half_capacity",
        "mostly_empty_experts", "big_groups", "big_groups_lora", "big_groups_capacity",
        "two_tile_groups", "two_tile_groups_lora_capacity"])
def test_layer_forward_whole(cfg):
    inp = synth.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    p = moe.problem_of(cfg)
    buf = run_forward(p, dev)
    L_gpu, idx, g, prob = check_routing(buf, p, inp)
    D = check_dispatch(buf, p, idx, dev["x"])
    ref = oracle.moe_forward(f64(inp["x"]), None, f64(inp["w_gate"]), f64(inp["w_up"]),
                             f64(inp["w_down"]), p.k, p.cap_num, p.cap_den,
                             lora=lora64(inp.get("lora")), s=p.lora_scale, logits=L_gpu)
    n = D["n_kept"]
    assert relerr(f64(buf.h[:n]), ref["h"]) <= RTOL_FP
    g_row = ref["gates"].reshape(-1)[D["row_slot"]]
    assert relerr(f64(buf.y_perm[:n]), g_row[:, None] * ref["o"]) <= RTOL_FP
    assert relerr(f64(buf.y), ref["y"]) <= RTOL_FP
    assert abs(float(buf.aux.item()) - ref["aux"]) <= 1e-5 * abs(ref["aux"])
    # tokens whose slots were all dropped give exact zeros
    dropped_all = [t for t in range(p.T) if (D["slot_row"][t * p.k:(t + 1) * p.k] < 0).all()]
    if dropped_all:
        assert (buf.y[dropped_all].float().abs().sum() == 0).item()


@pytest.mark.parametrize("cfg", [
    synth.config("c1"),
    small_cfg(T=777, d=320, E=9, k=3, F=448, r=24, alpha=48.0, cap_num=1, cap_den=1),
    small_cfg(cap_num=5, cap_den=4, zipf_bias=True),
], ids=["c1", "ragged_lora_capacity", "small_capacity_bias"])
def test_fused_gather_matches_permuted_path(cfg):
    """The permute fused into the expert GEMMs (rows gathered from x by slot) gives the same
    bits as the separate gather + x_perm path (same products, same order)."""
    dev = to_dev(synth.make_inputs(cfg, "cpu"))
    p = moe.problem_of(cfg)
    a = run_forward(p, dev, gather=False)
    b = run_forward(p, dev, gather=True)
    n = int(a.n_kept_dropped[0].item())
    for name in ("slot_row", "offsets", "counts"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert torch.equal(a.h[:n], b.h[:n])
    assert torch.equal(a.y_perm[:n], b.y_perm[:n])
    assert torch.equal(a.y, b.y)


def test_forward_is_deterministic():
    cfg = small_cfg(cap_num=5, cap_den=4, r=16, alpha=32.0)
    dev = to_dev(synth.make_inputs(cfg, "cpu"))
    p = moe.problem_of(cfg)
    a = run_forward(p, dev)
    b = run_forward(p, dev)
    for name in ("logits", "topk_idx", "topk_gate", "partials", "slot_row", "x_perm", "h",
                 "y_perm", "y", "aux"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name


def _route_logits_case(case, T, E):
    g = torch.Generator().manual_seed(3)
    if case == "ties":
        L = torch.randint(0, 4, (T, E), generator=g).float()
        L[:10] = 0.0
    elif case == "one_lane":
        # every large logit sits on experts = 5 (mod 32): one lane owns the whole top-k
        L = torch.randn((T, E), generator=g)
        L[:, 5::32] += 100.0
    elif case == "rounded":
        # logits on a 0.1 grid: ties among the selected experts (broken by lower index)
        L = torch.round(torch.randn((T, E), generator=g) * 30) / 10
    elif case == "neg_zero":
        L = torch.zeros((T, E))
        L[:, ::2] = -0.0
        L[:, 7] = 1e-30
    else:
        L = torch.randn((T, E), generator=g) * 3
    return L


@pytest.mark.parametrize("case, E, k", [("ties", 40, 6), ("ties", 896, 16), ("one_lane", 896, 16),
                                        ("neg_zero", 896, 32), ("normal", 1024, 32),
                                        ("normal", 33, 32), ("normal", 896, 16), ("normal", 64, 4),
                                        ("rounded", 896, 16), ("rounded", 200, 8)])
def test_route_from_logits_exact_selection(case, E, k):
    T = 200
    L = _route_logits_case(case, T, E)
    p = moe.Problem(T, 64, E, k, 64)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    part = torch.empty((moe.moe_route_num_partials(p), E), dtype=torch.float32, device="cuda")
    moe.moe_route_from_logits(p, L.cuda(), idx, gate, part)
    torch.cuda.synchronize()
    L64 = L.double().numpy()
    ref = oracle.topk_select(L64, k)
    assert np.array_equal(idx.cpu().numpy(), ref)
    if case == "ties":
        assert (idx[:10].cpu().numpy() == np.arange(k)).all()
    prob = oracle.softmax(L64)
    gref = oracle.renormalised_gates(prob, ref)
    assert relerr(f64(gate), gref) <= 1e-5
    assert relerr(f64(part).sum(axis=0), prob.sum(axis=0)) <= 1e-5


def test_bad_expert_id_is_reported_not_faulted():
    cfg = small_cfg(T=64)
    dev = to_dev(synth.make_inputs(cfg, "cpu"))
    p = moe.problem_of(cfg)
    buf = moe.LayerBuffers(p, "cuda")
    idx = torch.zeros((p.T, p.k), dtype=torch.int32)
    idx[:, 1] = 1
    idx[5, 0] = p.E + 3
    idx[9, 1] = -7
    ws = torch.empty(moe.moe_dispatch_workspace_size(p), dtype=torch.uint8, device="cuda")
    moe.moe_dispatch(p, idx.cuda(), dev["x"], buf.counts, buf.offsets, buf.slot_row,
                     buf.row_slot, buf.n_kept_dropped, buf.x_perm, ws, buf.dev_status)
    torch.cuda.synchronize()
    assert int(buf.dev_status.item()) == 6  # MOE_ERR_BAD_INDEX
    sr = buf.slot_row.cpu().numpy()
    assert sr[5 * p.k] == -1 and sr[9 * p.k + 1] == -1
    assert buf.n_kept_dropped.cpu().tolist() == [p.T * p.k - 2, 2]


# ----------------------------------------------------------------------------- full sizes

def _full_workload(name, n_sample, gather=False):
    cfg = synth.config(name)
    inp = synth.make_inputs(cfg, "cuda")
    p = moe.problem_of(cfg)
    buf = run_forward(p, inp, gather=gather)
    L_gpu, idx, g, prob = check_routing(buf, p, inp)
    D = check_dispatch(buf, p, idx, None if gather else inp["x"])
    rng = np.random.default_rng(1)
    tokens = sorted(set([0, p.T - 1] + list(rng.choice(p.T, n_sample, replace=False))))
    ys = oracle_tokens(inp, p, tokens, idx, g, D["slot_row"])
    assert relerr(f64(buf.y[tokens]), ys) <= RTOL_FP
    aux_ref = oracle.aux_loss(D["counts"], prob, p.T, p.k, p.E)
    assert abs(float(buf.aux.item()) - aux_ref) <= 1e-5 * aux_ref
    return buf, D


def test_full_c2_full_fanout():
    buf, D = _full_workload("c2", 12)
    assert D["n_dropped"] == 0


def _whole_batch_oracle(name, gather):
    """The oracle's whole forward of a full-size workload on the GPU's logits (selection on
    identical fp32 inputs), its expert weights fetched one expert at a time."""
    cfg = synth.config(name)
    inp = synth.make_inputs(cfg, "cuda")
    p = moe.problem_of(cfg)
    buf = run_forward(p, inp, gather=gather)
    L_gpu, idx, g, prob = check_routing(buf, p, inp, full_logits_check=False)
    check_dispatch(buf, p, idx)
    ref = oracle.moe_forward(f64(inp["x"]), None, DeviceExperts(inp["w_gate"]),
                             DeviceExperts(inp["w_up"]), DeviceExperts(inp["w_down"]), p.k,
                             p.cap_num, p.cap_den, logits=L_gpu)
    return cfg, p, buf, ref


def test_full_c2_whole_batch():
    """c2 at full size against the oracle's whole forward: y on all 4096 tokens, and h and
    y_perm on every row of 48 experts (first, last, and a seeded sample)."""
    cfg, p, buf, ref = _whole_batch_oracle("c2", gather=True)
    assert relerr(f64(buf.y), ref["y"]) <= RTOL_FP
    D = ref["disp"]
    offs = D["offsets"]
    rng = np.random.default_rng(7)
    experts = sorted(set([0, p.E - 1] + list(rng.choice(np.arange(1, p.E - 1), 46, replace=False))))
    rows = np.concatenate([np.arange(offs[e], offs[e + 1]) for e in experts])
    assert len(experts) >= 32 and len(rows) > 32 * 64
    assert relerr(f64(buf.h[torch.from_numpy(rows).cuda()]), ref["h"][rows]) <= RTOL_FP
    g_row = ref["gates"].reshape(-1)[D["row_slot"][rows]]
    assert relerr(f64(buf.y_perm[torch.from_numpy(rows).cuda()]),
                  g_row[:, None] * ref["o"][rows]) <= RTOL_FP
    # per expert too, so that one bad expert cannot hide in the aggregate
    for e in experts:
        lo, hi = int(offs[e]), int(offs[e + 1])
        assert relerr(f64(buf.h[lo:hi]), ref["h"][lo:hi]) <= RTOL_FP, e


def test_full_c3_whole_batch():
    """c3 at full size (skewed routing, capacity 366, about 89 % of the slots dropped): y on
    all 16384 tokens against the oracle's whole forward, and the all-dropped tokens exactly
    zero."""
    cfg, p, buf, ref = _whole_batch_oracle("c3", gather=False)
    assert ref["C"] == 366 and ref["disp"]["n_dropped"] > 0
    assert relerr(f64(buf.y), ref["y"]) <= RTOL_FP
    sr = ref["disp"]["slot_row"].reshape(p.T, p.k)
    dropped_all = np.where((sr < 0).all(axis=1))[0]
    if len(dropped_all):
        assert float(buf.y[torch.from_numpy(dropped_all).cuda()].float().abs().max()) == 0.0


def test_full_c2_fused_gather():
    cfg = synth.config("c2")
    inp = synth.make_inputs(cfg, "cuda")
    p = moe.problem_of(cfg)
    a = run_forward(p, inp, gather=False)
    b = run_forward(p, inp, gather=True)
    assert torch.equal(a.y, b.y)


def test_full_c3_skewed_capacity():
    buf, D = _full_workload("c3", 6, gather=True)
    assert oracle.capacity(16384, 16, 896, 5, 4) == 366
    assert D["n_dropped"] > 0 and (D["kept"] <= 366).all()


def test_full_c4_lora_shard_sampled_rows():
    cfg = synth.config("c4")
    inp = synth.make_inputs(cfg, "cuda")
    p = moe.problem_of(cfg)
    rows = cfg.T
    h = torch.empty((rows, p.F), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((rows, p.d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(moe.moe_expert_ffn_workspace_size(p, rows), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_expert_ffn(p, rows, inp["x_perm"], inp["offsets"], inp["row_slot"], inp["gates"],
                       inp["w_gate"], inp["w_up"], inp["w_down"], inp["lora"], h, y, None, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    offs = inp["offsets"].cpu().numpy()
    W = ExpertCache(inp)
    rng = np.random.default_rng(2)
    sel, refs = [], []
    for e in range(p.E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        rr = sorted(set([lo, hi - 1, lo + 127, lo + 128, lo + 255, lo + 256, hi - 129] +
                        list(rng.integers(lo, hi, 2))))
        Wg, Wu, Wd, L = W(e)
        X = f64(inp["x_perm"][rr])
        o = oracle.expert_forward(X, Wg, Wu, Wd, L, p.lora_scale)[3]
        sel += rr
        refs.append(f64(inp["gates"][rr])[:, None] * o)
    assert relerr(f64(y[sel]), np.concatenate(refs)) <= RTOL_FP


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait that nothing will ever satisfy gives up after its limit, reports
    MOE_ERR_TIMEOUT through the status word, and the context keeps working."""
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_selftest_wait_timeout(st, 20)
    torch.cuda.synchronize()
    assert int(st.item()) == 5  # MOE_ERR_TIMEOUT
    # the same context still runs the layer correctly afterwards
    cfg = small_cfg(T=64)
    inp = synth.make_inputs(cfg, "cpu")
    buf = run_forward(moe.problem_of(cfg), to_dev(inp))
    assert int(buf.dev_status.item()) == 0
