"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks the oracle against something it cannot agree with by construction:
brute force, closed forms, special cases that reduce to a textbook routine computed with a
library call, invariants, finite differences, or the hand-worked example in
tests/golden/hand_example.json.  The mutation tests at the end plant plausible mistakes in
the oracle (on the CPU) and check that one of these pins catches each.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import moe_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def _rng(seed=0):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- selection (top-k)

def brute_topk(row, k):
    return sorted(range(len(row)), key=lambda e: (-row[e], e))[:k]


def check_topk_bruteforce():
    rng = _rng(1)
    for trial in range(3):
        # integer-valued logits force many exact ties
        L = rng.integers(0, 4, size=(60, 16)).astype(np.float64) if trial < 2 \
            else rng.standard_normal((60, 16))
        for k in (1, 5, 16):
            idx = oracle.topk_select(L, k)
            for t in range(L.shape[0]):
                assert list(idx[t]) == brute_topk(list(L[t]), k)


def test_topk_bruteforce():
    check_topk_bruteforce()


def test_topk_all_zero_logits():
    idx = oracle.topk_select(np.zeros((7, 10)), 4)
    assert (idx == np.arange(4)[None, :]).all()


def test_softmax_two_experts_is_sigmoid():
    L = np.array([[0.3, -1.2], [5.0, 5.0], [-30.0, 2.0]])
    p = oracle.softmax(L)
    for t in range(3):
        assert p[t, 0] == pytest.approx(1.0 / (1.0 + math.exp(-(L[t, 0] - L[t, 1]))), rel=1e-14)


def test_gates_sum_to_one_and_follow_rank():
    L = _rng(2).standard_normal((100, 32))
    idx, g, p = oracle.route(L, 6)
    assert np.allclose(g.sum(axis=1), 1.0, atol=1e-14)
    assert (np.diff(g, axis=1) <= 1e-15).all()
    # gates are ratios of exp of selected logits (softmax denominator cancels)
    Ls = np.take_along_axis(L, idx, axis=1)
    ref = np.exp(Ls) / np.exp(Ls).sum(axis=1, keepdims=True)
    assert np.allclose(g, ref, rtol=1e-13)


# ---------------------------------------------------------------- capacity and dispatch

def test_capacity_values():
    assert oracle.capacity(16384, 16, 896, 5, 4) == 366   # ceil(5*262144/3584) = 366
    assert oracle.capacity(4, 2, 4, 1, 1) == 2
    assert oracle.capacity(10, 3, 7, 5, 4) == math.ceil(1.25 * 30 / 7)
    assert oracle.capacity(4096, 16, 896, 0, 0) is None


def check_dispatch_invariants(T=200, E=12, k=3, seed=3):
    rng = _rng(seed)
    L = rng.standard_normal((T, E))
    idx = oracle.topk_select(L, k)
    for C in (None, 1, 7, oracle.capacity(T, k, E, 5, 4), T):
        D = oracle.dispatch(idx, E, C)
        cnt = np.bincount(idx.ravel(), minlength=E)
        assert (D["counts"] == cnt).all()
        assert D["counts"].sum() == T * k
        kept = cnt if C is None else np.minimum(cnt, C)
        assert (D["kept"] == kept).all()
        assert D["n_kept"] + D["n_dropped"] == T * k
        assert D["offsets"][0] == 0 and (np.diff(D["offsets"]) == kept).all()
        assert D["offsets"][E] == D["n_kept"]
        if C is None:
            assert D["n_dropped"] == 0
        # arrival position by its definition: earlier tokens routed to the same expert
        for t in range(T):
            for j in range(k):
                e = idx[t, j]
                pos = int(np.sum(idx[:t] == e))
                assert D["pos"][t, j] == pos
                row = D["slot_row"][t * k + j]
                if C is None or pos < C:
                    assert row == D["offsets"][e] + pos
                    assert D["row_slot"][row] == t * k + j
                else:
                    assert row == -1
        # rows of an expert hold strictly ascending tokens, all routed to that expert
        for e in range(E):
            toks = D["row_slot"][D["offsets"][e]:D["offsets"][e + 1]] // k
            assert (np.diff(toks) > 0).all()
            assert all(e in idx[t] for t in toks)


def test_dispatch_invariants():
    check_dispatch_invariants()


def test_dispatch_all_zero_logits_with_capacity():
    T, E, k = 50, 8, 3
    idx = oracle.topk_select(np.zeros((T, E)), k)
    C = oracle.capacity(T, k, E, 5, 4)  # ceil(187.5/8) = 24
    D = oracle.dispatch(idx, E, C)
    assert list(D["counts"]) == [T] * k + [0] * (E - k)
    assert list(D["kept"]) == [C] * k + [0] * (E - k)
    for e in range(k):
        toks = D["row_slot"][D["offsets"][e]:D["offsets"][e + 1]] // k
        assert list(toks) == list(range(C))


# ---------------------------------------------------------------- router bias
# The router adds a per-expert bias to the logits before both the softmax and the selection
# (the skewed-routing workload's Zipf bias goes through this term).

def check_bias_two_experts_closed_form():
    # integer inputs: every logit is exact, so p0 has the textbook two-class closed form
    # p0 = sigma((w0 - w1) . x + b0 - b1)
    x = np.array([[1.0, 2.0, -1.0], [0.0, -2.0, 3.0]])
    W = np.array([[1.0, 0.0, 1.0], [0.0, 1.0, 0.0]])
    b = np.array([0.5, -0.25])
    L = oracle.router_logits(x, W, b)
    # token 0: L = [1 + 0 - 1 + 0.5, 2 - 0.25] = [0.5, 1.75]; token 1: [3 + 0.5, -2 - 0.25]
    assert L.tolist() == [[0.5, 1.75], [3.5, -2.25]]
    idx, g, p = oracle.route(L, 1)
    assert idx[:, 0].tolist() == [1, 0]
    assert p[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(1.25)), rel=1e-14)
    assert p[1, 0] == pytest.approx(1.0 / (1.0 + math.exp(-5.75)), rel=1e-14)
    assert g[:, 0].tolist() == [1.0, 1.0]


def check_bias_makes_expert0_win_with_drops():
    # W_r = 0, b = [3, 0, 2, 1]: every token's logits are b, so each selects experts 0 and 2
    # (k = 2).  T = 6, E = 4, cf = 1 -> C = ceil(6 * 2 / 4) = 3: tokens 0..2 are kept on both
    # experts, tokens 3..5 dropped on both (arrival order).
    T, E, k, d = 6, 4, 2, 3
    x = _rng(9).standard_normal((T, d))
    b = np.array([3.0, 0.0, 2.0, 1.0])
    Wz = np.zeros((E, d))
    Wg = _rng(10).standard_normal((E, 2, d))
    Wu = _rng(11).standard_normal((E, 2, d))
    Wd = _rng(12).standard_normal((E, d, 2))
    out = oracle.moe_forward(x, Wz, Wg, Wu, Wd, k, 1, 1, bias=b)
    assert out["C"] == 3
    assert out["idx"].tolist() == [[0, 2]] * T
    D = out["disp"]
    assert D["counts"].tolist() == [6, 0, 6, 0]
    assert D["kept"].tolist() == [3, 0, 3, 0]
    assert D["offsets"].tolist() == [0, 3, 3, 6, 6]
    assert D["slot_row"].tolist() == [0, 3, 1, 4, 2, 5] + [-1] * 6
    assert (D["n_kept"], D["n_dropped"]) == (6, 6)
    # gates: e^3 / (e^3 + e^2) = sigma(1), and its complement
    s1 = 1.0 / (1.0 + math.exp(-1.0))
    assert np.allclose(out["gates"], [[s1, 1.0 - s1]] * T, rtol=1e-14)
    # aux = E * (f0 P0 + f2 P2) with f0 = f2 = 1/2, P = softmax(b) for every token
    Z = math.exp(3) + 1.0 + math.exp(2) + math.exp(1)
    assert out["aux"] == pytest.approx(4 * 0.5 * (math.exp(3) + math.exp(2)) / Z, rel=1e-14)
    # dropped tokens contribute nothing
    assert (out["y"][3:] == 0).all() and np.abs(out["y"][:3]).sum() > 0


def check_bias_shift_invariance():
    # adding one constant to every expert's bias (the Zipf normaliser) shifts all logits of a
    # token equally: the selection, probabilities and gates do not change
    rng = _rng(13)
    x = rng.standard_normal((50, 16))
    W = rng.standard_normal((24, 16))
    b = rng.standard_normal(24)
    i1, g1, p1 = oracle.route(oracle.router_logits(x, W, b), 5)
    i2, g2, p2 = oracle.route(oracle.router_logits(x, W, b - 7.25), 5)
    assert np.array_equal(i1, i2)
    assert np.allclose(p1, p2, rtol=1e-12, atol=0) and np.allclose(g1, g2, rtol=1e-12, atol=0)
    # ... while a bias that is not constant over experts does change them
    i3, _, p3 = oracle.route(oracle.router_logits(x, W, b + np.arange(24)), 5)
    assert not np.array_equal(i1, i3) and not np.allclose(p1, p3)


def test_bias_two_experts_closed_form():
    check_bias_two_experts_closed_form()


def test_bias_makes_expert0_win_with_drops():
    check_bias_makes_expert0_win_with_drops()


def test_bias_shift_invariance():
    check_bias_shift_invariance()


def test_zipf_bias_values():
    # b_e = 1.5 ln(w_{e+1}), w_q = q^-1.1 / sum_q' q'^-1.1: expert 0 hottest, strictly
    # decreasing, and exp(b / 1.5) sums to one
    from top_routing_grouped_gemm_gb300 import synth
    b = synth.zipf_bias(896).double().numpy()
    assert (np.diff(b) < 0).all()
    assert np.exp(b / 1.5).sum() == pytest.approx(1.0, rel=1e-5)
    assert b[1] - b[0] == pytest.approx(-1.5 * 1.1 * math.log(2.0), rel=1e-5)


# ---------------------------------------------------------------- overflow remapping
# A slot beyond its expert's capacity moves to the token's next-preferred experts (slot j's
# alternatives are the token's preference ranks j + k, j + 2k, ...) in rounds, each expert
# taking proposals in arrival order into its remaining capacity; the gate stays g_j.

def check_remap_hand_example_k2():
    # orders (descending logit): t0 [0,1,2,3,4,5], t1 [0,1,4,5,2,3], t2 [1,0,2,5,4,3]
    L = np.array([[6, 5, 4, 3, 2, 1], [6, 5, 1, 0, 4, 3], [5, 6, 4, 0, 1, 3]], float)
    order = oracle.topk_select(L, 4)
    assert order.tolist() == [[0, 1, 2, 3], [0, 1, 4, 5], [1, 0, 2, 5]]
    D = oracle.dispatch_remap(order, 2, 6, 1, 1)
    # pass 0 (C = 1): t0 takes e0 and e1; t1's and t2's slots all overflow.  Round 1: slot
    # (t, j) proposes order[t][j + 2]: t1 -> e4, e5 (taken); t2 -> e2 (taken), e5 (full).
    assert D["slot_expert"].tolist() == [0, 1, 4, 5, 2, -1]
    assert D["slot_pass"].tolist() == [0, 0, 1, 1, 1, -1]
    assert D["kept"].tolist() == [1, 1, 1, 0, 1, 1]
    assert D["offsets"].tolist() == [0, 1, 2, 3, 3, 4, 5]
    assert D["slot_row"].tolist() == [0, 1, 3, 4, 2, -1]
    assert (D["n_kept"], D["n_dropped"]) == (5, 1)
    assert D["counts"].tolist() == [3, 3, 0, 0, 0, 0]   # the original selection, pre-drop


def check_remap_hand_example_k1():
    L = np.array([[3, 2, 1, 0], [3, 2, 1, 0], [3, 2, 1, 0], [0, 1, 2, 3]], float)
    order = oracle.topk_select(L, 2)
    D0 = oracle.dispatch_remap(order, 1, 4, 1, 0)
    assert D0["slot_expert"].tolist() == [0, -1, -1, 3]
    D1 = oracle.dispatch_remap(order, 1, 4, 1, 1)
    # round 1: t1 and t2 both propose e1; t1 arrives first and takes it, t2 is dropped
    assert D1["slot_expert"].tolist() == [0, 1, -1, 3]
    assert D1["row_slot"].tolist() == [0, 1, 3]


def check_remap_invariants():
    rng = _rng(21)
    for trial in range(6):
        T, E, k = 40, 10, 2 + trial % 2
        R = 1 + trial % 3
        if (R + 1) * k > E:
            R = E // k - 1
        L = rng.integers(0, 5, size=(T, E)).astype(float)   # ties exercise the order key
        order = oracle.topk_select(L, (R + 1) * k)
        C = oracle.capacity(T, k, E, 1, 2 + trial % 3)
        D = oracle.dispatch_remap(order, k, E, C, R)
        D_prev = oracle.dispatch_remap(order, k, E, C, R - 1)
        se, sp = D["slot_expert"], D["slot_pass"]
        assert (D["kept"] <= C).all()
        assert D["n_dropped"] <= D_prev["n_dropped"]
        # remapping only adds placements: every slot kept by the plain rule stays put
        plain = oracle.dispatch(order[:, :k], E, C)
        assert (se[plain["slot_row"] >= 0] == order[:, :k].reshape(-1)[plain["slot_row"] >= 0]).all()
        for t in range(T):
            placed = [int(se[t * k + j]) for j in range(k) if se[t * k + j] >= 0]
            assert len(placed) == len(set(placed))   # never two slots of a token on one expert
            for j in range(k):
                if sp[t * k + j] >= 0:
                    assert se[t * k + j] == order[t, j + k * sp[t * k + j]]
        for e in range(E):
            rows = D["row_slot"][D["offsets"][e]:D["offsets"][e + 1]]
            assert (se[rows] == e).all()
            keys = [(int(sp[s]), int(s)) for s in rows]
            assert keys == sorted(keys)       # placement order: pass, then arrival
        # a slot the last round rejected had every one of its proposals refused by a full
        # expert
        for slot in np.where(se < 0)[0]:
            t, j = divmod(int(slot), k)
            for r in range(R + 1):
                assert D["kept"][order[t, j + k * r]] == C


def test_remap_hand_examples():
    check_remap_hand_example_k2()
    check_remap_hand_example_k1()


def test_remap_invariants():
    check_remap_invariants()


def test_remap_zero_rounds_is_the_dropping_rule():
    rng = _rng(22)
    for C in (1, 3, 7, None):
        L = rng.standard_normal((50, 8))
        idx = oracle.topk_select(L, 3)
        D0 = oracle.dispatch(idx, 8, C)
        D1 = oracle.dispatch_remap(idx, 3, 8, C, 0)
        for key in ("counts", "kept", "offsets", "slot_row", "row_slot", "n_kept", "n_dropped"):
            assert np.array_equal(np.asarray(D0[key]), np.asarray(D1[key])), key


def test_remap_ample_capacity_places_everything_in_pass0():
    rng = _rng(23)
    L = rng.standard_normal((30, 8))
    order = oracle.topk_select(L, 6)
    D = oracle.dispatch_remap(order, 2, 8, 30, 2)
    assert (D["slot_pass"] == 0).all() and D["n_dropped"] == 0


def test_remap_hand_example_layer_output():
    """The four-token worked example with one remap round: the slot (t2, rank 0) that the
    dropping rule loses moves to t2's third-ranked expert e3 (which holds one of its two
    places), keeping its gate 1/2; every other output is the dropping rule's."""
    G = json.load(open(os.path.join(HERE, "golden", "hand_example.json")))
    L = np.array(G["logits"], float)
    x = np.array(G["x"], float)
    E, d = 4, 2
    Wg = np.array([[[1.0, 0.0]]] * E)
    Wu = np.array([[[0.0, 1.0]]] * E)
    Wd = np.array([[[e + 1.0], [-(e + 1.0)]] for e in range(E)])
    out = oracle.moe_forward(x, None, Wg, Wu, Wd, 2, 1, 1, logits=L, remap_rounds=1)
    D = out["disp"]
    assert D["slot_expert"].tolist() == [0, 1, 0, 1, 3, 2, 2, 3]
    assert D["n_dropped"] == 0 and D["row_slot"][D["offsets"][3]:].tolist() == [7, 4]
    silu = lambda z: z / (1.0 + math.exp(-z))
    y2 = 0.5 * (4 + 3) * silu(0.5) * (-1.0)     # (E_3 + E_2)(x_2) / 2, E_e = (e+1) silu(x0) x1
    assert np.allclose(out["y"][2], [y2, -y2], rtol=1e-14)
    ref = np.array(G["expected"]["y"])
    assert np.allclose(out["y"][[0, 1, 3]], ref[[0, 1, 3]], rtol=1e-14)
    assert out["aux"] == pytest.approx(G["expected"]["aux"], rel=1e-14)  # counts pre-drop


# ---------------------------------------------------------------- aux loss

def test_aux_is_one_for_uniform_probabilities():
    rng = _rng(4)
    T, E, k = 40, 9, 3
    x = rng.standard_normal((T, 5))
    L = oracle.router_logits(x, np.zeros((E, 5)))
    idx, g, p = oracle.route(L, k)
    D = oracle.dispatch(idx, E, None)
    assert oracle.aux_loss(D["counts"], p, T, k, E) == pytest.approx(1.0, abs=1e-14)


def test_aux_is_one_for_uniform_counts():
    rng = _rng(5)
    T, E, k = 12, 6, 2
    p = oracle.softmax(rng.standard_normal((T, E)))
    counts = np.full(E, T * k // E)
    assert oracle.aux_loss(counts, p, T, k, E) == pytest.approx(1.0, abs=1e-14)


# ---------------------------------------------------------------- hand-worked example

def test_hand_example():
    G = json.load(open(os.path.join(HERE, "golden", "hand_example.json")))
    ex = G["expected"]
    e = math.e
    sig1 = 1.0 / (1.0 + math.exp(-1.0))
    # the stored numbers are the closed forms written in the fixture's derivation
    rows = [[e * e, e, 1, 1], [1, 1, 1, 1], [1, e ** 3, e ** 3, e], [e, 1, e * e, e * e]]
    P = [sum(r[i] / sum(r) for r in rows) / 4 for i in range(4)]
    assert np.allclose(ex["P"], P, rtol=1e-15)
    assert ex["gates"][0] == pytest.approx([sig1, 1 - sig1], rel=1e-15)
    assert ex["aux"] == pytest.approx(4 * sum(f * q for f, q in zip([2 / 8, 3 / 8, 2 / 8, 1 / 8], P)), rel=1e-15)

    T, E, k = G["T"], G["E"], G["k"]
    Wg = np.zeros((E, 1, 2)); Wg[:, 0, 0] = 1
    Wu = np.zeros((E, 1, 2)); Wu[:, 0, 1] = 1
    Wd = np.zeros((E, 2, 1))
    for q in range(E):
        Wd[q, :, 0] = [q + 1, -(q + 1)]
    out = oracle.moe_forward(np.array(G["x"], float), None, Wg, Wu, Wd, k,
                             G["cap_num"], G["cap_den"], logits=np.array(G["logits"], float))
    D = out["disp"]
    assert out["C"] == 2
    assert out["idx"].tolist() == ex["idx"]
    assert np.allclose(out["gates"], ex["gates"], rtol=1e-15)
    for key in ("counts", "kept", "offsets", "slot_row", "row_slot"):
        assert D[key].tolist() == ex[key], key
    assert D["n_kept"] == ex["n_kept"] and D["n_dropped"] == ex["n_dropped"]
    assert np.allclose(out["p"].mean(axis=0), ex["P"], rtol=1e-14)
    assert out["aux"] == pytest.approx(ex["aux"], rel=1e-14)
    assert np.allclose(out["y"], ex["y"], rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- expert network, LoRA

def _rand_layer(rng, T, d, E, F, r=0):
    x = rng.standard_normal((T, d))
    Wr = 0.3 * rng.standard_normal((E, d))
    Wg = 0.3 * rng.standard_normal((E, F, d))
    Wu = 0.3 * rng.standard_normal((E, F, d))
    Wd = 0.3 * rng.standard_normal((E, d, F))
    lora = None
    if r:
        lora = dict(A_g=0.3 * rng.standard_normal((E, r, d)), B_g=0.3 * rng.standard_normal((E, F, r)),
                    A_u=0.3 * rng.standard_normal((E, r, d)), B_u=0.3 * rng.standard_normal((E, F, r)),
                    A_d=0.3 * rng.standard_normal((E, r, F)), B_d=0.3 * rng.standard_normal((E, d, r)))
    return x, Wr, Wg, Wu, Wd, lora


def _torch_swiglu(x, Wg, Wu, Wd):
    """Textbook dense SwiGLU MLP computed with torch's own silu and matmul in float64."""
    x = torch.from_numpy(x)
    a = torch.nn.functional.silu(x @ torch.from_numpy(Wg).T) * (x @ torch.from_numpy(Wu).T)
    return (a @ torch.from_numpy(Wd).T).numpy()


def check_single_expert_is_dense_mlp():
    rng = _rng(6)
    x, Wr, Wg, Wu, Wd, _ = _rand_layer(rng, 9, 6, 1, 5)
    out = oracle.moe_forward(x, Wr, Wg, Wu, Wd, 1)
    assert np.allclose(out["gates"], 1.0)
    assert np.allclose(out["y"], _torch_swiglu(x, Wg[0], Wu[0], Wd[0]), rtol=1e-12, atol=1e-12)


def test_single_expert_is_dense_mlp():
    check_single_expert_is_dense_mlp()


def check_all_experts_is_dense_softmax_mixture():
    rng = _rng(7)
    T, d, E, F = 8, 6, 5, 4
    x, Wr, Wg, Wu, Wd, _ = _rand_layer(rng, T, d, E, F)
    out = oracle.moe_forward(x, Wr, Wg, Wu, Wd, E)
    tx = torch.from_numpy(x)
    p = torch.softmax(tx @ torch.from_numpy(Wr).T, dim=1).numpy()
    ref = sum(p[:, e:e + 1] * _torch_swiglu(x, Wg[e], Wu[e], Wd[e]) for e in range(E))
    assert np.allclose(out["y"], ref, rtol=1e-12, atol=1e-12)


def test_all_experts_is_dense_softmax_mixture():
    check_all_experts_is_dense_softmax_mixture()


def test_lora_with_zero_B_equals_base():
    rng = _rng(8)
    x, Wr, Wg, Wu, Wd, lora = _rand_layer(rng, 10, 6, 4, 5, r=2)
    for nm in ("B_g", "B_u", "B_d"):
        lora[nm] = np.zeros_like(lora[nm])
    a = oracle.moe_forward(x, Wr, Wg, Wu, Wd, 2, lora=lora, s=2.0)
    b = oracle.moe_forward(x, Wr, Wg, Wu, Wd, 2)
    assert np.array_equal(a["y"], b["y"])


def check_lora_merge_identity():
    """Adapter (W0, A, B) with scale s equals the merged weight W0 + s B A with no adapter
    ("Adapting Trillion-Parameter MoE Models ...", section 3: merging dW back into the base)."""
    rng = _rng(9)
    s = 1.75
    x, Wr, Wg, Wu, Wd, lora = _rand_layer(rng, 12, 6, 4, 5, r=3)
    a = oracle.moe_forward(x, Wr, Wg, Wu, Wd, 2, 5, 4, lora=lora, s=s)
    mg = Wg + s * np.einsum("efr,erd->efd", lora["B_g"], lora["A_g"])
    mu = Wu + s * np.einsum("efr,erd->efd", lora["B_u"], lora["A_u"])
    md = Wd + s * np.einsum("edr,erf->edf", lora["B_d"], lora["A_d"])
    b = oracle.moe_forward(x, Wr, mg, mu, md, 2, 5, 4)
    assert np.allclose(a["y"], b["y"], rtol=1e-12, atol=1e-12)


def test_lora_merge_identity():
    check_lora_merge_identity()


# ---------------------------------------------------------------- backward

def _loss_fixed(x, dy, idx, disp, Wr, Wg, Wu, Wd, lora, s, bias=None):
    L = oracle.router_logits(x, Wr, bias)
    out = oracle.moe_forward_fixed_routing(x, L, idx, disp, Wg, Wu, Wd, lora, s)
    return float(np.sum(dy * out["y"]))


def _fd(f, arr, h=1e-6):
    g = np.zeros_like(arr)
    it = np.nditer(arr, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = arr[i]
        arr[i] = old + h
        fp = f()
        arr[i] = old - h
        fm = f()
        arr[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


def _relerr(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def check_backward_finite_differences(caps=(0, 0)):
    rng = _rng(10)
    T, d, E, k, F, r, s = 3, 8, 4, 2, 4, 2, 1.5
    x, Wr, Wg, Wu, Wd, lora = _rand_layer(rng, T, d, E, F, r)
    dy = rng.standard_normal((T, d))
    fwd = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k, caps[0], caps[1], lora=lora, s=s)
    if caps[1]:
        assert fwd["disp"]["n_dropped"] > 0
    bwd = oracle.moe_backward(fwd, x, dy, Wr, Wg, Wu, Wd, lora, s)
    f = lambda: _loss_fixed(x, dy, fwd["idx"], fwd["disp"], Wr, Wg, Wu, Wd, lora, s)
    assert _relerr(bwd["dx"], _fd(f, x)) < 1e-7
    for nm in ("A_g", "B_g", "A_u", "B_u", "A_d", "B_d"):
        assert _relerr(bwd["d" + nm], _fd(f, lora[nm])) < 1e-7, nm


@pytest.mark.parametrize("caps", [(0, 0), (1, 2)])
def test_backward_finite_differences(caps):
    check_backward_finite_differences(caps)


def test_backward_components_finite_differences():
    """dx splits into the expert path (gates held fixed) and the gate path (expert
    outputs held fixed); each matches its own finite difference."""
    rng = _rng(11)
    T, d, E, k, F, r, s = 4, 6, 5, 3, 4, 2, 2.0
    x, Wr, Wg, Wu, Wd, lora = _rand_layer(rng, T, d, E, F, r)
    dy = rng.standard_normal((T, d))
    fwd = oracle.moe_forward(x, Wr, Wg, Wu, Wd, k, lora=lora, s=s)
    bwd = oracle.moe_backward(fwd, x, dy, Wr, Wg, Wu, Wd, lora, s)
    idx, D = fwd["idx"], fwd["disp"]
    g0, o0 = fwd["gates"], fwd["o"]

    def expert_path():
        xp = oracle.permute(x, D["row_slot"], k)
        o = np.zeros_like(o0)
        for e in range(E):
            lo, hi = D["offsets"][e], D["offsets"][e + 1]
            if hi > lo:
                L = {n: v[e] for n, v in lora.items()}
                o[lo:hi] = oracle.expert_forward(xp[lo:hi], Wg[e], Wu[e], Wd[e], L, s)[3]
        return float(np.sum(dy * oracle.combine(o, g0, D["slot_row"], T, k)))

    def gate_path():
        g = oracle.renormalised_gates(oracle.softmax(oracle.router_logits(x, Wr)), idx)
        return float(np.sum(dy * oracle.combine(o0, g, D["slot_row"], T, k)))

    assert _relerr(bwd["dx_expert"], _fd(expert_path, x)) < 1e-7
    assert _relerr(bwd["dx_gate"], _fd(gate_path, x)) < 1e-7


def test_route_backward_vanishes_off_selection():
    rng = _rng(12)
    L = rng.standard_normal((20, 9))
    idx, g, p = oracle.route(L, 3)
    dl = oracle.route_backward(p, idx, g, rng.standard_normal((20, 3)), np.ones((20, 3)))
    mask = np.ones_like(dl, dtype=bool)
    np.put_along_axis(mask, idx, False, axis=1)
    assert np.abs(dl[mask]).max() < 1e-15
    # gates depend only on logit differences: gradient sums to zero per token
    assert np.abs(dl.sum(axis=1)).max() < 1e-14


# ---------------------------------------------------------------- planted mistakes

def _expect_failure(check, *args):
    with pytest.raises(AssertionError):
        check(*args)


def test_mutation_tie_break_caught(monkeypatch):
    def ties_to_higher_index(L, k):
        L = np.asarray(L, float)
        E = L.shape[1]
        return (E - 1 - np.argsort(-L[:, ::-1], axis=1, kind="stable"))[:, :k]
    monkeypatch.setattr(O, "topk_select", ties_to_higher_index)
    monkeypatch.setattr(oracle, "topk_select", ties_to_higher_index)
    _expect_failure(check_topk_bruteforce)


def test_mutation_silu_sign_caught(monkeypatch):
    monkeypatch.setattr(O, "silu", lambda z: np.asarray(z, float) / (1.0 + np.exp(np.asarray(z, float))))
    _expect_failure(check_single_expert_is_dense_mlp)


def test_mutation_lora_scale_dropped_caught(monkeypatch):
    orig = O.lora_linear
    monkeypatch.setattr(O, "lora_linear", lambda X, W, A=None, B=None, s=0.0: orig(X, W, A, B, 1.0))
    _expect_failure(check_lora_merge_identity)


def test_mutation_capacity_off_by_one_caught(monkeypatch):
    orig = O.dispatch
    monkeypatch.setattr(O, "dispatch", lambda idx, E, C: orig(idx, E, None if C is None else C + 1))
    monkeypatch.setattr(oracle, "dispatch", O.dispatch)
    _expect_failure(check_dispatch_invariants)


def test_mutation_transposed_down_weight_caught(monkeypatch):
    orig = O.expert_forward

    def wrong(X, Wg, Wu, Wd, lora=None, s=0.0):
        a_g, a_u, h, o = orig(X, Wg, Wu, Wd, lora, s)
        return a_g, a_u, h, o[:, ::-1]
    monkeypatch.setattr(O, "expert_forward", wrong)
    _expect_failure(check_all_experts_is_dense_softmax_mixture)


def test_mutation_backward_dropped_lora_term_caught(monkeypatch):
    orig = O.expert_backward

    def wrong(X, dO, Wg, Wu, Wd, lora=None, s=0.0):
        dX, g = orig(X, dO, Wg, Wu, Wd, lora, s)
        return dX, {n: (v * 0.5 if n == "A_d" else v) for n, v in g.items()}
    monkeypatch.setattr(O, "expert_backward", wrong)
    _expect_failure(check_backward_finite_differences)


def test_mutation_bias_sign_flipped_caught(monkeypatch):
    def minus_bias(x, w_router, bias=None):
        L = np.asarray(x, float) @ np.asarray(w_router, float).T
        return L if bias is None else L - np.asarray(bias, float)[None, :]
    monkeypatch.setattr(O, "router_logits", minus_bias)
    monkeypatch.setattr(oracle, "router_logits", minus_bias)
    _expect_failure(check_bias_two_experts_closed_form)
    _expect_failure(check_bias_makes_expert0_win_with_drops)


def test_mutation_bias_dropped_caught(monkeypatch):
    def no_bias(x, w_router, bias=None):
        return np.asarray(x, float) @ np.asarray(w_router, float).T
    monkeypatch.setattr(O, "router_logits", no_bias)
    monkeypatch.setattr(oracle, "router_logits", no_bias)
    _expect_failure(check_bias_two_experts_closed_form)
    _expect_failure(check_bias_makes_expert0_win_with_drops)


def test_mutation_bias_on_selection_only_caught(monkeypatch):
    # a bias that steers the selection but is left out of the gate probabilities (the
    # selection-only variant some routers use) changes the gates of the worked example
    orig_fixed = O.moe_forward_fixed_routing

    def gates_without_bias(x, logits, idx, disp, Wg, Wu, Wd, lora=None, s=0.0):
        return orig_fixed(x, logits - np.array([3.0, 0.0, 2.0, 1.0])[None, :], idx, disp,
                          Wg, Wu, Wd, lora, s)
    monkeypatch.setattr(O, "moe_forward_fixed_routing", gates_without_bias)
    _expect_failure(check_bias_makes_expert0_win_with_drops)


def test_mutation_remap_alternative_rank_caught(monkeypatch):
    # alternatives taken as the next ranks j + r (shared between a token's slots) instead
    # of j + k r
    orig = O.dispatch_remap

    def wrong(order, k, E, C, rounds):
        order = np.asarray(order).copy()
        T = order.shape[0]
        fixed = order.copy()
        for r in range(1, rounds + 1):
            for j in range(k):
                fixed[:, j + k * r] = order[:, min(j + r, order.shape[1] - 1)]
        return orig(fixed, k, E, C, rounds)
    monkeypatch.setattr(O, "dispatch_remap", wrong)
    monkeypatch.setattr(oracle, "dispatch_remap", wrong)
    _expect_failure(check_remap_hand_example_k2)


def test_mutation_remap_ignores_capacity_caught(monkeypatch):
    orig = O.dispatch_remap
    monkeypatch.setattr(O, "dispatch_remap",
                        lambda order, k, E, C, rounds: orig(order, k, E, None if rounds else C,
                                                            rounds))
    monkeypatch.setattr(oracle, "dispatch_remap", O.dispatch_remap)
    _expect_failure(check_remap_invariants)
