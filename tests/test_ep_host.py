"""The expert-parallel exchange on the CPU: the host plan (arrival bases, capacity, split
sizes) against hand-worked values, the in-process exchange, and world_size-2 gloo ranks
running the whole EP forward (with the oracle as each rank's compute backend), whose
gathered outputs and kept slots must equal the oracle's on the whole batch."""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))

import oracle
from top_routing_grouped_gemm_gb300 import ep, moe, synth
from ep_oracle_backend import OracleBackend


def test_plan_hand_example():
    # P = 2 ranks, E = 4 experts (2 per rank), capacity C = 3
    cnt = np.array([[2, 0, 4, 1],
                    [3, 1, 0, 2]])
    plan = ep.plan_exchange(cnt, 3)
    assert plan.base.tolist() == [[0, 0, 0, 0], [2, 0, 4, 1]]
    # rank 1's expert-0 slots start at 2: one of its 3 fits; expert 2 is full (4 >= 3)
    assert plan.kept.tolist() == [[2, 0, 3, 1], [1, 1, 0, 2]]
    assert plan.send_splits(0) == [2, 4] and plan.send_splits(1) == [2, 2]
    assert plan.recv_splits(0) == [2, 2] and plan.recv_splits(1) == [4, 2]
    assert plan.kept_local(1).tolist() == [[3, 1], [0, 2]]
    # unlimited capacity keeps every slot
    assert (ep.plan_exchange(cnt, None).kept == cnt).all()


def test_plan_matches_single_device_capacity():
    """kept over ranks = what one device keeps on the concatenated batch."""
    rng = np.random.default_rng(0)
    P, T, E, k = 4, 30, 8, 3
    L = rng.standard_normal((P * T, E))
    idx = oracle.topk_select(L, k)
    C = oracle.capacity(P * T, k, E, 5, 4)
    D = oracle.dispatch(idx, E, C)
    cnt = np.stack([np.bincount(idx[r * T:(r + 1) * T].ravel(), minlength=E) for r in range(P)])
    plan = ep.plan_exchange(cnt, C)
    assert (plan.kept.sum(axis=0) == D["kept"]).all()
    assert ep.capacity(P * T, k, E, 5, 4) == C


def test_chunk_plans_follow_global_arrival_order():
    """Chunks of ranks: the bases follow (rank, chunk, token) order, so the kept totals per
    expert are the single-device ones on the concatenated batch."""
    rng = np.random.default_rng(1)
    P, n, T, E, k = 2, 3, 24, 6, 2
    L = rng.standard_normal((P * T, E))
    idx = oracle.topk_select(L, k)
    C = oracle.capacity(P * T, k, E, 1, 2)
    D = oracle.dispatch(idx, E, C)
    bounds = ep.chunk_bounds(T, n)
    cnt = np.zeros((P, len(bounds), E), dtype=np.int64)
    for r in range(P):
        for c, (t0, t1) in enumerate(bounds):
            cnt[r, c] = np.bincount(idx[r * T + t0:r * T + t1].ravel(), minlength=E)
    plans = ep.plan_chunks(cnt, C)
    kept = sum(pl.kept for pl in plans)
    assert (kept.sum(axis=0) == D["kept"]).all()
    assert plans[1].base[0].tolist() == cnt[0, 0].tolist()
    assert plans[0].base[1].tolist() == cnt[0].sum(axis=0).tolist()


def test_chunk_bounds():
    assert ep.chunk_bounds(100, 3) == [(0, 40), (40, 80), (80, 100)]
    assert ep.chunk_bounds(5, 8) == [(0, 1), (1, 2), (2, 3), (3, 4), (4, 5)]
    assert ep.chunk_bounds(64, 1) == [(0, 64)]


def test_local_exchange_all_to_all():
    X = ep.LocalExchange(2)
    a = torch.arange(5).float()[:, None]
    b = 10 + torch.arange(3).float()[:, None]
    out = X.all_to_all([a, b], [[2, 3], [1, 2]], [[2, 1], [3, 2]])
    assert out[0].ravel().tolist() == [0, 1, 10]
    assert out[1].ravel().tolist() == [2, 3, 4, 11, 12]


def _inputs(cfg, P):
    """Seeded inputs of a P-rank batch (P * T tokens) in float64 (values exact in bf16)."""
    inp = synth.make_inputs(cfg, "cpu")
    f64 = lambda t: None if t is None else t.double()
    out = {n: f64(v) for n, v in inp.items() if n != "lora"}
    if "lora" in inp:
        out["lora"] = {n: v.double() for n, v in inp["lora"].items()}
    return out


def _ep_rank_run(rank, P, cfg, inp, xchg):
    T = cfg.T // P
    El = cfg.E // P
    sl = slice(rank * El, (rank + 1) * El)
    lora = None if "lora" not in inp else {n: v[sl] for n, v in inp["lora"].items()}
    r = ep.EPRank(rank=rank, x=inp["x"][rank * T:(rank + 1) * T], w_gate=inp["w_gate"][sl],
                  w_up=inp["w_up"][sl], w_down=inp["w_down"][sl], lora=lora)
    return r


def _problem(cfg, P):
    return moe.Problem(T=cfg.T // P, d=cfg.d, E=cfg.E, k=cfg.k, F=cfg.F, r=cfg.r,
                       lora_scale=cfg.lora_scale, cap_num=cfg.cap_num, cap_den=cfg.cap_den)


def _oracle_whole(cfg, inp):
    lora = None if "lora" not in inp else {n: v.numpy() for n, v in inp["lora"].items()}
    return oracle.moe_forward(inp["x"].numpy(), inp["w_router"].numpy(), inp["w_gate"].numpy(),
                              inp["w_up"].numpy(), inp["w_down"].numpy(), cfg.k, cfg.cap_num,
                              cfg.cap_den, bias=None if inp.get("bias") is None else
                              inp["bias"].numpy(), lora=lora, s=cfg.lora_scale)


CASES = [
    synth.MoEConfig("ep_small", T=96, d=64, E=8, k=2, F=64),
    synth.MoEConfig("ep_capacity", T=120, d=64, E=8, k=3, F=64, cap_num=5, cap_den=4,
                    zipf_bias=True),
    synth.MoEConfig("ep_lora", T=64, d=64, E=4, k=2, F=64, r=8, alpha=16.0, cap_num=1,
                    cap_den=1),
]


def _check_rank(cfg, P, rank, out, ref):
    T = cfg.T // P
    y = out["y"].numpy()
    assert np.allclose(y, ref["y"][rank * T:(rank + 1) * T], rtol=1e-12, atol=1e-12)
    # the kept slots of this rank's tokens are the oracle's kept slots of those tokens
    kept = sum(int(pl.kept[rank].sum()) for pl in out["plans"])
    ref_sr = ref["disp"]["slot_row"][rank * T * cfg.k:(rank + 1) * T * cfg.k]
    assert kept == int((ref_sr >= 0).sum())
    assert np.array_equal(out["state"].topk_idx.numpy(), ref["idx"][rank * T:(rank + 1) * T])
    assert abs(float(out["aux"][0]) - ref["aux"]) <= 1e-12 * abs(ref["aux"])


@pytest.mark.parametrize("chunks", [1, 3])
@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_local_exchange_two_ranks_equal_whole_batch_oracle(cfg, chunks):
    P = 2
    inp = _inputs(cfg, P)
    ref = _oracle_whole(cfg, inp)
    xchg = ep.LocalExchange(P)
    ranks = [_ep_rank_run(r, P, cfg, inp, xchg) for r in range(P)]
    outs = ep.ep_forward(_problem(cfg, P), ranks, inp["w_router"], inp.get("bias"), xchg,
                         OracleBackend(), n_chunks=chunks)
    for r, out in enumerate(outs):
        _check_rank(cfg, P, r, out, ref)
    if cfg.cap_den:
        assert ref["disp"]["n_dropped"] > 0


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _gloo_rank(rank, world, port, case, res):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, HERE)
    import torch.distributed as dist
    from top_routing_grouped_gemm_gb300 import ep as ep_
    from ep_oracle_backend import OracleBackend as OB
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = CASES[case]
        inp = _inputs(cfg, world)
        xchg = ep_.DistExchange()
        r = _ep_rank_run(rank, world, cfg, inp, xchg)
        out = ep_.ep_forward(_problem(cfg, world), [r], inp["w_router"], inp.get("bias"), xchg,
                             OB(), n_chunks=1 + case)[0]
        ref = _oracle_whole(cfg, inp)
        _check_rank(cfg, world, rank, out, ref)
        res[rank] = "ok"
    except Exception as e:  # reported to the parent
        res[rank] = repr(e)
    finally:
        dist.barrier()
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [0, 1, 2], ids=[c.name for c in CASES])
def test_gloo_two_ranks_equal_whole_batch_oracle(case):
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        res = mgr.dict()
        mp.start_processes(_gloo_rank, args=(world, _free_port(), case, res), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(res)
    assert res == {0: "ok", 1: "ok"}, res
