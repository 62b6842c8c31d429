"""The expert-parallel forward on the GPU through the C ABI: P ranks held in one process and
run in lockstep on one device (the exchange moves tensors directly, so no kernel waits for
another rank).  Each rank routes its own slice of the batch and computes only its E/P
experts; the gathered result must be the single-device layer's on the whole batch, bit for
bit (same routing, same kept slots in global arrival order, row for row the same expert
products, same summation order in combine)."""

import numpy as np
import pytest
import torch

import oracle
from top_routing_grouped_gemm_gb300 import ep, moe, synth
from parity_util import RTOL_FP, f64, lora64, relerr, run_forward, to_dev

pytestmark = pytest.mark.gpu


def _ep_run(cfg, dev, P, chunks=1):
    T = cfg.T // P
    El = cfg.E // P
    ranks = []
    for r in range(P):
        sl = slice(r * El, (r + 1) * El)
        lora = None if dev.get("lora") is None else {n: v[sl] for n, v in dev["lora"].items()}
        ranks.append(ep.EPRank(rank=r, x=dev["x"][r * T:(r + 1) * T], w_gate=dev["w_gate"][sl],
                               w_up=dev["w_up"][sl], w_down=dev["w_down"][sl], lora=lora))
    p = moe.Problem(T=T, d=cfg.d, E=cfg.E, k=cfg.k, F=cfg.F, r=cfg.r,
                    lora_scale=cfg.lora_scale, cap_num=cfg.cap_num, cap_den=cfg.cap_den)
    outs = ep.ep_forward(p, ranks, dev["w_router"], dev.get("bias"), ep.LocalExchange(P),
                         ep.CudaBackend(), n_chunks=chunks)
    torch.cuda.synchronize()
    for o in outs:
        assert int(o["state"].dev_status.item()) == 0
    return outs


CASES = [
    (2, synth.MoEConfig("ep_small", T=512, d=192, E=8, k=2, F=192)),
    (4, synth.MoEConfig("ep_capacity", T=1024, d=256, E=16, k=4, F=128, cap_num=5, cap_den=4,
                        zipf_bias=True)),
    (2, synth.MoEConfig("ep_lora", T=256, d=128, E=12, k=3, F=192, r=16, alpha=32.0,
                        cap_num=1, cap_den=1)),
    (8, synth.MoEConfig("ep_many_ranks_few_tokens", T=64, d=128, E=64, k=8, F=64,
                        cap_num=1, cap_den=2)),
]


@pytest.mark.parametrize("chunks", [1, 3])
@pytest.mark.parametrize("P, cfg", CASES, ids=[c.name for _, c in CASES])
def test_ep_lockstep_equals_single_device(P, cfg, chunks):
    inp = synth.make_inputs(cfg, "cpu")
    dev = to_dev(inp)
    buf = run_forward(moe.problem_of(cfg), dev)
    outs = _ep_run(cfg, dev, P, chunks)
    T = cfg.T // P
    for r, o in enumerate(outs):
        st = o["state"]
        assert torch.equal(st.topk_idx, buf.topk_idx[r * T:(r + 1) * T]), r
        kept_ep = sum(int(pl.kept[r].sum()) for pl in o["plans"])
        kept_1 = int((buf.slot_row[r * T * cfg.k:(r + 1) * T * cfg.k] >= 0).sum().item())
        assert kept_ep == kept_1, r
        assert torch.equal(o["y"], buf.y[r * T:(r + 1) * T]), r
        assert abs(float(o["aux"].item()) - float(buf.aux.item())) <= 1e-6 * float(buf.aux.item())
    if cfg.cap_den:
        assert int(buf.n_kept_dropped[1].item()) > 0


@pytest.mark.parametrize("chunks", [2, 4])
def test_single_device_chunk_pipeline_c3(chunks):
    """P = 1 with chunks: the single-device layer with each chunk's dispatch overlapping the
    previous chunk's expert GEMMs (c3: capacity decided across chunks in arrival order), bit
    for bit the unchunked layer."""
    cfg = synth.config("c3")
    dev = synth.make_inputs(cfg, "cuda")
    buf = run_forward(moe.problem_of(cfg), dev, gather=False)
    outs = _ep_run(cfg, dev, 1, chunks)
    assert torch.equal(outs[0]["y"], buf.y)
    kept = sum(int(pl.kept.sum()) for pl in outs[0]["plans"])
    assert kept == int(buf.n_kept_dropped[0].item())


def test_ep_c2_four_ranks_against_oracle_sampled():
    """c2 (896 experts, top-16) split over 4 ranks of 224 experts: bit-exact against the
    single-device layer, and the oracle on sampled tokens of every rank."""
    cfg = synth.config("c2")
    P = 4
    dev = synth.make_inputs(cfg, "cuda")
    buf = run_forward(moe.problem_of(cfg), dev)
    outs = _ep_run(cfg, dev, P)
    T = cfg.T // P
    y = torch.cat([o["y"] for o in outs])
    assert torch.equal(y, buf.y)
    L = f64(buf.logits)
    idx = oracle.topk_select(L, cfg.k)
    g = oracle.renormalised_gates(oracle.softmax(L), idx)
    rng = np.random.default_rng(3)
    tokens = sorted(set(int(t) for r in range(P) for t in rng.integers(r * T, (r + 1) * T, 3)))
    from parity_util import oracle_tokens
    sr = buf.slot_row.cpu().numpy()
    ys = oracle_tokens(dev, moe.problem_of(cfg), tokens, idx, g, sr)
    assert relerr(f64(y[tokens]), ys) <= RTOL_FP
