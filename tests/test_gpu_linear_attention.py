"""GPU parity of the chunked gated delta-rule linear attention against the fp64 token-by-
token recurrence of the oracle, through the C ABI: outputs, the final state and the state at
every chunk start, on ragged lengths, both key/value widths, strong and weak decay, and with
an initial state."""

import numpy as np
import pytest
import torch

from oracle import linear_attention as LA
from top_routing_grouped_gemm_gb300 import moe, synth
from parity_util import f64, relerr

pytestmark = pytest.mark.gpu

RTOL_O = 5e-3      # o is rounded once to bf16
RTOL_S = 1e-4      # the fp32 state (the scan's products: two bf16 pieces per fp32 operand)


def run_gdr(cfg, inp, checkpoints=False, keep_w=False):
    B, T, H, dk, dv = cfg.B, cfg.T, cfg.H, cfg.dk, cfg.dv
    dev = {n: (None if t is None else t.cuda()) for n, t in inp.items()}
    o = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device="cuda")
    ST = torch.empty((B, H, dv, dk), dtype=torch.float32, device="cuda")
    nch = (T + 63) // 64
    Sc = torch.empty((B, H, nch, dv, dk), dtype=torch.float32, device="cuda") if checkpoints else None
    Wc = torch.empty((B, H, nch, 64, dv), dtype=torch.float32, device="cuda") if keep_w else None
    ws = torch.empty(moe.moe_gdr_workspace_size(B, T, H, dk, dv), dtype=torch.uint8, device="cuda")
    moe.moe_gdr_forward(B, T, H, dk, dv, dev["q"], dev["k"], dev["v"], dev["beta"], dev["g"],
                        dev["S0"], dk ** -0.5, o, ST, Sc, ws, W_chunks=Wc)
    torch.cuda.synchronize()
    assert moe.moe_gdr_device_status() == moe.MOE_OK
    if keep_w:
        return o, ST, Sc, Wc
    return o, ST, Sc


def ref_of(inp, T=None):
    sl = slice(None) if T is None else slice(0, T)
    return LA.gated_delta_rule(f64(inp["q"][:, sl]), f64(inp["k"][:, sl]), f64(inp["v"][:, sl]),
                               f64(inp["beta"][:, sl]), f64(inp["g"][:, sl]),
                               S0=f64(inp["S0"]))


CASES = [
    synth.la_config("la_small"),
    synth.LAConfig("la_one_chunk", B=1, T=64, H=2, dk=64, dv=128),
    synth.LAConfig("la_ragged_64x64", B=1, T=333, H=3, dk=64, dv=64, with_state=True),
    synth.LAConfig("la_dk128_dv64", B=1, T=130, H=2, dk=128, dv=64),
    synth.LAConfig("la_one_token", B=3, T=1, H=1),
]


@pytest.mark.parametrize("cfg", CASES, ids=[c.name for c in CASES])
def test_gdr_forward_whole(cfg):
    inp = synth.make_la_inputs(cfg)
    o, ST, Sc = run_gdr(cfg, inp, checkpoints=True)
    o_ref, S_ref = ref_of(inp)
    assert relerr(f64(o), o_ref) <= RTOL_O
    assert relerr(f64(ST), S_ref) <= RTOL_S
    # the state at the start of chunk c is the recurrence's state after 64 c tokens
    nch = (cfg.T + 63) // 64
    for c in sorted({0, nch // 2, nch - 1}):
        if c == 0:
            ref_c = np.zeros_like(S_ref) if inp["S0"] is None else f64(inp["S0"])
        else:
            ref_c = ref_of(inp, 64 * c)[1]
        assert relerr(f64(Sc[:, :, c]), ref_c) <= RTOL_S or np.abs(ref_c).max() == 0, c


def test_gdr_strong_decay_and_full_writes():
    """Fast forgetting (alpha down to e^-3) and beta = 1 writes: the chunk factors span many
    orders of magnitude of decay, and a full-strength write must be retrieved exactly."""
    cfg = synth.LAConfig("la_decay", B=1, T=300, H=2, dk=128, dv=128)
    inp = synth.make_la_inputs(cfg)
    gen = torch.Generator().manual_seed(5)
    inp["g"] = -3.0 * torch.rand((1, 300, 2), generator=gen)
    inp["beta"][:, 100] = 1.0
    inp["q"][:, 100] = inp["k"][:, 100]
    o, ST, _ = run_gdr(cfg, inp)
    o_ref, S_ref = ref_of(inp)
    assert relerr(f64(o), o_ref) <= RTOL_O
    assert relerr(f64(ST), S_ref) <= RTOL_S
    # retrieval right after the beta = 1 write: o = scale v
    assert relerr(f64(o[:, 100]), (128 ** -0.5) * f64(inp["v"][:, 100])) <= RTOL_O


def test_gdr_long_sequence_sampled_heads():
    """The bench shape (one sequence of 32768 tokens, 16 heads) on the GPU; two heads checked
    against the recurrence over the whole sequence."""
    cfg = synth.la_config("la")
    inp = synth.make_la_inputs(cfg)
    o, ST, _ = run_gdr(cfg, inp)
    for h in (0, cfg.H - 1):
        sub = {n: (None if t is None else t[:, :, h:h + 1]) for n, t in inp.items() if n != "S0"}
        sub["S0"] = None
        o_ref, S_ref = ref_of(sub)
        assert relerr(f64(o[:, :, h:h + 1]), o_ref) <= RTOL_O, h
        assert relerr(f64(ST[:, h:h + 1]), S_ref) <= 10 * RTOL_S, h


# ---------------------------------------------------------------- backward

RTOL_G = 5e-3


def run_gdr_bwd(cfg, inp, d_o, dST, keep_w=False):
    B, T, H, dk, dv = cfg.B, cfg.T, cfg.H, cfg.dk, cfg.dv
    Wc = None
    if keep_w:
        _, _, Sc, Wc = run_gdr(cfg, inp, checkpoints=True, keep_w=True)
    else:
        _, _, Sc = run_gdr(cfg, inp, checkpoints=True)
    dev = {n: (None if t is None else t.cuda()) for n, t in inp.items()}
    out = {"dq": torch.empty((B, T, H, dk), device="cuda"),
           "dk": torch.empty((B, T, H, dk), device="cuda"),
           "dv": torch.empty((B, T, H, dv), device="cuda"),
           "dbeta": torch.empty((B, T, H), device="cuda"),
           "dg": torch.empty((B, T, H), device="cuda"),
           "dS0": torch.empty((B, H, dv, dk), device="cuda")}
    ws = torch.empty(moe.moe_gdr_backward_workspace_size(B, T, H, dk, dv), dtype=torch.uint8,
                     device="cuda")
    moe.moe_gdr_backward(B, T, H, dk, dv, dev["q"], dev["k"], dev["v"], dev["beta"], dev["g"],
                         dk ** -0.5, d_o.cuda(), None if dST is None else dST.cuda(), Sc,
                         out["dq"], out["dk"], out["dv"], out["dbeta"], out["dg"], out["dS0"], ws,
                         W_chunks=Wc)
    torch.cuda.synchronize()
    assert moe.moe_gdr_device_status() == moe.MOE_OK
    return out


BWD_CASES = [
    synth.LAConfig("la_bwd_small", B=1, T=200, H=2, dk=128, dv=128, with_state=True),
    synth.LAConfig("la_bwd_64x128", B=2, T=130, H=1, dk=64, dv=128),
    synth.LAConfig("la_bwd_128x64_one_chunk", B=1, T=64, H=3, dk=128, dv=64, with_state=True),
    synth.LAConfig("la_bwd_ragged", B=1, T=333, H=2, dk=64, dv=64),
    # 16 chunks (the last of 40 tokens): the backward scan's chain over many steps
    synth.LAConfig("la_bwd_long", B=1, T=1000, H=2, dk=128, dv=128, with_state=True),
]


@pytest.mark.parametrize("with_dST", [False, True])
@pytest.mark.parametrize("cfg", BWD_CASES, ids=[c.name for c in BWD_CASES])
def test_gdr_backward_whole(cfg, with_dST):
    inp = synth.make_la_inputs(cfg)
    gen = torch.Generator().manual_seed(11)
    d_o = torch.randn((cfg.B, cfg.T, cfg.H, cfg.dv), generator=gen).to(torch.bfloat16)
    dST = torch.randn((cfg.B, cfg.H, cfg.dv, cfg.dk), generator=gen) if with_dST else None
    got = run_gdr_bwd(cfg, inp, d_o, dST)
    ref = LA.gated_delta_rule_backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]),
                                       f64(inp["beta"]), f64(inp["g"]), f64(d_o),
                                       dS_T=f64(dST), S0=f64(inp["S0"]))
    for name in ("dq", "dk", "dv", "dbeta", "dg", "dS0"):
        assert relerr(f64(got[name]), ref[name]) <= RTOL_G, name


@pytest.mark.parametrize("cfg", [BWD_CASES[0], BWD_CASES[3]], ids=["dk128_dv128", "dk64_dv64"])
def test_gdr_backward_with_forward_w(cfg):
    """The backward reading the forward's W_chunks (formed by the tensor-core scan) matches the
    oracle and the backward that forms W itself."""
    inp = synth.make_la_inputs(cfg)
    gen = torch.Generator().manual_seed(5)
    d_o = torch.randn((cfg.B, cfg.T, cfg.H, cfg.dv), generator=gen).to(torch.bfloat16)
    got = run_gdr_bwd(cfg, inp, d_o, None, keep_w=True)
    own = run_gdr_bwd(cfg, inp, d_o, None)
    ref = LA.gated_delta_rule_backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]),
                                       f64(inp["beta"]), f64(inp["g"]), f64(d_o),
                                       S0=f64(inp["S0"]))
    for name in ("dq", "dk", "dv", "dbeta", "dg", "dS0"):
        assert relerr(f64(got[name]), ref[name]) <= RTOL_G, name
        assert relerr(f64(got[name]), f64(own[name])) <= 1e-3, name


def test_gdr_backward_is_deterministic():
    cfg = BWD_CASES[0]
    inp = synth.make_la_inputs(cfg)
    d_o = torch.randn((cfg.B, cfg.T, cfg.H, cfg.dv)).to(torch.bfloat16)
    a = run_gdr_bwd(cfg, inp, d_o, None)
    b = run_gdr_bwd(cfg, inp, d_o, None)
    for name in a:
        assert torch.equal(a[name], b[name]), name
