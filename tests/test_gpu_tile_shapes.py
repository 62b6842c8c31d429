"""GPU parity of the grouped expert GEMMs on every tile shape they choose, with group sizes
at the tile boundaries: experts of 0, 1, 127..129, 255..257 rows (two-tile groups: the gate/up
GEMM on CTA pairs, whose second CTA often holds no valid row, and the dx GEMM on 256-row
tiles) and of over 1024 rows (every expert GEMM, forward and backward, on CTA pairs).
Forward (h, y_perm, saved activations) and backward (dx_perm and the six LoRA gradients)
against the fp64 oracle, expert by expert, through the C ABI on pre-permuted rows."""

import numpy as np
import pytest
import torch

import oracle
from top_routing_grouped_gemm_gb300 import moe
from parity_util import RTOL_FP, f64, relerr

pytestmark = pytest.mark.gpu

GRADS = ("A_g", "B_g", "A_u", "B_u", "A_d", "B_d")


def _bf(g, *shape, std=1.0):
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).cuda()


@pytest.mark.parametrize("counts", [
    [128, 129, 256, 1, 255, 257, 0, 300, 127],   # 128 < mean <= 256
    [1024, 1025, 2048, 1, 3000, 0, 1400],         # mean > 1024
], ids=["two_tile_groups", "big_groups"])
def test_expert_gemms_at_tile_boundaries(counts):
    E, d, F, r, s = len(counts), 192, 320, 16, 2.0
    N = int(sum(counts))
    g = torch.Generator().manual_seed(N)
    p = moe.Problem(T=N, d=d, E=E, k=1, F=F, r=r, lora_scale=s)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32).cuda()
    x_perm = _bf(g, N, d)
    row_slot = torch.arange(N, dtype=torch.int32).cuda()
    gates = (torch.rand(N, generator=g) * 0.9 + 0.1).float().cuda()
    W = {"w_gate": _bf(g, E, F, d, std=0.02), "w_up": _bf(g, E, F, d, std=0.02),
         "w_down": _bf(g, E, d, F, std=0.02)}
    lora = {"A_g": _bf(g, E, r, d, std=0.02), "B_g": _bf(g, E, F, r, std=0.01),
            "A_u": _bf(g, E, r, d, std=0.02), "B_u": _bf(g, E, F, r, std=0.01),
            "A_d": _bf(g, E, r, F, std=0.02), "B_d": _bf(g, E, d, r, std=0.01)}
    h = torch.empty(N, F, dtype=torch.bfloat16, device="cuda")
    y_perm = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    saved = {"a_gate": torch.empty(N, F, dtype=torch.bfloat16, device="cuda"),
             "a_up": torch.empty(N, F, dtype=torch.bfloat16, device="cuda")}
    for nm in ("u_gate", "u_up", "u_down"):
        saved[nm] = torch.empty(N, r, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(moe.moe_expert_ffn_workspace_size(p, N), dtype=torch.uint8, device="cuda")
    moe.moe_expert_ffn(p, N, x_perm, offsets, row_slot, gates, W["w_gate"], W["w_up"],
                       W["w_down"], lora, h, y_perm, saved, ws, st)
    dz = _bf(g, N, d)
    dx_perm = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    grads = {"dA_g": torch.empty(E, r, d, device="cuda"), "dB_g": torch.empty(E, F, r, device="cuda"),
             "dA_u": torch.empty(E, r, d, device="cuda"), "dB_u": torch.empty(E, F, r, device="cuda"),
             "dA_d": torch.empty(E, r, F, device="cuda"), "dB_d": torch.empty(E, d, r, device="cuda")}
    wsb = torch.empty(moe.moe_expert_ffn_bwd_workspace_size(p, N), dtype=torch.uint8,
                      device="cuda")
    moe.moe_expert_ffn_bwd(p, N, x_perm, offsets, W["w_gate"], W["w_up"], W["w_down"], lora,
                           saved, h, dz, dx_perm, grads, wsb, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    offs = offsets.cpu().numpy()
    # LoRA gradients compared over all experts at once, as in the other backward tests: the
    # gradient of an expert with a single row is one outer product, and the bf16 rounding of
    # its inputs alone can move a near-cancelling entry of v by far more than 5e-3
    ref = {nm: np.zeros(tuple(grads["d" + nm].shape)) for nm in GRADS}
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        Le = {nm: f64(lora[nm][e]) for nm in GRADS}
        Wg, Wu, Wd = f64(W["w_gate"][e]), f64(W["w_up"][e]), f64(W["w_down"][e])
        if hi > lo:
            X = f64(x_perm[lo:hi])
            a_g, a_u, h_ref, o = oracle.expert_forward(X, Wg, Wu, Wd, Le, s)
            assert relerr(f64(h[lo:hi]), h_ref) <= RTOL_FP, ("h", e)
            assert relerr(f64(saved["a_gate"][lo:hi]), a_g) <= RTOL_FP, ("a_gate", e)
            assert relerr(f64(y_perm[lo:hi]), f64(gates[lo:hi])[:, None] * o) <= RTOL_FP, ("y", e)
            dX, ge = oracle.expert_backward(X, f64(dz[lo:hi]), Wg, Wu, Wd, Le, s)
            assert relerr(f64(dx_perm[lo:hi]), dX) <= RTOL_FP, ("dx", e)
            for nm in GRADS:
                ref[nm][e] = ge[nm]
                if hi - lo >= 64:
                    assert relerr(f64(grads["d" + nm][e]), ge[nm]) <= RTOL_FP, (nm, e)
        else:
            for nm in GRADS:
                assert float(grads["d" + nm][e].abs().max()) == 0.0, (nm, e)
    for nm in GRADS:
        assert relerr(f64(grads["d" + nm]), ref[nm]) <= RTOL_FP, nm
