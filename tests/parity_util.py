"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI and compute
the fp64 oracle on the same seeded inputs (whole problem, or sampled tokens/rows)."""

import numpy as np
import torch

import oracle
from top_routing_grouped_gemm_gb300 import moe

RTOL_FP = 5e-3       # relative Frobenius error bound on floating-point outputs
RTOL_LOGITS = 1e-5   # fp32-accurate router logits (split bf16 product, fp32 accumulate)


def f64(t):
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()


def relerr(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def to_dev(inp, device="cuda"):
    out = {}
    for k, v in inp.items():
        if isinstance(v, dict):
            out[k] = {kk: vv.to(device) for kk, vv in v.items()}
        elif v is None:
            out[k] = None
        else:
            out[k] = v.to(device)
    return out


def run_forward(p, inp, train=False, gather=False):
    buf = moe.LayerBuffers(p, "cuda", train=train)
    moe.layer_forward(buf, inp["x"], inp["w_router"], inp.get("bias"), inp["w_gate"],
                      inp["w_up"], inp["w_down"], inp.get("lora"), gather=gather)
    torch.cuda.synchronize()
    assert int(buf.dev_status.item()) == 0
    return buf


def lora64(lora, e=None):
    if lora is None:
        return None
    if e is None:
        return {n: f64(v) for n, v in lora.items()}
    return {n: f64(v[e]) for n, v in lora.items()}


class ExpertCache:
    """fp64 host copies of the weights of single experts, fetched on demand."""

    def __init__(self, inp):
        self.inp = inp
        self.cache = {}

    def __call__(self, e):
        if e not in self.cache:
            self.cache[e] = (f64(self.inp["w_gate"][e]), f64(self.inp["w_up"][e]),
                             f64(self.inp["w_down"][e]), lora64(self.inp.get("lora"), e))
        return self.cache[e]


def oracle_tokens(inp, p, tokens, idx, gates64, slot_row):
    """y for selected tokens by the oracle's expert network, with the given routing (the
    routing is checked separately and bit-exactly), in fp64.  Weights are fetched one
    expert at a time and dropped after use, so host memory stays small at full sizes."""
    x = f64(inp["x"][tokens])
    ys = np.zeros((len(tokens), p.d))
    users = {}
    for n, t in enumerate(tokens):
        for j in range(p.k):
            if slot_row[t * p.k + j] >= 0:
                users.setdefault(int(idx[t, j]), []).append((n, t, j))
    for e in sorted(users):
        Wg, Wu, Wd = f64(inp["w_gate"][e]), f64(inp["w_up"][e]), f64(inp["w_down"][e])
        L = lora64(inp.get("lora"), e)
        for n, t, j in users[e]:
            o = oracle.expert_forward(x[n:n + 1], Wg, Wu, Wd, L, p.lora_scale)[3]
            ys[n] += gates64[t, j] * o[0]
    return ys


class DeviceExperts:
    """[E, rows, cols] weight table read from a device tensor one expert at a time (as
    float32, exact for bf16 values), so the oracle's per-expert loops can run at full size
    without a host copy of every expert."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        return self.t[int(e)].float().cpu().numpy()


def oracle_experts_backward(inp, p, slots_by_expert, gates64, x64, dy64):
    """For the slots (t, j) of each expert, the oracle's expert forward and backward:
    o[(t, j)] (ungated expert output) and dX[(t, j)] (input gradient with dO = g dy).
    Weights are fetched one expert at a time."""
    o, dX = {}, {}
    for e in sorted(slots_by_expert):
        sl = slots_by_expert[e]
        ts = [t for t, _ in sl]
        Wg, Wu, Wd = f64(inp["w_gate"][e]), f64(inp["w_up"][e]), f64(inp["w_down"][e])
        L = lora64(inp.get("lora"), e)
        X = x64[ts]
        oe = oracle.expert_forward(X, Wg, Wu, Wd, L, p.lora_scale)[3]
        dO = np.array([gates64[t, j] for t, j in sl])[:, None] * dy64[ts]
        dXe, _ = oracle.expert_backward(X, dO, Wg, Wu, Wd, L, p.lora_scale)
        for n, (t, j) in enumerate(sl):
            o[(t, j)] = oe[n]
            dX[(t, j)] = dXe[n]
    return o, dX
