"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random tensors; it holds none of the layer's arithmetic, so both
the CUDA path and the fp64 oracle can consume what it produces.  All draws use torch's
seeded generators (CPU: Mersenne-Twister based; CUDA: Philox), seed 0 by default.
Values that the workload stores in bf16 are rounded to bf16 (round-to-nearest-even) once,
here, so both sides see identical bits.

Workloads (sizes from the pages' model: 896 routed experts, 16 active per token):

  c1  T=256,   d=512,  E=64,  k=4,  F=256                      capacity factor inf
  c2  T=4096,  d=2048, E=896, k=16, F=512                      capacity factor inf
  c3  T=16384, d=4096, E=896, k=16, F=1024, Zipf router bias,  capacity factor 5/4
  c4  14-expert shard (896 / EP 64), 65536 pre-permuted rows, d=7168, F=2048,
      LoRA r=16, alpha=32 on gate/up/down
  c5  T=8192,  d=4096, E=896, k=16, F=1024, LoRA r=32, alpha=64, upstream dy,
      capacity factor inf

Distributions: x ~ N(0,1) bf16, router W_r ~ N(0, 0.02) fp32, expert weights
~ N(0, 0.02) bf16, LoRA A ~ N(0, 0.02) and B ~ N(0, 0.01) bf16, dy ~ N(0, 1) bf16.
Weight layouts: W_g, W_u [E, F, d]; W_d [E, d, F]; A_g, A_u [E, r, d]; B_g, B_u [E, F, r];
A_d [E, r, F]; B_d [E, d, r] (all row-major, "out x in" like a linear layer).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    E: int
    k: int
    F: int
    r: int = 0
    alpha: float = 0.0
    cap_num: int = 0
    cap_den: int = 0          # 0 -> infinite capacity factor
    zipf_bias: bool = False   # router bias b_e = 1.5 ln(Zipf(1.1) weight of rank e+1)
    prepermuted: bool = False  # rows given already grouped by expert (local shard)
    backward: bool = False
    remap_rounds: int = 0      # overflowing slots remapped to later preferences (rounds)
    chunks: int = 1            # token chunks pipelined (dispatch of chunk i+1 during chunk i)

    @property
    def lora_scale(self) -> float:
        return self.alpha / self.r if self.r else 0.0

    @property
    def slots(self) -> int:
        return self.T * self.k


CONFIGS = {
    "c1": MoEConfig("c1", T=256, d=512, E=64, k=4, F=256),
    "c2": MoEConfig("c2", T=4096, d=2048, E=896, k=16, F=512),
    "c3": MoEConfig("c3", T=16384, d=4096, E=896, k=16, F=1024, cap_num=5, cap_den=4,
                    zipf_bias=True),
    # c3 with one remap round: slots beyond capacity move to the token's next preferences
    "c3_remap": MoEConfig("c3_remap", T=16384, d=4096, E=896, k=16, F=1024, cap_num=5,
                          cap_den=4, zipf_bias=True, remap_rounds=1),
    # c3 in 4 token chunks, each chunk's dispatch overlapping the previous chunk's experts
    "c3_chunked": MoEConfig("c3_chunked", T=16384, d=4096, E=896, k=16, F=1024, cap_num=5,
                            cap_den=4, zipf_bias=True, chunks=4),
    "c4": MoEConfig("c4", T=65536, d=7168, E=14, k=1, F=2048, r=16, alpha=32.0,
                    prepermuted=True),
    "c5": MoEConfig("c5", T=8192, d=4096, E=896, k=16, F=1024, r=32, alpha=64.0,
                    backward=True),
    # small case of the c2 kernels for hardware-counter captures (0.8 GB of weights, about
    # 80 rows per expert like c2's 73): same shapes per expert, fewer experts and tokens
    "c2_small": MoEConfig("c2_small", T=640, d=2048, E=128, k=16, F=512),
    # small case of the c4 kernels (0.35 GB of expert weights, 4096 rows per expert like
    # c4's 4681): same shapes per expert, four experts
    "c4_small": MoEConfig("c4_small", T=16384, d=7168, E=4, k=1, F=2048, r=16, alpha=32.0,
                          prepermuted=True),
    # small case of the c5 kernels with c5's rows per expert (1024 x 16 / 112 = 146; 2.8 GB
    # of expert weights, larger than L2): hardware-counter captures of the c5 GEMMs, whose
    # DRAM traffic then scales to c5 by the number of experts (x 8)
    "c5_shard": MoEConfig("c5_shard", T=1024, d=4096, E=112, k=16, F=1024, r=32, alpha=64.0,
                          backward=True),
    # small case of the c5 kernels (3.2 GB of expert weights, about 256 rows per expert)
    "c5_small": MoEConfig("c5_small", T=2048, d=4096, E=128, k=16, F=1024, r=32, alpha=64.0,
                          backward=True),
}


def config(name: str, **overrides) -> MoEConfig:
    cfg = CONFIGS[name]
    return replace(cfg, **overrides) if overrides else cfg


def zipf_bias(E: int, s: float = 1.1, scale: float = 1.5) -> torch.Tensor:
    """b_e = scale * ln(w_{e+1}), w_q = q^-s / sum_{q'=1..E} q'^-s (expert 0 is hottest)."""
    Z = sum(q ** -s for q in range(1, E + 1))
    return torch.tensor([scale * math.log((q ** -s) / Z) for q in range(1, E + 1)],
                        dtype=torch.float32)


def _normal(gen, shape, std, device, dtype):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _per_expert(gen, E, shape, std, device):
    """Draw an [E, *shape] bf16 tensor one expert at a time (bounded fp32 temporaries)."""
    out = torch.empty((E,) + tuple(shape), device=device, dtype=torch.bfloat16)
    for e in range(E):
        out[e] = _normal(gen, shape, std, device, torch.bfloat16)
    return out


def balanced_offsets(rows: int, E: int) -> torch.Tensor:
    """Segment starts that spread ``rows`` over E experts as evenly as possible, the
    first ``rows % E`` experts taking one extra row (65536 over 14: 4682, 4682, 4681...)."""
    base, extra = divmod(rows, E)
    counts = [base + (1 if e < extra else 0) for e in range(E)]
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    return torch.tensor(offs, dtype=torch.int32)


def make_inputs(cfg: MoEConfig, device="cpu", seed: int = 0, weights: bool = True):
    """Every tensor of one workload, drawn in a fixed order from one seeded generator."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    out = {}
    if cfg.prepermuted:
        rows = cfg.T * cfg.k
        out["x_perm"] = _normal(gen, (rows, cfg.d), 1.0, dev, torch.bfloat16)
        out["offsets"] = balanced_offsets(rows, cfg.E).to(dev)
        out["row_slot"] = torch.arange(rows, dtype=torch.int32, device=dev)
        u = torch.rand((rows,), generator=gen, device=dev, dtype=torch.float32)
        out["gates"] = (1.0 - 0.95 * u)  # U(0.05, 1]
    else:
        out["x"] = _normal(gen, (cfg.T, cfg.d), 1.0, dev, torch.bfloat16)
        out["w_router"] = _normal(gen, (cfg.E, cfg.d), 0.02, dev, torch.float32)
        out["bias"] = zipf_bias(cfg.E).to(dev) if cfg.zipf_bias else None
    if weights:
        out["w_gate"] = _per_expert(gen, cfg.E, (cfg.F, cfg.d), 0.02, dev)
        out["w_up"] = _per_expert(gen, cfg.E, (cfg.F, cfg.d), 0.02, dev)
        out["w_down"] = _per_expert(gen, cfg.E, (cfg.d, cfg.F), 0.02, dev)
        if cfg.r:
            r = cfg.r
            out["lora"] = {
                "A_g": _per_expert(gen, cfg.E, (r, cfg.d), 0.02, dev),
                "B_g": _per_expert(gen, cfg.E, (cfg.F, r), 0.01, dev),
                "A_u": _per_expert(gen, cfg.E, (r, cfg.d), 0.02, dev),
                "B_u": _per_expert(gen, cfg.E, (cfg.F, r), 0.01, dev),
                "A_d": _per_expert(gen, cfg.E, (r, cfg.F), 0.02, dev),
                "B_d": _per_expert(gen, cfg.E, (cfg.d, r), 0.01, dev),
            }
    if cfg.backward:
        out["dy"] = _normal(gen, (cfg.T, cfg.d), 1.0, dev, torch.bfloat16)
    return out


# ----------------------------------------------------------------------------- linear attention

@dataclass(frozen=True)
class LAConfig:
    """Gated delta-rule linear attention: B sequences of T tokens, H heads, key width dk,
    value width dv."""
    name: str
    B: int
    T: int
    H: int
    dk: int = 128
    dv: int = 128
    with_state: bool = False   # start from a random state S0 instead of zero


LA_CONFIGS = {
    # one long sequence (the pages fine-tune with micro-batch 1 and long context), 16 heads
    "la": LAConfig("la", B=1, T=32768, H=16),
    "la_small": LAConfig("la_small", B=2, T=1000, H=4, with_state=True),
    # the same 16 heads on a 4096-token sequence (a hardware-counter capture case)
    "la_mid": LAConfig("la_mid", B=1, T=4096, H=16),
}


def la_config(name: str, **overrides) -> LAConfig:
    cfg = LA_CONFIGS[name]
    return replace(cfg, **overrides) if overrides else cfg


def make_la_inputs(cfg: LAConfig, device="cpu", seed: int = 0):
    """q, k, v ~ N(0, 1) bf16; beta = sigmoid(N(0, 1)); decay alpha = sigmoid(a), a ~ N(4, 1)
    (close to 1, as forget gates are), g = log(alpha) = -softplus(-a); S0 ~ N(0, 0.1)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    sh = (cfg.B, cfg.T, cfg.H)
    out = {"q": _normal(gen, sh + (cfg.dk,), 1.0, dev, torch.bfloat16),
           "k": _normal(gen, sh + (cfg.dk,), 1.0, dev, torch.bfloat16),
           "v": _normal(gen, sh + (cfg.dv,), 1.0, dev, torch.bfloat16)}
    out["beta"] = torch.sigmoid(torch.randn(sh, generator=gen, device=dev))
    a = torch.randn(sh, generator=gen, device=dev) + 4.0
    out["g"] = -torch.nn.functional.softplus(-a)
    out["S0"] = (torch.randn((cfg.B, cfg.H, cfg.dv, cfg.dk), generator=gen, device=dev) * 0.1
                 if cfg.with_state else None)
    return out
