"""The unpermute fused into the down GEMM's epilogue (moe_expert_ffn_combine): y must be
bit for bit the separate combine's, on whole problems with drops, all-dropped tokens, LoRA,
ragged widths, CTA-pair tiles, the fused permute, and c2 at full size."""

import pytest
import torch

from top_routing_grouped_gemm_gb300 import moe, synth
from parity_util import to_dev

pytestmark = pytest.mark.gpu


def _run(cfg, dev, fuse, gather):
    p = moe.problem_of(cfg)
    buf = moe.LayerBuffers(p, "cuda")
    moe.layer_forward(buf, dev["x"], dev["w_router"], dev.get("bias"), dev["w_gate"],
                      dev["w_up"], dev["w_down"], dev.get("lora"), gather=gather,
                      fuse_combine=fuse)
    torch.cuda.synchronize()
    assert int(buf.dev_status.item()) == 0
    return buf


def small(**kw):
    base = dict(name="fc", T=300, d=192, E=6, k=2, F=192)
    base.update(kw)
    return synth.MoEConfig(**base)


CASES = [
    synth.config("c1"),
    small(cap_num=1, cap_den=2, zipf_bias=True),
    small(T=777, d=320, E=9, k=3, F=448, r=24, alpha=48.0, cap_num=1, cap_den=1),
    small(T=50, d=64, E=16, k=4, F=64, cap_num=0, cap_den=1),      # every slot dropped
    small(T=200, d=128, E=1024, k=32, F=64),
    small(T=2600, d=192, E=4, k=2, F=192),                          # CTA-pair tiles
    small(T=400, d=192, E=4, k=2, F=192),                           # two-tile groups
]


@pytest.mark.parametrize("gather", [False, True], ids=["x_perm", "gathered"])
@pytest.mark.parametrize("cfg", CASES, ids=["c1", "capacity_bias", "ragged_lora", "all_dropped",
                                            "k32", "big_groups", "two_tile_groups"])
def test_fused_combine_bit_exact(cfg, gather):
    dev = to_dev(synth.make_inputs(cfg, "cpu"))
    a = _run(cfg, dev, False, gather)
    b = _run(cfg, dev, True, gather)
    n = int(a.n_kept_dropped[0].item())
    assert torch.equal(a.y_perm[:n], b.y_perm[:n])
    assert torch.equal(a.y, b.y)


def test_fused_combine_c2_full():
    cfg = synth.config("c2")
    inp = synth.make_inputs(cfg, "cuda")
    a = _run(cfg, inp, False, True)
    b = _run(cfg, inp, True, True)
    assert torch.equal(a.y, b.y)
    c = _run(cfg, inp, True, True)     # run to run: same bits
    assert torch.equal(b.y, c.y)
