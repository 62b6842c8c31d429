#!/usr/bin/env python
"""Throughput of the sparse-MoE layer (route -> dispatch -> grouped SwiGLU experts with LoRA
-> combine -> aux loss, and for training workloads the LoRA backward) on one GB300, through
the C ABI of libmoe.so.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5] [--impl ours|reference]

The headline workload is c5 (T=8192 tokens, d=4096, 896 experts, top-16, F=1024, LoRA r=32:
forward plus the whole LoRA backward), the configuration with the most work per step.  The
line also carries sub-records for c2 (full-fanout routing), c3 (skewed routing with capacity
drops) and c4 (LoRA forward on one 14-expert shard, the tensor-bound grouped GEMM), each
with its own roofline.  One step is one pass of the whole layer over one batch of the
workload's seeded synthetic tokens, every input already resident in HBM.  Rank 0 prints one
JSON line.

  value        tokens/s over all ranks (each rank runs its own batch: weak scaling, no
               collective on the data path), CUDA events around K steps replayed as one CUDA
               graph, max over ranks
  e2e          the same through the public API with host buffers: pinned inputs copied in
               and outputs copied out inside the timed region, every step
  roofline     the dominant kernel, timed live by CUDA events the library records around its
               launches, against MEASURED_PEAKS.json
  cpu_baseline the fp64 oracle on a bounded sample of the same batch, on every host core
               (one thread per token shard, one BLAS thread each), plus the same oracle on
               one core
  --impl reference  times the oracle alone (the slow reference program of this build) on
               the host cores, same workload, metric and unit
"""

from __future__ import annotations

import os

# The oracle runs numpy with one BLAS thread per worker thread (set before numpy loads).
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import argparse
import concurrent.futures as cf
import hashlib
import json
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s and grouped-GEMM TFLOP/s (% BF16 peak), 1×GB300"
KERNEL_SOURCES = ["gemm.cuh", "ptx.cuh", "gemm_fwd.cu", "gemm_bwd.cu", "moe_internal.h"]
DEFAULT_WORKLOAD = "c5"
# sub-records carried by the headline line
DEFAULT_SUBS = {"c5": ["c2", "c3", "c3_remap", "c3_chunked", "c4", "la"]}
# tokens per host thread of the oracle baseline (forward-only workloads run more tokens:
# their oracle step is cheaper)
CPU_TOKENS_PER_THREAD = {"train": 2, "fwd": 16, "prepermuted_rows": 64}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--sub-workloads", default="auto",
                    help="comma-separated workloads reported as sub-records of the line; "
                         "'auto': c2,c3,c3_remap,c4 under the c5 headline; 'none': no "
                         "sub-records")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="host threads of the oracle baseline and the reference arm (0: all "
                         "cores this process may run on)")
    ap.add_argument("--cpu-tokens-per-thread", type=int, default=0,
                    help="tokens (rows for c4) per host thread of the oracle baseline "
                         "(0: the workload's default)")
    ap.add_argument("--ref-tokens-per-step", type=int, default=0,
                    help="tokens per step of the --impl reference arm (0: one per thread)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--permute", default="auto", choices=["auto", "fused", "separate"],
                    help="fused: gather token rows inside the expert GEMM; separate: write "
                         "x_perm in dispatch; auto: the library binding's default")
    ap.add_argument("--combine", default="separate", choices=["separate", "fused"],
                    help="fused: the unpermute inside the down GEMM's epilogue (same bits)")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch every step from the host instead of replaying a CUDA graph")
    return ap.parse_args(argv)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained"), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


def _code_only(src: str) -> str:
    """C++ source without comments and whitespace, so that editing a comment does not
    invalidate a hardware-counter capture of unchanged code."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return re.sub(r"\s+", "", src)


def kernel_source_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        src = open(os.path.join(ROOT, "top_routing_grouped_gemm_gb300", "csrc", f)).read()
        h.update(_code_only(src).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the kernel
    sources as they are now (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if "=" in line and line.strip().startswith(("traffic_bytes_per_launch", "source_hash")):
            k, v = line.strip().split("=", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_hash") != kernel_source_hash():
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def host_threads():
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def host_mem_available():
    """Bytes of host memory available (MemAvailable), or a large number if unknown."""
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 1 << 50


# ------------------------------------------------------------------------ multi-rank

def max_over_ranks(v, world, device):
    """Largest per-rank value (the step time the whole job waits for)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_rank, ms_step):
    """Whole-job rate: every rank processes its own batch of units (weak scaling)."""
    return world * units_per_rank / (ms_step * 1e-3)


# ------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in self.samples if num(s[1])]
        mx = [num(s[2]) for s in self.samples if num(s[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in self.samples:
            for n, v in zip(names, s[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(self.samples)}


# ------------------------------------------------------------------------ oracle baseline
#
# The oracle is timed as it stands: its public moe_forward / moe_backward / expert_forward
# on shards of a token sample, one shard per host thread.  numpy releases the interpreter
# lock inside its array kernels (matrix products, dtype conversions, exp), so the shards
# run side by side; every thread uses one BLAS thread.

class HostExperts:
    """[E, rows, cols] weight table of which only the experts a sample touches are held on
    the host, as bf16 torch tensors; an access returns the expert as float32 numpy (exact for
    bf16 values), which the oracle converts to float64."""

    def __init__(self, E, rows, cols):
        self.shape = (E, rows, cols)
        self.store = {}

    def __getitem__(self, e):
        return self.store[int(e)].float().numpy()


def run_sharded(fn, shards, threads):
    """Run fn(shard) for every shard on `threads` host threads; wall seconds."""
    t0 = time.perf_counter()
    if threads == 1:
        for s in shards:
            fn(s)
    else:
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(fn, shards))
    return time.perf_counter() - t0


class OracleProblem:
    """Host copies of one workload's inputs (only the experts a token sample touches) and the
    oracle step on a shard of that sample: the whole forward (and the LoRA backward for
    training workloads) of those tokens, or, for a pre-permuted shard, the expert forward of
    those rows."""

    def __init__(self, cfg, x, w_router, bias, dy, tables, lora, rows=None):
        self.cfg = cfg
        self.x, self.w_router, self.bias, self.dy = x, w_router, bias, dy
        self.tables = tables
        self.lora = lora
        self.rows = rows   # pre-permuted: blocks (expert, first row, end row) of x

    def step(self, shard):
        import oracle
        cfg = self.cfg
        s = cfg.lora_scale
        if cfg.prepermuted:
            for e, lo, hi in shard:
                L = None if self.lora is None else {n: v[e] for n, v in self.lora.items()}
                oracle.expert_forward(self.x[lo:hi], self.tables[0][e], self.tables[1][e],
                                      self.tables[2][e], L, s)
            return
        xs = self.x[shard]
        fwd = oracle.moe_forward(xs, self.w_router, self.tables[0], self.tables[1],
                                 self.tables[2], cfg.k, cfg.cap_num, cfg.cap_den,
                                 bias=self.bias, lora=self.lora, s=s)
        if cfg.backward:
            oracle.moe_backward(fwd, xs, self.dy[shard], self.w_router, self.tables[0],
                                self.tables[1], self.tables[2], self.lora, s)


def _touched_experts(cfg, x64, wr64, bias64):
    import numpy as np
    import oracle
    idx = oracle.topk_select(oracle.router_logits(x64, wr64, bias64), cfg.k)
    return [int(e) for e in np.unique(idx)]


def _lora_host(cfg, get, experts):
    """float64 LoRA factors [E, ...] with the touched experts filled (others never read)."""
    import numpy as np
    if not cfg.r:
        return None
    shapes = {"A_g": (cfg.r, cfg.d), "B_g": (cfg.F, cfg.r), "A_u": (cfg.r, cfg.d),
              "B_u": (cfg.F, cfg.r), "A_d": (cfg.r, cfg.F), "B_d": (cfg.d, cfg.r)}
    out = {n: np.zeros((cfg.E,) + sh) for n, sh in shapes.items()}
    for e in experts:
        for n in shapes:
            out[n][e] = get(n, e)
    return out


def oracle_problem_from_device(inp, cfg, n_tokens):
    """The oracle's inputs for the first n_tokens tokens (rows, for c4) of the device batch:
    the same values the CUDA path consumes."""
    import numpy as np
    f64 = lambda t: t.detach().float().cpu().double().numpy()
    names = ("w_gate", "w_up", "w_down")
    shapes = ((cfg.E, cfg.F, cfg.d), (cfg.E, cfg.F, cfg.d), (cfg.E, cfg.d, cfg.F))
    tabs = [HostExperts(*sh) for sh in shapes]
    if cfg.prepermuted:
        # the first rows of every expert, copied compactly; blocks (expert, start, end) index
        # the compact copy
        offs = inp["offsets"].cpu().tolist()
        per = max(1, n_tokens // cfg.E)
        blocks, sel = [], []
        for e in range(cfg.E):
            lo = offs[e]
            hi = min(offs[e + 1], lo + per)
            if hi > lo:
                blocks.append((e, len(sel), len(sel) + hi - lo))
                sel.extend(range(lo, hi))
        x = f64(inp["x_perm"][sel])
        experts = sorted({e for e, _, _ in blocks})
        for e in experts:
            for tab, n in zip(tabs, names):
                tab.store[e] = inp[n][e].cpu()
        lora = _lora_host(cfg, lambda n, e: f64(inp["lora"][n][e]), experts)
        return OracleProblem(cfg, x, None, None, None, tabs, lora, blocks), len(sel)
    n = min(n_tokens, cfg.T)
    wr = f64(inp["w_router"])
    bias = None if inp.get("bias") is None else f64(inp["bias"])
    while True:
        x = f64(inp["x"][:n])
        experts = _touched_experts(cfg, x, wr, bias)
        # the touched experts' bf16 weights are held on the host: keep them well inside the
        # host memory (halve the sample until they fit)
        if n == 1 or len(experts) * 6 * cfg.d * cfg.F <= 0.3 * host_mem_available():
            break
        n //= 2
    for e in experts:
        for tab, nm in zip(tabs, names):
            tab.store[e] = inp[nm][e].cpu()
    lora = _lora_host(cfg, lambda nm, e: f64(inp["lora"][nm][e]), experts)
    dy = f64(inp["dy"][:n]) if cfg.backward else None
    return OracleProblem(cfg, x, wr, bias, dy, tabs, lora), n


def shards_of(prob, n_units, threads):
    """Split the sample into `threads` contiguous shards."""
    import numpy as np
    if prob.cfg.prepermuted:
        blocks = prob.rows
        return [blocks[i::threads] for i in range(threads) if blocks[i::threads]]
    parts = np.array_split(np.arange(n_units), threads)
    return [p for p in parts if len(p)]


def cpu_baseline(inp, cfg, args):
    """The oracle on every host core (the timed CPU baseline) and on one core."""
    threads = args.cpu_threads or host_threads()
    kind = "prepermuted_rows" if cfg.prepermuted else ("train" if cfg.backward else "fwd")
    per = args.cpu_tokens_per_thread or CPU_TOKENS_PER_THREAD[kind]
    prob, n = oracle_problem_from_device(inp, cfg, per * threads)
    shards = shards_of(prob, n, threads)
    unit = "token-slots/s" if cfg.prepermuted else "tokens/s"
    size = (lambda sh: sum(hi - lo for _, lo, hi in sh)) if cfg.prepermuted else len
    wall = run_sharded(prob.step, shards, len(shards))
    one = shards[0]
    wall1 = run_sharded(prob.step, [one], 1)
    what = ("expert forward (SwiGLU with LoRA) of the first rows of every expert"
            if cfg.prepermuted else
            "fp64 router over all experts, top-k, dispatch, the selected experts' SwiGLU"
            + (" with LoRA" if cfg.r else "") + ", combine, aux"
            + (" + the LoRA backward (dx, dA, dB)" if cfg.backward else ""))
    return {"value": n / wall, "unit": unit, "cores": len(shards), "kind": "oracle",
            "sample": f"first {n} {'rows' if cfg.prepermuted else 'tokens'} of the {cfg.name} "
                      f"batch in {len(shards)} shards, one host thread each (numpy, 1 BLAS "
                      f"thread per shard): {what}",
            "seconds": wall,
            "single_core": {"value": size(one) / wall1, "unit": unit, "cores": 1,
                            "seconds": wall1, "units": size(one)}}


def run_reference(args):
    """The oracle as the reference program: every step the same bounded sample of a
    workload-shaped batch (host-generated, seeded), on every host core."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import torch
    from top_routing_grouped_gemm_gb300 import synth
    cfg = synth.config(args.workload)
    threads = getattr(args, "cpu_threads", 0) or host_threads()
    torch.set_num_threads(threads)
    n = getattr(args, "ref_tokens_per_step", 0) or threads
    g = torch.Generator().manual_seed(0)
    bf = lambda t: t.to(torch.bfloat16)
    names = ("w_gate", "w_up", "w_down")
    shapes = ((cfg.F, cfg.d), (cfg.F, cfg.d), (cfg.d, cfg.F))
    tabs = [HostExperts(cfg.E, *sh) for sh in shapes]

    def expert_weights(e):
        ge = torch.Generator().manual_seed(1000 + int(e))
        for tab, sh in zip(tabs, shapes):
            tab.store[int(e)] = bf(torch.randn(sh, generator=ge) * 0.02)

    def lora_of(nm, e):
        ge = torch.Generator().manual_seed(5000 + 7 * int(e) + "A_g B_g A_u B_u A_d B_d".split().index(nm))
        sh = {"A_g": (cfg.r, cfg.d), "B_g": (cfg.F, cfg.r), "A_u": (cfg.r, cfg.d),
              "B_u": (cfg.F, cfg.r), "A_d": (cfg.r, cfg.F), "B_d": (cfg.d, cfg.r)}[nm]
        std = 0.02 if nm.startswith("A") else 0.01
        return bf(torch.randn(sh, generator=ge) * std).double().numpy()

    if cfg.prepermuted:
        per = max(1, n * CPU_TOKENS_PER_THREAD["prepermuted_rows"] // cfg.E)
        rows = [(e, e * per, (e + 1) * per) for e in range(cfg.E)]
        x = bf(torch.randn((cfg.E * per, cfg.d), generator=g)).double().numpy()
        experts = list(range(cfg.E))
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(expert_weights, experts))
        prob = OracleProblem(cfg, x, None, None, None, tabs, _lora_host(cfg, lora_of, experts),
                             rows)
        shards = [rows[i::threads] for i in range(threads) if rows[i::threads]]
        units = cfg.E * per
        unit = "token-slots/s"
    else:
        x = bf(torch.randn((n, cfg.d), generator=g)).double().numpy()
        wr = (torch.randn((cfg.E, cfg.d), generator=g) * 0.02).double().numpy()
        bias = synth.zipf_bias(cfg.E).double().numpy() if cfg.zipf_bias else None
        dy = bf(torch.randn((n, cfg.d), generator=g)).double().numpy() if cfg.backward else None
        experts = _touched_experts(cfg, x, wr, bias)
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(expert_weights, experts))
        prob = OracleProblem(cfg, x, wr, bias, dy, tabs, _lora_host(cfg, lora_of, experts))
        shards = shards_of(prob, n, threads)
        units = n
        unit = "tokens/s"
    times = []
    for s in range(args.steps + args.warmup):
        dt = run_sharded(prob.step, shards, len(shards))
        if s >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = units * len(times) / total
    sample = (f"{units} {'rows' if cfg.prepermuted else 'tokens'} per step of a "
              f"{cfg.name}-shaped batch (host-generated, seed 0; the same sample every step), "
              f"in {len(shards)} shards on {len(shards)} host threads: fp64 oracle "
              + ("expert forward" if cfg.prepermuted else "forward")
              + (" + LoRA backward" if cfg.backward else "") + ", numpy, 1 BLAS thread each")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * total / max(1, len(times)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg),
        "cpu_baseline": {"value": value, "unit": unit, "cores": len(shards), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(cfg):
    c = {"workload": f"{cfg.name}: "
                     + (f"{cfg.T * cfg.k} pre-permuted rows over {cfg.E} experts"
                        if cfg.prepermuted else f"T={cfg.T} top-{cfg.k}")
                     + f" d={cfg.d} E={cfg.E} F={cfg.F}"
                     + (f" LoRA r={cfg.r} alpha={cfg.alpha:g}" if cfg.r else "")
                     + (f" capacity {cfg.cap_num}/{cfg.cap_den}" if cfg.cap_den else " capacity inf")
                     + (" Zipf(1.1) router bias" if cfg.zipf_bias else "")
                     + (f" {cfg.remap_rounds} remap round(s)" if cfg.remap_rounds else "")
                     + (f" in {cfg.chunks} pipelined chunks" if cfg.chunks > 1 else "")
                     + (" forward + LoRA backward" if cfg.backward else " forward"),
         "tokens_per_gpu": cfg.T, "experts": cfg.E, "top_k": cfg.k, "d_model": cfg.d,
         "d_ffn": cfg.F, "lora_rank": cfg.r, "seed": 0,
         "l2": "inputs larger than L2: the expert weights streamed every step exceed 129 MB"}
    return c


# ------------------------------------------------------------------------ GPU arm

def kernel_model(cfg, kept, nonempty, train, gather, fused_combine=False):
    """Algorithmic bytes and flops of one launch of each timed kernel (units: non-empty
    experts, kept rows, tokens), and which roofline bounds it.  With the permute fused into
    the expert GEMM (gather), its A operand is the token matrix, read once (T rows), and
    dispatch writes only the index maps."""
    d, F, E, T, k, r = cfg.d, cfg.F, cfg.E, cfg.T, cfg.k, cfg.r
    m = {}
    a_rows = T if gather else kept
    gu_b = nonempty * 2 * F * d * 2 + a_rows * d * 2 + kept * F * 2
    gu_f = kept * 4.0 * d * F
    dn_b = nonempty * d * F * 2 + kept * F * 2 + kept * d * 2
    dn_f = kept * 2.0 * d * F
    if r:
        gu_b += kept * 2 * r * 2 + nonempty * 2 * F * r * 2
        gu_f += kept * 2.0 * 2 * F * r
        dn_b += kept * r * 2 + nonempty * d * r * 2
        dn_f += kept * 2.0 * d * r
    if train:
        gu_b += kept * 2 * F * 2
    if fused_combine:  # the down GEMM also reads the kept rows back and writes y
        dn_b += kept * d * 2 + T * d * 2 + T * k * 4
    m["gateup_gemm"] = (gu_b, gu_f)
    m["down_gemm"] = (dn_b, dn_f)
    if not cfg.prepermuted:
        m["router_gemm"] = (T * d * 2 + E * d * 4 + T * E * 4, 2.0 * 2 * T * d * E)
        m["topk"] = (T * E * 4 + T * k * 8, 0.0)
        m["dispatch"] = (T * k * 4 * 3 + (0 if gather else T * d * 2 + kept * d * 2), 0.0)
        m["combine"] = (kept * d * 2 + T * d * 2 + T * k * 4, 0.0)
    if train:
        m["bwd_dh_gemm"] = (nonempty * d * F * 2 + kept * d * 2 + kept * F * 2 * 4
                            + (kept * r * 2 + nonempty * r * F * 2 if r else 0),
                            kept * 2.0 * d * F + (kept * 2.0 * F * r if r else 0))
        m["bwd_dx_gemm"] = (nonempty * 2 * d * F * 2 + kept * F * 2 * 2 + kept * d * 2
                            + (kept * 2 * r * 2 + nonempty * 2 * r * d * 2 if r else 0),
                            kept * 4.0 * d * F + (kept * 4.0 * d * r if r else 0))
        if r:
            m["wgrad"] = (kept * (2 * d + 3 * F) * 2 + kept * 5 * r * 2
                          + E * r * (3 * d + 3 * F) * 4,
                          kept * 2.0 * r * (3 * d + 3 * F))
        # dz_perm = g dy (dy read, kept rows written; slot maps and gates read, dgate zeroed)
        m["combine_bwd"] = (T * d * 2 + kept * d * 2 + T * k * 12, 0.0)
        # dx = sum of the kept dx_perm rows + the router path (W_r read once, fp32 dx written)
        m["dispatch_route_bwd"] = (kept * d * 2 + T * k * 16 + E * d * 4 + T * d * 4, 0.0)
    return m


class Ctx:
    def __init__(self, args, rank, world, local, barrier):
        self.args, self.rank, self.world, self.local, self.barrier = (args, rank, world, local,
                                                                      barrier)


def fp32_alu_peak_tflops():
    """fp32 FMA rate of the SIMT pipes: 152 SMs x 128 lanes x 2 flop x 2.07 GHz (the
    maximum SM clock of these GPUs; the recipe's unit counts and clock)."""
    return 152 * 128 * 2 * 2.07e9 / 1e12


def la_flops_per_chunk(dk, dv, C=64):
    """Multiply-adds of one 64-token chunk of one head in the chunked algorithm, x 2:
    chunk factors (the K^K^T and Q^K^T triangles, the triangular inverse, Y and U) and the
    scan (W = U - Y S^T, O = gamma Q^ S^T + P W, the state update)."""
    tri = C * (C + 1) // 2
    chunk = 2 * tri * dk + C ** 3 // 6 + tri * dk + tri * dv
    scan = C * dv * dk + (C * dv * dk + tri * dv) + dv * dk * C
    return 2.0 * (chunk + scan)


def la_bwd_flops_per_chunk(dk, dv, C=64):
    """Multiply-adds of the backward of one 64-token chunk of one head, x 2: the chunk factors
    rebuilt (as in the forward), the state-gradient scan (dW = s P^T dO + E dS1^T, and
    dS0 = gamma_C dS1 + s dO^T diag(gamma) Q^ - dW^T Y), and the chunk-local backward
    (W = U - Y S0^T, dP = s dO W^T, dQ^ and dK^ from Gam . dP and from S0 / dS1, dBv = A^-T dW,
    dBk = -dBv S0, dM from dBv U^T + dBk Y^T, (Z + Z^T) K^)."""
    tri = C * (C + 1) // 2
    factors = 2 * tri * dk + C ** 3 // 6 + tri * dk + tri * dv
    scan = tri * dv + 3 * C * dk * dv
    local = 4 * C * dk * dv + 3 * tri * dv + 3 * tri * dk + C * C * dk
    return 2.0 * (factors + scan + local)


def run_linear_attention(name, ctx):
    """The chunked gated delta-rule linear attention on its workload: the forward, and the
    training step (the forward keeping every chunk-start state, then the backward); K steps
    of each replayed as one CUDA graph, per-kernel CUDA events from a host-launched pass."""
    import torch
    from top_routing_grouped_gemm_gb300 import moe, synth
    args = ctx.args
    cfg = synth.la_config(name)
    inp = synth.make_la_inputs(cfg, "cuda", seed=ctx.rank)
    B, T, H, dk, dv = cfg.B, cfg.T, cfg.H, cfg.dk, cfg.dv
    o = torch.empty((B, T, H, dv), dtype=torch.bfloat16, device="cuda")
    ST = torch.empty((B, H, dv, dk), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.moe_gdr_workspace_size(B, T, H, dk, dv), dtype=torch.uint8,
                     device="cuda")

    def step():
        moe.moe_gdr_forward(B, T, H, dk, dv, inp["q"], inp["k"], inp["v"], inp["beta"],
                            inp["g"], inp["S0"], dk ** -0.5, o, ST, None, ws)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    K = args.steps
    kernels = ["gdr_chunk", "gdr_scan"]
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)] for n in kernels}
    for n in kernels:
        for a, b in ev[n]:
            a.record()
            b.record()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(K):
            step()
    torch.cuda.synchronize()
    clocks = ClockSampler(ctx.local)
    ctx.barrier()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    graph.replay()
    s1.record()
    torch.cuda.synchronize()
    ctx.barrier()
    clocks.stop()
    for i in range(K):
        for n in kernels:
            moe.moe_set_kernel_events(n, ev[n][i][0], ev[n][i][1])
        step()
    for n in kernels:
        moe.moe_set_kernel_events(n, None, None)
    torch.cuda.synchronize()
    ms = max_over_ranks(s0.elapsed_time(s1) / K, ctx.world, "cuda")
    us = {n: 1000.0 * sum(a.elapsed_time(b) for a, b in ev[n]) / K for n in kernels}
    nch = (T + 63) // 64
    flops = la_flops_per_chunk(dk, dv) * nch * B * H
    peak = fp32_alu_peak_tflops()
    tot_us = sum(us.values())
    achieved = flops / (tot_us * 1e-6) / 1e12
    peak_src = "fp32 FMA pipes: 152 SMs x 128 lanes x 2 x 2.07 GHz"

    # training step: the forward keeping every chunk-start state, then the backward
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1000 + ctx.rank)
    d_o = torch.randn((B, T, H, dv), generator=gen, device="cuda").to(torch.bfloat16)
    Schk = torch.empty((B, H, nch, dv, dk), dtype=torch.float32, device="cuda")
    Wchk = torch.empty((B, H, nch, 64, dv), dtype=torch.float32, device="cuda")
    dq = torch.empty((B, T, H, dk), dtype=torch.float32, device="cuda")
    dkk = torch.empty_like(dq)
    dvv = torch.empty((B, T, H, dv), dtype=torch.float32, device="cuda")
    dbeta = torch.empty((B, T, H), dtype=torch.float32, device="cuda")
    dg = torch.empty_like(dbeta)
    dS0 = torch.empty((B, H, dv, dk), dtype=torch.float32, device="cuda")
    ws_b = torch.empty(moe.moe_gdr_backward_workspace_size(B, T, H, dk, dv), dtype=torch.uint8,
                       device="cuda")

    def train_step():
        moe.moe_gdr_forward(B, T, H, dk, dv, inp["q"], inp["k"], inp["v"], inp["beta"],
                            inp["g"], inp["S0"], dk ** -0.5, o, ST, Schk, ws, W_chunks=Wchk)
        moe.moe_gdr_backward(B, T, H, dk, dv, inp["q"], inp["k"], inp["v"], inp["beta"],
                             inp["g"], dk ** -0.5, d_o, None, Schk, dq, dkk, dvv, dbeta, dg, dS0,
                             ws_b, W_chunks=Wchk)
    for _ in range(max(args.warmup, 3)):
        train_step()
    torch.cuda.synchronize()
    tk = kernels + ["gdr_bwd_factors", "gdr_bwd_scan", "gdr_bwd"]
    tev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)] for n in tk}
    for n in tk:
        for a, b in tev[n]:
            a.record()
            b.record()
    tgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tgraph):
        for _ in range(K):
            train_step()
    torch.cuda.synchronize()
    tclocks = ClockSampler(ctx.local)
    ctx.barrier()
    s0.record()
    tgraph.replay()
    s1.record()
    torch.cuda.synchronize()
    ctx.barrier()
    tclocks.stop()
    for i in range(K):
        for n in tk:
            moe.moe_set_kernel_events(n, tev[n][i][0], tev[n][i][1])
        train_step()
    for n in tk:
        moe.moe_set_kernel_events(n, None, None)
    torch.cuda.synchronize()
    t_ms = max_over_ranks(s0.elapsed_time(s1) / K, ctx.world, "cuda")
    t_us = {n: 1000.0 * sum(a.elapsed_time(b) for a, b in tev[n]) / K for n in tk}
    t_flops = flops + la_bwd_flops_per_chunk(dk, dv) * nch * B * H
    t_ach = t_flops / (sum(t_us.values()) * 1e-6) / 1e12
    train = {"value": job_throughput(ctx.world, B * T, t_ms), "unit": "tokens/s",
             "ms_per_step": t_ms, "cuda_graph": True, "gpu_launches": 5 * K,
             "what": "forward (chunk-start states and W kept) + backward to q, k, v, beta, g, S0",
             "kernels": {n: {"us": t_us[n]} for n in tk},
             "roofline": {"kernel": "all five", "bound": "alu", "achieved": t_ach,
                          "peak": peak, "unit": "TFLOP/s", "frac": t_ach / peak,
                          "traffic": None, "algorithmic_flops": t_flops,
                          "peak_source": peak_src},
             "clocks": tclocks.summary()}
    return {"value": job_throughput(ctx.world, B * T, ms), "unit": "tokens/s",
            "ms_per_step": ms, "cuda_graph": True, "gpu_launches": 2 * K,
            "config": {"workload": f"{cfg.name}: gated delta-rule linear attention, B={B} "
                                   f"T={T} H={H} dk={dk} dv={dv}, 64-token chunks, forward",
                       "seed": 0},
            "kernels": {n: {"us": us[n]} for n in kernels},
            "roofline": {"kernel": "gdr_chunk + gdr_scan", "bound": "alu",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None,
                         "algorithmic_flops": flops, "peak_source": peak_src},
            "train": train,
            "clocks": clocks.summary()}


def run_chunked(cfg, ctx):
    """The layer with its tokens in cfg.chunks chunks, each chunk's dispatch running on a
    second stream during the previous chunk's expert GEMMs (the expert-parallel driver with
    one rank).  Host-launched (its exchange plan reads the per-chunk counts on the host), so
    no CUDA graph; K steps between CUDA events."""
    import torch
    from top_routing_grouped_gemm_gb300 import ep, moe, synth
    args = ctx.args
    inp = synth.make_inputs(cfg, "cuda", seed=ctx.rank)
    p = moe.problem_of(cfg)
    r = ep.EPRank(rank=0, x=inp["x"], w_gate=inp["w_gate"], w_up=inp["w_up"],
                  w_down=inp["w_down"], lora=inp.get("lora"))
    be = ep.CudaBackend()

    def step():
        return ep.ep_forward(p, [r], inp["w_router"], inp.get("bias"), ep.LocalExchange(1), be,
                             n_chunks=cfg.chunks)[0]
    for _ in range(max(args.warmup, 3)):
        out = step()
    torch.cuda.synchronize()
    if int(out["state"].dev_status.item()) != 0:
        raise RuntimeError(f"{cfg.name}: device status after warm-up")
    clocks = ClockSampler(ctx.local)
    ctx.barrier()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = moe.moe_launch_count()
    s0.record()
    for _ in range(args.steps):
        out = step()
    s1.record()
    torch.cuda.synchronize()
    ctx.barrier()
    clocks.stop()
    ms = max_over_ranks(s0.elapsed_time(s1) / args.steps, ctx.world, "cuda")
    kept = sum(int(pl.kept.sum()) for pl in out["plans"])
    return {"value": job_throughput(ctx.world, cfg.T, ms), "unit": "tokens/s",
            "ms_per_step": ms, "config": workload_config(cfg), "chunks": cfg.chunks,
            "kept_rows": kept, "cuda_graph": False,
            "gpu_launches": moe.moe_launch_count() - launches0, "clocks": clocks.summary(),
            "note": "host-launched steps (the per-chunk plan reads counts on the host); "
                    "bit-exact with the unchunked layer (tests/test_gpu_ep.py)"}


def run_workload(name, ctx, with_cpu):
    """Time one workload on this rank's GPU; returns the fields of its JSON record."""
    import torch
    from top_routing_grouped_gemm_gb300 import moe, synth

    args, world, rank = ctx.args, ctx.world, ctx.rank
    if name in synth.LA_CONFIGS:
        return run_linear_attention(name, ctx)
    cfg = synth.config(name)
    if cfg.chunks > 1:
        return run_chunked(cfg, ctx)
    train = cfg.backward
    fused = {"fused": True, "separate": False}.get(
        args.permute, moe.fused_permute_default(moe.problem_of(cfg), train))
    fused = fused and not train and not cfg.prepermuted
    inp = synth.make_inputs(cfg, "cuda", seed=rank)
    p = moe.problem_of(cfg)
    stream = torch.cuda.current_stream()
    lora = inp.get("lora")

    if cfg.prepermuted:
        # one EP shard's experts on pre-permuted rows: the expert GEMMs alone
        rows = cfg.T * cfg.k
        h = torch.empty((rows, cfg.F), dtype=torch.bfloat16, device="cuda")
        y_perm = torch.empty((rows, cfg.d), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(moe.moe_expert_ffn_workspace_size(p, rows), dtype=torch.uint8,
                         device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")

        def step():
            moe.moe_expert_ffn(p, rows, inp["x_perm"], inp["offsets"], inp["row_slot"],
                               inp["gates"], inp["w_gate"], inp["w_up"], inp["w_down"], lora, h,
                               y_perm, None, ws, status)
        kernels = ["gateup_gemm", "down_gemm"]
        offs = inp["offsets"].cpu()
        kept = int(offs[-1])
        nonempty = int((offs[1:] - offs[:-1] > 0).sum())
        out_bytes = (rows * cfg.d * 2, rows * cfg.d * 2)
    else:
        buf = moe.LayerBuffers(p, "cuda", train=train, keep_logits=train,
                               remap_rounds=cfg.remap_rounds)
        status = buf.dev_status

        fuse_combine = args.combine == "fused"

        def step():
            moe.layer_forward(buf, inp["x"], inp["w_router"], inp["bias"], inp["w_gate"],
                              inp["w_up"], inp["w_down"], lora,
                              gather=fused, fuse_combine=fuse_combine)
            if train:
                moe.layer_backward(buf, inp["dy"], inp["x"], inp["w_router"], inp["w_gate"],
                                   inp["w_up"], inp["w_down"], lora)
        kernels = ["router_gemm", "topk", "dispatch", "gateup_gemm", "down_gemm"] + \
            ([] if fuse_combine else ["combine"])
        if train:
            kernels += ["combine_bwd", "bwd_dh_gemm", "bwd_dx_gemm"] + \
                (["wgrad"] if cfg.r else []) + ["dispatch_route_bwd"]

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"{name}: device status {moe.STATUS_NAMES.get(st, st)} after warm-up")
    if not cfg.prepermuted:
        kept = int(buf.n_kept_dropped[0].item())
        nonempty = int((buf.offsets[1:] - buf.offsets[:-1] > 0).sum().item())

    K = args.steps
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)] for n in kernels}
    # torch creates the CUDA event behind an Event on its first record: record each once so
    # that the raw handles handed to the library are live
    for n in kernels:
        for a, b2 in ev[n]:
            a.record(stream)
            b2.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def kernel_timed_steps():
        for i in range(K):
            for n in kernels:
                moe.moe_set_kernel_events(n, ev[n][i][0], ev[n][i][1])
            step()
        for n in kernels:
            moe.moe_set_kernel_events(n, None, None)

    # Headline: the K steps captured once into a CUDA graph and replayed as one unit (no host
    # launch overhead in the timed region).  Per-kernel durations: the same K steps launched
    # from the host with the library recording CUDA events around each kernel (event timing
    # is not available for events recorded inside a graph).
    graph = None
    launches0 = moe.moe_launch_count()
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="relaxed"):
            for _ in range(K):
                step()
        torch.cuda.synchronize()
        launches = moe.moe_launch_count() - launches0
    clocks = ClockSampler(ctx.local)
    time.sleep(0.3)
    ctx.barrier()
    torch.cuda.synchronize()
    launches0 = moe.moe_launch_count()
    start.record(stream)
    if graph is not None:
        graph.replay()
    else:
        kernel_timed_steps()
    end.record(stream)
    torch.cuda.synchronize()
    ctx.barrier()
    if graph is None:
        launches = moe.moe_launch_count() - launches0
    else:
        kernel_timed_steps()
        torch.cuda.synchronize()
    clocks.stop()
    ms_step = max_over_ranks(start.elapsed_time(end) / K, world, "cuda")
    kern_us = {n: 1000.0 * sum(a.elapsed_time(b2) for a, b2 in ev[n]) / K for n in kernels}
    del graph

    pk = peaks()
    hbm = pk["hbm_gbs"]
    tpeak = pk["bf16_tflops"]
    tpeak_sus = pk["bf16_tflops_sustained"] or tpeak
    model = kernel_model(cfg, kept, nonempty, train, gather=fused,
                         fused_combine=(not cfg.prepermuted) and args.combine == "fused")
    kstats = {}
    for n in kernels:
        by, fl = model[n]
        us = kern_us[n]
        t_hbm = by / (hbm * 1e9)
        t_tc = fl / (tpeak * 1e12)
        bound = "tensor" if t_tc > t_hbm else "hbm"
        ent = {"us": us, "GB/s": by / (us * 1e-6) / 1e9, "bound": bound,
               "algorithmic_bytes": by}
        if fl:
            ent["TFLOP/s"] = fl / (us * 1e-6) / 1e12
            ent["flops"] = fl
        ent["frac"] = (ent["TFLOP/s"] / tpeak) if bound == "tensor" else (ent["GB/s"] / hbm)
        kstats[n] = ent
    dominant = max(kernels, key=lambda n: kern_us[n])
    dm = kstats[dominant]
    if dm["bound"] == "tensor":
        roof = {"kernel": dominant, "bound": "tensor", "achieved": dm["TFLOP/s"], "peak": tpeak,
                "unit": "TFLOP/s", "frac": dm["TFLOP/s"] / tpeak,
                "frac_of_sustained": dm["TFLOP/s"] / tpeak_sus,
                "traffic": profiled_traffic(dominant, name),
                "algorithmic_flops": dm["flops"], "launch_us": dm["us"],
                "peak_source": pk["source"] + " bf16 burst"}
    else:
        roof = {"kernel": dominant, "bound": "hbm", "achieved": dm["GB/s"], "peak": hbm,
                "unit": "GB/s", "frac": dm["GB/s"] / hbm,
                "traffic": profiled_traffic(dominant, name),
                "algorithmic_bytes": dm["algorithmic_bytes"], "launch_us": dm["us"],
                "peak_source": pk["source"]}
    gemms = [n for n in kernels if n.endswith("gemm") and n != "router_gemm"] + \
        (["wgrad"] if "wgrad" in kernels else [])
    g_us = sum(kern_us[n] for n in gemms)
    g_fl = sum(model[n][1] for n in gemms)
    g_by = sum(model[n][0] for n in gemms)
    g_roof_us = max(g_by / (hbm * 1e9), g_fl / (tpeak * 1e12)) * 1e6

    # ---------------------------------------------------------------- end to end (host buffers)
    # Serving loop: each step copies its inputs in from pinned host memory and its outputs
    # back out.  Two buffer sets alternate; inputs and outputs move on two copy streams (one
    # per direction), so step i's copies overlap the neighbours' compute and each other.
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    main_stream = torch.cuda.current_stream()
    if cfg.prepermuted:
        # the expert FFN alone: permuted rows in, gated expert outputs out
        in_src = [inp["x_perm"]]
        y_dev = [y_perm, torch.empty_like(y_perm)]

        def outputs(cur):
            return [y_dev[cur]]

        def compute(cur, dev_in):
            moe.moe_expert_ffn(p, rows, dev_in[0], inp["offsets"], inp["row_slot"], inp["gates"],
                               inp["w_gate"], inp["w_up"], inp["w_down"], lora, h, y_dev[cur],
                               None, ws, status)
    else:
        # the whole layer: tokens (and dy for training) in; y, aux (and dx) out
        bufs = [buf, moe.LayerBuffers(p, "cuda", train=train, keep_logits=train,
                                      remap_rounds=cfg.remap_rounds)]
        in_src = [inp["x"]] + ([inp["dy"]] if train else [])

        def outputs(cur):
            b = bufs[cur]
            return [b.y, b.aux] + ([b.dx] if train else [])

        def compute(cur, dev_in):
            b = bufs[cur]
            moe.layer_forward(b, dev_in[0], inp["w_router"], inp["bias"], inp["w_gate"],
                              inp["w_up"], inp["w_down"], lora, gather=fused,
                              fuse_combine=fuse_combine)
            if train:
                moe.layer_backward(b, dev_in[1], dev_in[0], inp["w_router"], inp["w_gate"],
                                   inp["w_up"], inp["w_down"], lora)
    in_host = [t.cpu().pin_memory() for t in in_src]
    in_dev = [[torch.empty_like(t) for t in in_src] for _ in range(2)]
    out_host = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outputs(c)]
                for c in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    ev_back = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        h2d_stream.wait_stream(main_stream)
        d2h_stream.wait_stream(main_stream)
        with torch.cuda.stream(h2d_stream):
            for d, hst in zip(in_dev[0], in_host):
                d.copy_(hst, non_blocking=True)
            ev_in[0].record(h2d_stream)
        for i in range(n):
            cur, nxt = i % 2, 1 - i % 2
            main_stream.wait_event(ev_in[cur])
            if i >= 2:
                main_stream.wait_event(ev_back[cur])  # step i-2's outputs copied out
            compute(cur, in_dev[cur])
            ev_out[cur].record(main_stream)
            if i + 1 < n:
                with torch.cuda.stream(h2d_stream):
                    if i >= 1:
                        h2d_stream.wait_event(ev_out[nxt])  # step i-1 done with in_dev[nxt]
                    for d, hst in zip(in_dev[nxt], in_host):
                        d.copy_(hst, non_blocking=True)
                    ev_in[nxt].record(h2d_stream)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(ev_out[cur])
                for hst, o in zip(out_host[cur], outputs(cur)):
                    hst.copy_(o, non_blocking=True)
                ev_back[cur].record(d2h_stream)
        main_stream.wait_stream(h2d_stream)
        main_stream.wait_stream(d2h_stream)

    if cfg.prepermuted:
        h2d, d2h = out_bytes
    else:
        h2d = cfg.T * cfg.d * 2 * (2 if train else 1)
        d2h = cfg.T * cfg.d * 2 + 4 + (cfg.T * cfg.d * 4 if train else 0)

    for _ in range(3):
        e2e_run(1)
    torch.cuda.synchronize()

    g2 = None
    if args.graph:
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, capture_error_mode="relaxed"):
            e2e_run(K)
        torch.cuda.synchronize()
    ctx.barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    if g2 is not None:
        g2.replay()
    else:
        e2e_run(K)
    e2.record(stream)
    torch.cuda.synchronize()
    ctx.barrier()
    ms_e2e = max_over_ranks(s2.elapsed_time(e2) / K, world, "cuda")
    del g2

    units = cfg.T * cfg.k if cfg.prepermuted else cfg.T
    unit = "token-slots/s" if cfg.prepermuted else "tokens/s"
    rec = {
        "value": job_throughput(world, units, ms_step),
        "unit": unit,
        "ms_per_step": ms_step,
        "config": workload_config(cfg),
        "grouped_gemm": {"TFLOP/s": g_fl / (g_us * 1e-6) / 1e12,
                         "pct_bf16_peak": 100.0 * g_fl / (g_us * 1e-6) / 1e12 / tpeak,
                         "pct_bf16_sustained": 100.0 * g_fl / (g_us * 1e-6) / 1e12 / tpeak_sus,
                         "us": g_us, "roofline_us": g_roof_us,
                         "frac_of_roofline": g_roof_us / g_us, "flops": g_fl,
                         "kernels": gemms, "kept_rows": kept, "nonempty_experts": nonempty},
        "roofline": roof,
        "kernels": kstats,
        "e2e": {"value": job_throughput(world, units, ms_e2e), "unit": unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "cuda_graph": bool(args.graph),
        "fused_permute": bool(fused),
        "fused_combine": (not cfg.prepermuted) and args.combine == "fused",
        "clocks": clocks.summary(),
    }
    if not cfg.prepermuted:
        rec["dropped_slots"] = int(buf.n_kept_dropped[1].item())
    if with_cpu:
        rec["cpu_baseline"] = cpu_baseline(inp, cfg, args)
    return rec


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import torch.distributed as dist

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")

    def barrier():
        if world > 1:
            dist.barrier()

    ctx = Ctx(args, rank, world, local, barrier)
    if args.sub_workloads == "auto":
        subs = DEFAULT_SUBS.get(args.workload, [])
    elif args.sub_workloads in ("", "none"):
        subs = []
    else:
        subs = [w for w in args.sub_workloads.split(",") if w and w != args.workload]

    with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    head = run_workload(args.workload, ctx, with_cpu=False)
    torch.cuda.empty_cache()
    sub_recs = {}
    for w in subs:
        sub_recs[w] = run_workload(w, ctx, with_cpu=False)
        torch.cuda.empty_cache()
    if with_cpu:
        # the oracle baseline runs after every GPU timing, so it never overlaps one
        from top_routing_grouped_gemm_gb300 import synth
        cfg = synth.config(args.workload)
        inp = synth.make_inputs(cfg, "cuda", seed=rank)
        head["cpu_baseline"] = cpu_baseline(inp, cfg, args)
        del inp
        torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": head["value"],
            "unit": head["unit"],
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": head["ms_per_step"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
        }
        line.update({k: v for k, v in head.items() if k not in line})
        line.setdefault("cpu_baseline", None)
        if sub_recs:
            line["workloads"] = sub_recs
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
