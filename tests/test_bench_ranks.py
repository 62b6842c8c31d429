"""bench.py's multi-rank logic on CPU: two gloo ranks agree on the slowest rank's step time,
and the job rate counts every rank's own batch (no collective touches the data path)."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 1.0 + rank * 0.5  # rank 1 is slower
    ms = bench.max_over_ranks(local_ms, world, "cpu")
    out[rank] = (ms, bench.job_throughput(world, 4096, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == pytest.approx(1.5)
    assert value == pytest.approx(2 * 4096 / 1.5e-3)


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    args = bench.argparse.Namespace(steps=1, warmup=0, workload="c2", cpu_sample=32, gpus=2)
    bench.run_reference(args)
    assert capsys.readouterr().out == ""


def test_oracle_baseline_runs_every_shard_on_host_threads():
    sys.path.insert(0, ROOT)
    import bench
    from top_routing_grouped_gemm_gb300 import synth
    cfg = synth.config("c5", T=32, d=128, E=16, F=64)
    inp = synth.make_inputs(cfg, "cpu")
    args = bench.parse(["--cpu-threads", "3", "--cpu-tokens-per-thread", "2"])
    r = bench.cpu_baseline(inp, cfg, args)
    assert r["kind"] == "oracle" and r["cores"] == 3 and r["value"] > 0
    assert r["single_core"]["cores"] == 1 and r["single_core"]["units"] == 2
    assert "first 6 tokens" in r["sample"]


def test_reference_arm_line(capsys):
    sys.path.insert(0, ROOT)
    import json
    import bench
    args = bench.parse(["--impl", "reference", "--workload", "c1", "--steps", "2", "--warmup",
                        "1", "--cpu-threads", "2"])
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "tokens/s" and line["value"] > 0 and line["higher_is_better"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["cores"] == 2
    assert line["config"]["workload"].startswith("c1:")
