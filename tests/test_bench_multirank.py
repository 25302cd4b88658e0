"""bench.py's multi-rank path on CPU (gloo, world size 2): timings reduce to
the slowest rank, throughput counts every rank's tokens, and the reference
arm runs on rank 0 only."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.reduce_max([10.0 + rank, 5.0 - rank], True, "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_timings_reduce_to_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(world))
    assert res[0] == res[1] == [11.0, 5.0]


def test_job_throughput_counts_all_ranks():
    assert bench.job_throughput(4, 32, 100, 200.0) == pytest.approx(4 * 32 * 100 / 0.2)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.main.__globals__["argparse"].Namespace(steps=3, warmup=3)
    assert bench.run_reference(args, bench.inputs.CONFIGS["decode"]) == 0


def test_reference_arm_prints_its_line_on_cpu():
    """The whole reference arm (the oracle, timed) on the small configuration,
    run as the driver runs it; the JSON line carries the contract's keys."""
    import json
    import subprocess
    import sys
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, bench.__file__, "--impl", "reference", "--config", "tiny",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                       env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2
    for k in ("metric", "unit", "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["cpu_baseline"]["kind"] == "oracle"
