"""The benchmark's several-rank logic (replicas, one per GPU) on CPU ranks over gloo: the
job time is the slowest rank's, the rate counts every rank's tokens, and the reference arm runs
on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(2.0 + 3.0 * rank, world, "cpu")
    rate = bench.job_rate(1000, world, ms)
    dist.barrier()
    q.put((rank, ms, rate))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate in got:
        assert ms == 5.0                      # the slower rank's 2.0 + 3.0
        assert rate == pytest.approx(1000 * world / 5e-3)


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, 1, "cpu") == 1.25
    assert bench.job_rate(4096, 1, 2.0) == pytest.approx(4096 / 2e-3)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    """The reference arm (the CPU oracle) prints one line whose config equals our arm's, whose
    steps each take the measured time it reports, and whose tokens per step are stated."""
    sys.path.insert(0, ROOT)
    import json
    import time

    import bench
    import moe_synth
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_fp32", "--steps", "3", "--warmup", "1"], env=env,
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 3
    assert line["config"] == bench.config_of(moe_synth.TINY, 1)
    assert line["steps"] * line["ms_per_step"] / 1e3 <= wall
    assert line["tokens_per_step"] >= 1
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
