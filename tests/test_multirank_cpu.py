"""The multi-process path of bench.py on the CPU: world_size-2 process groups
over gloo, no GPU.  bench.py runs one replica of the verify step per GPU (the
step needs no collective); what crosses ranks is host bookkeeping -- the
slowest rank's time, the whole-job throughput -- and the reference arm runs on
rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(times[rank], dist, "cpu")
    gbs = bench.job_gbs(world, 1_000_000, 10, ms)
    dist.barrier()
    out.put((rank, ms, gbs))
    dist.destroy_process_group()


@pytest.mark.parametrize("times", [(12.5, 10.0), (3.0, 7.25)])
def test_slowest_rank_sets_the_job_time(times):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, list(times), q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slow = max(times)
    for rank, ms, gbs in res:
        assert ms == slow
        # two replicas of 1 MB per step, 10 steps, in the slowest rank's time
        assert gbs == pytest.approx(2 * 1_000_000 * 10 / (slow / 1e3) / 1e9)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.5, None, "cpu") == 4.5
    assert bench.job_gbs(1, 4_737_024, 1, 1.0) == pytest.approx(4.737024)


def test_reference_arm_under_two_ranks_prints_once():
    """`bench.py --impl reference` launched like the native arm with two ranks:
    rank 0 times the oracle and prints one line, rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    # the same workload description as the native arm's line
    sys.path.insert(0, ROOT)
    import bench
    assert d["config"] == bench.headline_config()
