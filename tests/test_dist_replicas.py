"""Multi-process (gloo, world size 2) checks of the replica logic of bench.py:
the path has no exchange step, so N GPUs run N replicas, the timed region is
bracketed by a barrier on every rank and the slowest rank's time counts."""

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    class A:
        pass

    ws, r, local = bench.dist_setup(A())
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    # each rank "measured" a different time; every rank must see the maximum
    ms = 10.0 + 5.0 * rank
    mx = bench.max_over_ranks(ms, ws)
    out[rank] = mx
    bench.barrier(ws)
    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="gloo replica test runs on CPU hosts")
def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 15.0


def test_whole_job_rate_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench

    # 2 ranks x 100 steps in 50 ms (slowest rank) -> 4000 steps/s for the job
    assert bench.whole_job_rate(100, 50.0, 2) == pytest.approx(4000.0)
    assert bench.whole_job_rate(100, 50.0, 1) == pytest.approx(2000.0)


def test_reference_arm_is_decode_only():
    """The reference arm times the oracle on the decode path; other paths say
    so on one JSON line instead of timing this library's kernels."""
    import json
    import subprocess
    for path in ("build", "fullkv"):
        r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--path", path],
                           capture_output=True, text=True, timeout=300, cwd=ROOT)
        assert r.returncode == 0, r.stderr
        line = json.loads(r.stdout.strip().splitlines()[-1])
        assert line["impl"] == "reference" and "unavailable" in line


def test_profiled_traffic_covers_its_own_workload_only():
    """The committed ncu summary's DRAM bytes are reported only for the
    workload it was taken on (and only while the kernel sources match)."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.profiled_traffic("qwen2_7b_stress") is None
    t = bench.profiled_traffic("llama3_8b_128k")
    assert t is None or (isinstance(t, int) and t > 0)
