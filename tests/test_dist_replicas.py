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


def test_profiled_traffic_covers_its_own_workload_only(tmp_path, monkeypatch):
    """DRAM bytes per launch are reported only for the workload the capture
    covers, and only while the kernel sources match the capture."""
    sys.path.insert(0, ROOT)
    import bench
    csv_path = tmp_path / "cap.csv"
    hdr = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
           '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
           '"Metric Value"\n')
    rows = []
    for i, (rd, wr) in enumerate([(60.0, 1.5), (62.0, 1.5)]):
        for m, v in (("dram__bytes_read.sum", rd), ("dram__bytes_write.sum", wr)):
            rows.append(f'"{i}","1","python","h","void sekv::decode_kernel<2>(sekv::DecodeParams)",'
                        f'"1","7","(256, 1, 1)","(19, 8, 1)","0","10.3","Command line profiler '
                        f'metrics","{m}","Mbyte","{v}"\n')
    rows.append('"2","1","python","h","other_kernel","1","7","(1,1,1)","(1,1,1)","0","10.3",'
                '"x","dram__bytes_read.sum","Mbyte","999"\n')
    csv_path.write_text("==PROF== noise\n" + hdr + "".join(rows))
    out = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(out))
    bench.write_traffic(str(csv_path), "llama3_8b_128k", 8.0, "cmd")
    # mean of (61.5, 63.5) MB per captured launch, scaled by 8
    assert bench.profiled_traffic("llama3_8b_128k") == 8 * 62_500_000
    assert bench.profiled_traffic("qwen2_7b_stress") is None
    monkeypatch.setattr(bench, "decode_source_hash", lambda: "changed")
    assert bench.profiled_traffic("llama3_8b_128k") is None


def test_reference_arm_times_units_and_names_them():
    """--impl reference: each timed sample is one (layer, sequence, KV head)
    unit, ms_per_step is that sample's time (so steps x ms_per_step is the
    timed wall time), the value is extrapolated to whole steps, and the
    config is the sekv arm's."""
    import json
    import subprocess
    sys.path.insert(0, ROOT)
    import bench
    import synth
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3",
                        "--warmup", "1", "--config", "llama3_8b_32k", "--layers", "2"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    w = synth.get_config("llama3_8b_32k", layers=2)
    assert line["impl"] == "reference" and line["steps"] == 3
    assert line["units_per_step"] == 1 * 8 * 2
    assert line["value"] == pytest.approx(1e3 / (line["ms_per_step"] * 16), rel=1e-9)
    assert line["config"] == bench.decode_config(w, 1)
