"""Multi-process checks (world size 2, gloo, CPU) of bench.py's replica
logic: every rank runs the whole workload, the job's time is the slowest
rank's, its rate counts every replica's work, and the reference arm runs on
rank 0 alone (the other ranks exit 0 without work)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out = {
        "max": bench._max_over_ranks(3.5 * (rank + 1), "cpu"),
        "steps": int(bench._max_over_ranks(100 + 7 * rank, "cpu")),
        "env": bench._dist_env(),
    }
    dist.barrier()
    dist.destroy_process_group()
    queue.put((rank, out))


def test_max_over_ranks_with_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(queue.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    for rank in (0, 1):
        assert results[rank]["max"] == 7.0
        assert results[rank]["steps"] == 107
        assert tuple(results[rank]["env"][:2]) == (rank, 2)


def test_max_over_ranks_without_a_group():
    import bench
    assert bench._max_over_ranks(2.5, "cpu") == 2.5


def test_whole_job_rate_counts_every_replica():
    import bench
    # 10 steps of 1 TFLOP in 1000 ms on the slowest rank
    assert bench._whole_job_tflops(1, 1e12, 10, 1000.0) == pytest.approx(10.0)
    assert bench._whole_job_tflops(2, 1e12, 10, 1000.0) == pytest.approx(20.0)
    assert bench._whole_job_tflops(8, 1e12, 10, 2000.0) == pytest.approx(40.0)


def test_reference_arm_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("workload", [1, 2, 3, 4, 5, 6, 7, 8])
def test_reference_arm_runs_every_workload(workload):
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
           "--workload", str(workload)]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["dtype"] == "f64"


def test_e4m3_widens_exactly_to_bfloat16():
    """The reference arm evaluates the FP8 workload's sampled rows on
    bfloat16-widened inputs: every E4M3 code must survive the widening."""
    import torch
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
    f32 = codes.to(torch.float32)
    bf = codes.to(torch.bfloat16).to(torch.float32)
    nan = torch.isnan(f32)
    assert torch.equal(nan, torch.isnan(bf))
    assert torch.equal(f32[~nan], bf[~nan])
