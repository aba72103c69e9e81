"""The bench's multi-rank host logic on CPU (gloo, world size 2).

The path shards with no exchange: under torchrun each rank runs an independent
replica of the workload, and the only cross-rank steps are a barrier around the
timed region and the max over ranks of the timings (the slowest replica sets
the job's time); the whole-job value counts every replica's bytes. These run
here as two gloo processes on 127.0.0.1, with no GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r "measured" r+1 ms per step and 10-r ms end to end
        ms, e2e = bench.max_over_ranks([rank + 1.0, 10.0 - rank], dist, "cpu")
        value = bench.job_gbs(world, 1_000_000, ms)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "e2e": e2e, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo(tmp_path):
    world = 2
    ctx = torch.multiprocessing.get_context("spawn")
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r in res:
        assert r["ms"] == 2.0            # max of 1, 2
        assert r["e2e"] == 10.0          # max of 10, 9
        # 2 replicas x 1 MB in 2 ms = 1 GB/s
        assert abs(r["value"] - 1.0) < 1e-12


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2], None, "cpu") == [1.5, 2.0]
    assert abs(bench.job_gbs(1, 5e9, 1000.0) - 5.0) < 1e-12


def test_reference_arm_prints_on_rank_0_only(tmp_path):
    """Under torchrun with 2 ranks the reference arm prints one JSON line from
    rank 0; rank 1 exits 0 without work."""
    env = dict(os.environ, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--steps", "1", "--warmup", "3", "--cpu-seconds", "0.5"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
