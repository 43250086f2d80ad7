"""Host logic of the multi-rank benchmark, on CPU with gloo (world size 2):
the slowest rank's time decides the whole-job value, and under torchrun the
reference arm runs on rank 0 alone while the other ranks exit cleanly."""
import json
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


def _worker(rank, world, port, local_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    total = bench.max_over_ranks(local_ms[rank], world, dist, "cpu")
    value = bench.job_value(32, world, 10, total)
    out.put((rank, total, value))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world, local_ms = 2, [3.0, 5.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, local_ms, q))
             for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, value in got:
        assert total == 5.0  # every rank sees the slowest rank's time
        # 2 ranks x 32 queries x 10 steps in 5 ms
        assert value == pytest.approx(2 * 32 * 10 / 5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_value(16, 1, 4, 2.0) == pytest.approx(16 * 4 / 2e-3)


def test_dominant_stage_is_the_slowest_counted_one():
    sys.path.insert(0, ROOT)
    import bench
    alg = {"indexer_topk": {"bytes": 1}, "attention": {"bytes": 1}}
    assert bench.dominant_stage({"indexer_topk": 5.0, "attention": 1.5}, alg) == "indexer_topk"
    assert bench.dominant_stage({"indexer_topk": 1.0, "attention": 1.5, "x": 9.0},
                                alg) == "attention"


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload",
           "csa_decode_tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
