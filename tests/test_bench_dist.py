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


def test_kernel_algorithmic_bytes():
    # the scoring kernel of a 128K-context decode batch: 32 queries over 32768
    # visible entries, each a 128-byte bf16 key row read and a 4-byte score
    # written, plus 4 heads x (128-byte query row + 4-byte weight) per query
    sys.path.insert(0, ROOT)
    import bench
    import synth
    wl = synth.WORKLOADS["csa_decode_128k"]
    # the fp32 score written per entry is workspace overhead, reported apart
    assert bench.kernel_algorithmic(wl, "indexer_score") == {
        "bytes": 32 * 32768 * 128 + 32 * 4 * (128 + 4), "overhead_bytes": 32 * 32768 * 4}
    # E4M3 keys: 64 code bytes + a 4-byte scale per row
    wl8 = synth.WORKLOADS["csa_decode_1m_fp8"]
    assert bench.kernel_algorithmic(wl8, "indexer_score") == {
        "bytes": 8 * 262144 * 68 + 8 * 4 * (68 + 4), "overhead_bytes": 8 * 262144 * 4}
    # FP4 keys: 32 code bytes + 4 E4M3 block scales per row
    wl4 = synth.WORKLOADS["csa_decode_1m_fp4"]
    assert bench.kernel_algorithmic(wl4, "indexer_score") == {
        "bytes": 8 * 262144 * 36 + 8 * 4 * (36 + 4), "overhead_bytes": 8 * 262144 * 4}
    hca = synth.WORKLOADS["hca_decode_1m"]
    assert bench.kernel_algorithmic(hca, "attention") == bench.algorithmic(hca)["attention"]


def test_oracle_sample_of_overlapping_prefill():
    # the CPU baseline's bounded sample of the overlap workload: its blocks
    # read span - m older rows (whole blocks), which the sample includes
    sys.path.insert(0, ROOT)
    import bench
    import synth
    wl = synth.WORKLOADS["csa_prefill_4k_overlap"]
    assert wl.cspan == 2 * wl.m
    inp = synth.make_inputs(wl, seed=0, device="cpu")
    assert inp["raw_idx"].shape[1] == wl.T + wl.m and inp["idx_base"] == wl.L - wl.m
    assert inp["gate_k"][1].shape == (wl.cspan, wl.D)
    run = bench.OracleRunner(wl, inp, 8)
    assert run.arr["block0"] == 1 and run.arr["raw_new_k"].shape[1] == wl.m * (1 + 2)
    run()


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


def test_gpus_flag_without_torchrun_starts_the_ranks():
    # --gpus 2 run as a plain process: bench.py starts two ranks itself and
    # the one line it prints says n_gpus 2
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--workload", "csa_decode_tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env={k: v for k, v in dict(os.environ, OMP_NUM_THREADS="2").items()
                            if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["n_gpus"] == 2


def test_gpus_flag_that_contradicts_the_launch_fails():
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--gpus", "4", "--steps", "1",
           "--warmup", "3", "--workload", "csa_decode_tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0"))
    assert r.returncode != 0
    assert "WORLD_SIZE=2" in r.stderr
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_fp8kv_algorithmic_bytes():
    sys.path.insert(0, ROOT)
    import bench
    import synth
    # FP8-stored entries: K 64 E4M3 codes + fp32 scale + 64 bf16 RoPE channels,
    # V 128 E4M3 codes + fp32 scale (328 B a pair instead of 512); window rows
    # stay bf16
    wl8, wl = synth.WORKLOADS["hca_decode_1m_fp8kv"], synth.WORKLOADS["hca_decode_1m"]
    assert bench.cmp_row_bytes(wl8) == 328 and bench.cmp_row_bytes(wl) == 512
    n = 8192 * 16
    d = bench.algorithmic(wl)["attention"]["bytes"] - bench.algorithmic(wl8)["attention"]["bytes"]
    assert d == n * (512 - 328)
    c8 = bench.algorithmic(synth.WORKLOADS["csa_decode_128k_fp8kv"])
    c = bench.algorithmic(synth.WORKLOADS["csa_decode_128k"])
    assert c["attention"]["bytes"] - c8["attention"]["bytes"] == 32 * 1024 * (512 - 328)
    assert c["indexer_topk"] == c8["indexer_topk"]
