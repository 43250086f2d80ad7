#!/usr/bin/env python
"""Benchmark of the CSA / HCA hot path on B300 GPUs (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--cpu-seconds S] [--no-cpu-baseline]

A step is one pass of the workload's hot path over one batch of synthetic
inputs resident in HBM (see synth.WORKLOADS; default: CSA decode at 128K
context, batch 32).  The whole step is captured once as a CUDA graph and
replayed (each stage is also captured and timed on its own for the
breakdown); L2 is flushed (a 2x-L2 write, then a 2x-L2 read) before every timed
step, outside the
timed events.  ``value`` is whole-job queries/s (tokens/s for prefill) over
all ranks; ``e2e`` is the same metric through the public Python API with the
step's inputs copied from pinned host memory and its output copied back
inside the timed region.  ``roofline`` rates the dominant stage (the one that
takes the most time per step) against the measured peaks in
MEASURED_PEAKS.json.  ``cpu_baseline`` times the CPU oracle
on a bounded sample on this host.  ``--impl reference`` times only the CPU
oracle, as the reference arm.

Under torchrun each rank runs its own batch (weak scaling, no collective in
the data path); rank 0 prints the line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "CSA/HCA decode queries/s and achieved HBM GB/s vs peak at 128K and 1M context"
DEFAULT_WORKLOAD = "csa_decode_128k"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ---------------------------------------------------------------- workload arithmetic

def units(wl) -> int:
    """Queries per step: decode = sequences, prefill = new tokens."""
    return wl.B * wl.T


def unit_name(wl) -> str:
    return "tokens/s" if wl.kind == "csa_prefill" else "queries/s"


def n_vis_decode(wl):
    return [min(n // wl.m, n // wl.m) for n in wl.lens]


def idx_row_bytes(wl) -> int:
    """Bytes of one indexer key or query-head vector: bf16 codes; E4M3 codes +
    an fp32 scale; FP4 codes (two per byte) + one E4M3 scale per 16 channels."""
    if wl.idx_fp4:
        return wl.d_I // 2 + wl.d_I // 16
    if wl.idx_fp8:
        return wl.d_I + 4
    return wl.d_I * 2


def cmp_row_bytes(wl) -> int:
    """Bytes of one compressed K/V entry pair: bf16 K and V rows, or FP8
    storage (K: 64 E4M3 codes + fp32 scale + 64 bf16 RoPE channels; V: 128
    E4M3 codes + fp32 scale)."""
    if getattr(wl, "kv_fp8", False):
        return (64 + 4 + 64 * 2) + (wl.D + 4)
    return 2 * wl.D * 2


def algorithmic(wl) -> dict:
    """Algorithmic bytes (HBM) or FLOPs per stage per step, from the method's
    own data movement: every byte a stage must read or write at least once."""
    D, H, W = wl.D, wl.H, wl.W
    qo = 2 * H * D * 2  # q in + out, bf16
    crow = cmp_row_bytes(wl)
    if wl.kind == "hca_decode":
        nb = sum(n // wl.m * crow + min(W, n) * 2 * D * 2 for n in wl.lens)
        return {"attention": {"bytes": nb + wl.B * qo}}
    if wl.kind == "csa_decode":
        row, qrow = idx_row_bytes(wl), idx_row_bytes(wl)
        idx_b = sum(nv * row for nv in n_vis_decode(wl)) + wl.B * (
            wl.H_I * qrow + wl.H_I * 4 + wl.k * 4)
        att_b = sum(min(wl.k, n // wl.m) * crow + min(W, n) * 2 * D * 2
                    for n in wl.lens) + wl.B * qo
        st = {"indexer_topk": {"bytes": idx_b}, "attention": {"bytes": att_b}}
        if wl.proj_groups:
            # the weights once, the attention output in, the projection out
            K = (H // wl.proj_groups) * D
            st["out_proj"] = {"bytes": wl.proj_groups * wl.proj_dim * K * 2 + wl.B * H * D * 2
                              + wl.B * wl.proj_groups * wl.proj_dim * 2}
        if wl.stream_compress:
            per_seq = wl.m * (2 * D * 2 + wl.d_I * 2) + 2 * D * 2 + idx_row_bytes(wl)
            weights = (2 * D * D + wl.d_I * wl.d_I) * 2 + wl.m * (2 * D + wl.d_I) * 4
            st["compress"] = {"bytes": wl.B * per_seq + weights}
        return st
    # prefill: contraction FLOPs of the indexer and the attention
    nvis = [min(wl.N_cap, (wl.L + t + 1) // wl.m) for t in range(wl.T)]
    idx_f = wl.B * sum(nvis) * wl.H_I * wl.d_I * 2
    att_f = wl.B * wl.T * H * (wl.k + W) * D * 4
    # compression: each of the T/m new blocks evaluates span gate logits per
    # channel, a d x d contraction per token of its span, for K, V (d = D)
    # and the indexer keys (d = d_I)
    cmp_f = wl.B * (wl.T // wl.m) * wl.cspan * (2 * D * D + wl.d_I * wl.d_I) * 2
    return {"indexer_topk": {"flops": idx_f}, "attention": {"flops": att_f},
            "compress": {"flops": cmp_f}}


def kernel_algorithmic(wl, name: str) -> dict:
    """Algorithmic bytes or FLOPs of one launch of the kernel that
    ``kernel_probe`` runs alone: the indexer's scoring reads each visible key
    row once plus the query rows and head weights (the method's bytes); the
    fp32 score it writes per visible entry is workspace traffic, not the
    method's, and is reported beside them ("overhead_bytes"), not counted in
    the roofline.  The attention kernels are their whole stage."""
    if name == "indexer_score":
        row, qrow = idx_row_bytes(wl), idx_row_bytes(wl)
        nv = sum(n_vis_decode(wl))
        return {"bytes": nv * row + wl.B * wl.H_I * (qrow + 4), "overhead_bytes": nv * 4}
    return algorithmic(wl)[name]


# ---------------------------------------------------------------- ranks

def max_over_ranks(x: float, world: int, dist=None, device="cpu") -> float:
    """The maximum of a per-rank number over all ranks (the slowest rank's
    time decides the whole job's throughput)."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: int, world: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time."""
    return units_per_rank * world * steps / (total_ms / 1e3)


# ---------------------------------------------------------------- environment

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# the source file of each kernel whose DRAM traffic the bench reports
KERNEL_SOURCE = {"indexer_score": "indexer.cu", "indexer_gemm": "indexer_gemm.cu",
                 "attention": "attn.cu", "compress": "compress.cu", "out_proj": "out_proj.cu"}


def src_hash(kernel: str = None) -> str:
    """Hash of a kernel's source file and every shared header (all of csrc
    when no kernel is named)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_28_b300", "csrc")
    mine = KERNEL_SOURCE.get(kernel)
    for n in sorted(os.listdir(csrc)):
        if mine and n.endswith(".cu") and n != mine:
            continue
        with open(os.path.join(csrc, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def traffic_record(wl_name: str, kernel: str):
    """DRAM bytes per launch of the kernel from the committed ncu summary, or
    None if absent or taken on other sources of that kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(wl_name, {}).get(kernel)
    if not rec or rec.get("src_hash") != src_hash(kernel):
        return None
    return rec.get("dram_bytes")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


class L2Flush:
    """Evicts L2 between timed steps: writes one 2x-L2 buffer, then reads a
    second one, so that L2 ends up holding clean unrelated lines (a write-only
    flush would leave dirty lines whose write-back lands in the timed step)."""

    def __init__(self, l2_bytes: int, dev):
        self.w = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
        self.r = torch.ones(2 * l2_bytes // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.sink = self.r.sum()


# ---------------------------------------------------------------- CPU oracle leg

class OracleRunner:
    """The CPU oracle run on a bounded sample of the workload (``units`` per call)."""

    def __init__(self, wl, inp: dict, n_units: int):
        import oracle  # the oracle is test infrastructure: only this leg uses it
        from oracle.feed import idx_dtype, oracle_inputs
        self.o = oracle
        self.idx_dtype = idx_dtype(wl)
        self.wl = wl
        self.n = n_units
        self.arr = oracle_inputs(wl, inp, n_units)

    def __call__(self):
        o, wl, a = self.o, self.wl, self.arr
        if wl.kind == "hca_decode":
            o.hca_decode(a["q"], a["k_cmp"], a["v_cmp"], a["n_cmp"], wl.m, a["k_win"], a["v_win"],
                         a["seq_len"], wl.W, a["sink"], 1.0, a["raw_base"])
            return
        if wl.kind == "csa_decode":
            if wl.stream_compress:
                for s in ("k", "v", "idx"):
                    y = o.compress(a["raw_new_" + s], *a["gate_" + s], wl.m, 0, 1)
                    if s == "idx" and wl.idx_fp4:
                        o.quantize_fp4_rows(y)
                    elif s == "idx" and wl.idx_fp8:
                        o.quantize_e4m3_rows(y)
                    else:
                        o.quantize_bf16(y)
            sc, nv = o.indexer_scores(a["q_idx"], a["w"], a["k_idx"], a["q_pos"], a["n_cmp"],
                                      wl.m, self.idx_dtype,
                                      a.get("q_scale"), a.get("k_scale"))
            idx = o.topk(sc, nv, wl.k)
            ro, _ = o.csa_decode(a["q"], a["k_cmp"], a["v_cmp"], idx[:, 0, :], a["k_win"],
                                 a["v_win"], a["seq_len"], wl.W, a["sink"], 1.0, a["raw_base"])
            if wl.proj_groups:
                o.grouped_out_proj(o.quantize_bf16(ro), a["W_o"])
            return
        # prefill sample: the sampled tokens' blocks, scores, top-k, attention
        for s in ("k", "v", "idx"):
            o.quantize_bf16(o.compress(a["raw_new_" + s], *a["gate_" + s], wl.m, a["block0"],
                                       a["n_blocks"]))
        sc, nv = o.indexer_scores(a["q_idx"], a["w"], a["k_idx"], a["q_pos"], a["n_cmp"], wl.m)
        idx = o.topk(sc, nv, wl.k)
        o.csa_prefill(a["q"], a["k_cmp"], a["v_cmp"], idx, a["k_raw"], a["v_raw"], a["q_pos"],
                      wl.W, a["sink"], 1.0, a["raw_base"])


def oracle_sample_units(wl, cores: int) -> int:
    if wl.kind == "csa_prefill":
        return max(8, min(64, 2 * cores))
    return max(1, min(wl.B, cores))


def time_oracle(runner, budget_s: float):
    t0 = time.perf_counter()
    reps = 0
    while True:
        runner()
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return reps * runner.n / el, reps, el


# ---------------------------------------------------------------- feed probes

def run_probes(dev, l2_bytes: int):
    """`--probe`: the read rates behind the kernels' rooflines, one JSON line
    each (mean of 10 timed launches after 3 warm-up ones, L2 flushed clean
    before each).  (1) a contiguous stream read once, the size of the
    csa_decode_128k indexer keys (134 MB), for several CTAs per SM and loads
    in flight; (2) 512-byte row gathers into shared memory, 34 stages x 64
    rows per CTA like the prefill attention: 4096 CTAs from an L2-resident
    table of the csa_prefill_4k caches' size (43 MB: 88,000 rows), and 888
    CTAs reading distinct rows of a 1 GB table (every row from DRAM); for
    ring depths of 2, 4 and 6 stages (3, 1 and 1 CTAs per SM by shared
    memory), with 16-byte cp.async copies by 256 or 512 threads and with TMA
    tile::gather4 issued by one, four or eight warps; each CTA's row indices
    are staged in shared memory first."""
    import sparse_attention_28_b300 as csa
    flush = L2Flush(l2_bytes, dev)
    sink = torch.zeros(1, dtype=torch.float32, device=dev)

    def timed(fn, flush_each=True):
        for _ in range(3):
            fn()
        ms = []
        for _ in range(10):
            if flush_each:
                flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize(dev)
            ms.append(a.elapsed_time(b))
        return sum(ms) / len(ms)

    keys = torch.zeros(32 * 32768 * 128, dtype=torch.uint8, device=dev)
    for cps in (1, 2, 3):
        for k in (1, 4, 8):
            ms = timed(lambda: csa.probe_stream_read(keys, sink, cps, k))
            print(json.dumps({"probe": "stream_read", "bytes": keys.numel(), "ctas_per_sm": cps,
                              "in_flight": k, "us": round(ms * 1e3, 2),
                              "GB/s": round(keys.numel() / ms / 1e6, 1)}), flush=True)
    del keys
    stages = 34
    g = torch.Generator(device="cpu").manual_seed(1)
    # an L2-resident table (the csa_prefill_4k caches' size), indices drawn
    # with repeats, 4096 CTAs; and a 1 GB table read without repeats (every
    # row from DRAM), 888 CTAs
    for where, n_rows, ctas in (("l2", 88000, 4096), ("dram", 1 << 21, 888)):
        n_idx = ctas * stages * 64
        table = torch.zeros((n_rows, 512), dtype=torch.uint8, device=dev)
        if where == "l2":
            idx = torch.randint(0, n_rows, (n_idx,), generator=g, dtype=torch.int32)
        else:
            idx = torch.randperm(n_rows, generator=g, dtype=torch.int32)[:n_idx]
        idx = idx.to(dev)
        moved = n_idx * 512
        for tma, wide, issuers, who in ((False, False, 0, "256 threads"),
                                        (False, True, 0, "512 threads"),
                                        (True, False, 1, "1 warp"), (True, False, 4, "4 warps"),
                                        (True, False, 8, "8 warps")):
            for ring in (2, 4, 6):
                # the L2 case keeps the table in L2 between launches; the
                # DRAM case flushes L2 before each launch
                ms = timed(lambda: csa.probe_row_gather(table, idx, ctas, stages, ring, sink,
                                                        tma, wide, issuers),
                           flush_each=where == "dram")
                print(json.dumps({
                    "probe": "row_gather", "copies": "tma_gather4" if tma else "cp.async",
                    "issuers": who,
                    "table": where, "rows": n_rows, "row_bytes": 512, "ctas": ctas,
                    "stages": stages, "ring": ring, "us": round(ms * 1e3, 1),
                    "GB/s": round(moved / ms / 1e6, 1)}), flush=True)
        del table, idx
    torch.cuda.synchronize(dev)
    if sink.item() == 2.0:
        print(json.dumps({"probe": "row_gather", "error": "a bounded wait gave up"}), flush=True)


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--probe", action="store_true",
                    help="time the feed probes (stream read, row gathers) instead of a step")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")

    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # one process per GPU: start them under torchrun and pass its status on
        sys.exit(relaunch_under_torchrun(args.gpus))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch one rank per GPU "
              f"(torchrun --nproc-per-node {args.gpus}) or drop --gpus", file=sys.stderr)
        sys.exit(2)
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    wl = synth.WORKLOADS[args.workload]
    cfg = {"workload": wl.name, "kind": wl.kind, "B": wl.B, "L": wl.L, "T": wl.T, "m": wl.m,
           "span": wl.cspan, "batch_invariant_keys_per_split": wl.batch_invariant,
           "out_proj": ({"groups": wl.proj_groups, "d_g": wl.proj_dim} if wl.proj_groups
                        else None),
           "H": wl.H, "D": wl.D, "k": wl.k, "window": wl.W, "H_I": wl.H_I, "d_I": wl.d_I,
           "indexer_dtype": "e2m1" if wl.idx_fp4 else "e4m3" if wl.idx_fp8 else "bf16",
           "kv_dtype": "e4m3 (RoPE channels bf16)" if wl.kv_fp8 else "bf16",
           "stream_compress": wl.stream_compress, "parallelism": f"replicas{world}"}

    if args.impl == "reference":
        return run_reference(args, wl, cfg, world, rank)

    import torch.distributed as dist
    import sparse_attention_28_b300 as csa
    from sparse_attention_28_b300.steps import make_step

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    csa.lib()  # fail loudly now if the library is missing
    if args.probe:
        run_probes(dev, torch.cuda.get_device_properties(dev).L2_cache_size)
        return

    inp = synth.make_inputs(wl, seed=args.seed + 7919 * rank, device=dev)
    step = make_step(inp, dev)
    stages = step.stages()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # one CUDA graph per stage, replayed back to back
    graphs = []
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(torch.cuda.current_stream())
    for name, fn in stages:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn()
        graphs.append((name, g))
    torch.cuda.synchronize()
    for _, g in graphs:
        g.replay()
    torch.cuda.synchronize()

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(l2, dev)
    stream = torch.cuda.current_stream(dev)
    n_st = len(graphs)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_st + 1)]
           for _ in range(args.steps)]

    # the whole step as one CUDA graph: the timed region
    whole = step.graphed()
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]

    sampler = ClockSampler(dev.index)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.25)
    for i in range(args.steps):
        flush()
        ev0[i].record(stream)
        whole()
        ev1[i].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    step_ms = [ev0[i].elapsed_time(ev1[i]) for i in range(args.steps)]

    # per-stage breakdown (each stage its own graph, L2 flushed before each step)
    for i in range(args.steps):
        flush()
        evs[i][0].record(stream)
        for s, (_, g) in enumerate(graphs):
            g.replay()
            evs[i][s + 1].record(stream)
    torch.cuda.synchronize()
    stage_ms = {name: statistics.mean(evs[i][s].elapsed_time(evs[i][s + 1])
                                      for i in range(args.steps))
                for s, (name, _) in enumerate(graphs)}
    total_ms = max_over_ranks(sum(step_ms), world, dist, dev)
    ms_per_step = total_ms / args.steps  # mean over the K timed steps
    median_ms = max_over_ranks(statistics.median(step_ms), world, dist, dev)
    value = job_value(units(wl), world, args.steps, total_ms)

    # e2e: public API, inputs from pinned host memory, result back to host
    e2e = run_e2e(args, wl, inp, step, dev, world, dist)

    # roofline of the dominant kernel: launched alone (its own CUDA graph) on
    # the step's buffers, L2 flushed before every launch, CUDA events
    peaks, peaks_src = load_peaks()
    alg = algorithmic(wl)
    kname, kfn = step.kernel_probe()
    kfn()
    torch.cuda.synchronize()
    kg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(kg, stream=cap):
        kfn()
    torch.cuda.synchronize()
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        kev[i][0].record(stream)
        kg.replay()
        kev[i][1].record(stream)
    torch.cuda.synchronize()
    k_times = [a.elapsed_time(b) for a, b in kev]
    k_ms = statistics.mean(k_times)
    kalg = kernel_algorithmic(wl, kname)
    if "bytes" in kalg:
        achieved = kalg["bytes"] / (k_ms / 1e3) / 1e9
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "unit": "GB/s"}
    else:
        achieved = kalg["flops"] / (k_ms / 1e3) / 1e12
        peak = float(peaks["bf16_tflops"])
        roof = {"bound": "tensor", "unit": "TFLOP/s"}
    roof.update({"achieved": round(achieved, 2), "peak": peak, "frac": round(achieved / peak, 4),
                 "traffic": traffic_record(wl.name, kname), "kernel": kname,
                 "kernel_ms": round(k_ms, 5),
                 "kernel_ms_median": round(statistics.median(k_times), 5), "algorithmic": kalg,
                 "peak_source": peaks_src + " (burst)"})

    stage_report = {}
    for name, ms in stage_ms.items():
        r = {"ms": round(ms, 5)}
        a = alg.get(name, {})
        if "bytes" in a:
            r["GB/s"] = round(a["bytes"] / (ms / 1e3) / 1e9, 1)
        if "flops" in a:
            r["TFLOP/s"] = round(a["flops"] / (ms / 1e3) / 1e12, 1)
        stage_report[name] = r
    step_bytes = sum(a.get("bytes", 0) for a in alg.values())
    if step_bytes:
        stage_report["step_GB/s"] = round(step_bytes / (ms_per_step / 1e3) / 1e9, 1)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args, wl, inp)

    launches = launches_per_step(wl, csa) * args.steps
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": unit_name(wl), "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "ms_per_step_median": round(median_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e2m1-indexer+bf16" if wl.idx_fp4 else "e4m3-indexer+bf16" if wl.idx_fp8
                  else "bf16"), "data": "synthetic",
        "config": dict(cfg, l2="flushed before every device-timed step (2x L2 write + 2x L2 "
                              "read, untimed); the end-to-end loop runs its steps back to back "
                              "on e2e.replicas copies of the workload in turn, so that no step "
                              "finds its data in L2",
                       timing="whole step as one CUDA graph, CUDA events per step; "
                              "ms_per_step and value use the mean of the K timed steps "
                              "(their total / K), ms_per_step_median beside it; stages and "
                              "the roofline kernel timed separately (means)"),
        "roofline": roof, "stages": stage_report, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": clocks, "gpu_launches": launches,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def relaunch_under_torchrun(n: int) -> int:
    """Run this same command as n ranks (one per GPU) under torchrun on this
    node, rendezvous on 127.0.0.1; returns torchrun's exit status."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def launches_per_step(wl, csa) -> int:
    """Kernels of the library launched per step (memsets not counted)."""
    n = 0
    q = units(wl)
    if wl.kind in ("csa_decode", "csa_prefill"):
        n += 2 * ((q + 255) // 256)  # score, select per chunk of 256 queries
        n += 1 + (csa.attn_workspace(wl.B, wl.T, wl.H, wl.k + wl.W) > 0)
        if wl.stream_compress or wl.kind == "csa_prefill":
            n += 3
    else:
        n += 1 + (csa.attn_workspace(wl.B, 1, wl.H, wl.N_cap + wl.W) > 0)
    return n


def e2e_replicas(wl, l2_bytes: int) -> int:
    """Step replicas the end-to-end loop uses in turn: enough that a step's
    caches were last touched two L2 sizes of other traffic ago (so no step
    finds its data in L2, as with the flush between device-timed steps), at
    least two so that copies and compute can overlap, at most eight."""
    per_step = max(1, sum(a.get("bytes", 0) for a in algorithmic(wl).values()))
    if wl.kind == "csa_prefill":  # caches re-read within a step: count them once
        per_step = max(per_step, 3 * wl.N_cap * wl.D * 2 * wl.B)
    return int(min(8, max(2, math.ceil(2 * l2_bytes / per_step))))


def run_e2e(args, wl, inp, step, dev, world, dist):
    """End to end through the public API, as a serving loop runs it: every
    step copies its inputs (one buffer: queries, positions, lengths, indexer
    queries and weights) from pinned host memory to the device, runs the step
    (one CUDA graph of library calls) and copies its output back to pinned
    host memory.  Copies and compute are pipelined over three streams: the
    next step's upload and the previous step's download run while a step
    computes.  Steps use R replicas of the workload in turn (each its own
    caches and buffers), so that no step finds its data in L2.  The timed
    region is the whole loop, first upload to last download."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = min(e2e_replicas(wl, l2), max(1, args.steps))
    from sparse_attention_28_b300.steps import make_step
    reps = [step] + [make_step(inp, dev) for _ in range(R - 1)]
    host_in, host_out = [], []
    for r in reps:
        h = torch.empty(r.inputs.shape, dtype=torch.uint8, pin_memory=True)
        h.copy_(r.inputs)
        host_in.append(h)
        host_out.append(torch.empty(r.out.shape, dtype=r.out.dtype, pin_memory=True))
        r()  # warm-up outside the capture
    h2d = host_in[0].numel()
    d2h = host_out[0].numel() * host_out[0].element_size()
    torch.cuda.synchronize(dev)

    # the K pipelined steps as one CUDA graph (a serving loop would submit
    # them the same way; launching them one by one from Python cannot keep
    # up with steps of tens of microseconds)
    comp = torch.cuda.Stream(device=dev)
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    computed = [None] * R   # replica r's last step computed (its inputs and output free)
    downloaded = [None] * R  # replica r's last output copied to the host
    g = torch.cuda.CUDAGraph()
    comp.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.graph(g, stream=comp):
        up.wait_stream(comp)
        down.wait_stream(comp)
        for i in range(args.steps):
            r = i % R
            with torch.cuda.stream(up):
                if computed[r] is not None:
                    up.wait_event(computed[r])
                reps[r].inputs.copy_(host_in[r], non_blocking=True)
                uploaded = torch.cuda.Event()
                uploaded.record(up)
            comp.wait_event(uploaded)
            if downloaded[r] is not None:
                comp.wait_event(downloaded[r])
            reps[r]()
            computed[r] = torch.cuda.Event()
            computed[r].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(computed[r])
                host_out[r].copy_(reps[r].out, non_blocking=True)
                downloaded[r] = torch.cuda.Event()
                downloaded[r].record(down)
        comp.wait_stream(up)
        comp.wait_stream(down)
    torch.cuda.synchronize(dev)
    g.replay()  # once untimed (the graph's first launch uploads it)
    torch.cuda.synchronize(dev)
    for h in host_out:
        h.zero_()
    stream = torch.cuda.current_stream(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    g.replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    # the round trips really moved the steps' data: each replica's host copy
    # of its output equals its device output
    for r in range(min(R, args.steps)):
        assert torch.equal(host_out[r], reps[r].out.cpu()), "e2e output did not reach the host"
    total = max_over_ranks(t0.elapsed_time(t1), world, dist, dev)
    return {"value": round(job_value(units(wl), world, args.steps, total), 2),
            "unit": unit_name(wl), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(total / args.steps, 5), "pipelined": True, "replicas": R}


def cpu_baseline(args, wl, inp):
    import oracle
    cores = oracle.num_threads()
    n = oracle_sample_units(wl, cores)
    runner = OracleRunner(wl, inp, n)
    value, reps, el = time_oracle(runner, args.cpu_seconds)
    what = "tokens" if wl.kind == "csa_prefill" else "sequences"
    return {"value": round(value, 4), "unit": unit_name(wl), "cores": cores, "kind": "oracle",
            "sample": f"{n} {what} of the workload, full step each, repeated {reps}x "
                      f"in {el:.1f} s (fp64 C oracle, OpenMP)"}


def run_reference(args, wl, cfg, world, rank):
    """The reference arm: the CPU oracle as it stands, on host cores."""
    if rank != 0:
        return
    import oracle
    cores = oracle.num_threads()
    inp = synth.make_inputs(wl, seed=args.seed, device="cpu")
    n = oracle_sample_units(wl, cores)
    runner = OracleRunner(wl, inp, n)
    for _ in range(args.warmup):
        runner()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        runner()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = n * args.steps / total
    what = "tokens" if wl.kind == "csa_prefill" else "sequences"
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": unit_name(wl), "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": cfg, "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": unit_name(wl), "cores": cores,
                         "kind": "oracle",
                         "sample": f"{n} {what} of the workload per step (fp64 C oracle)"},
        "e2e": {"value": round(value, 4), "unit": unit_name(wl), "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
