"""Seeded synthetic inputs for the CSA / HCA hot path.

This module only draws random tensors and lays them out; it holds none of the
method's arithmetic.  Both the CUDA path (tests, benchmark) and the CPU oracle
consume what it returns.

Recipe (the same for every workload):

* one ``torch.Generator`` per tensor, seeded ``seed * 1000 + tensor_id``;
* values are N(0, 1) drawn in fp32, then cast to bf16 by torch (round to
  nearest even); the attention query is multiplied by 1/sqrt(128) before the
  cast;
* sink logits and indexer head weights are N(0, 1) fp32;
* gate projections W are N(0, 1)/sqrt(d) cast to bf16, positional biases are
  N(0, 1) fp32;
* FP8 indexer keys / queries: N(0, 1) fp32 values x, a per-row fp32 scale
  s = max|x| / 448, codes = torch's float8_e4m3fn cast of x / s (torch's
  library cast, not the oracle's codec nor the kernels' conversion);
* FP8-stored compressed K/V (mixed precision): K's 64 non-RoPE channels and
  V's 128 channels drawn as the FP8 indexer keys are (own scale per entry and
  stream), K's 64 RoPE channels N(0, 1) bf16;
* compressed caches of decode workloads are drawn directly (they are inputs
  of the decode calls); raw caches hold only the rows a step may read (the
  sliding window, plus the newest block where a step compresses one).

The page text gives million-token workloads but no data; these shapes stand in
for them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

D_HEAD = 128
WINDOW = 128
H_IDX = 4
D_IDX = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    """One workload shape.  ``kind`` is csa_decode, hca_decode or csa_prefill."""
    name: str
    kind: str
    B: int
    L: int                   # raw context length incl. the current token (decode)
    m: int                   # compression ratio (m' for HCA)
    H: int
    k: int = 0               # top-k (CSA)
    T: int = 1               # query tokens per sequence
    idx_fp8: bool = False    # FP8 E4M3 indexer keys / queries
    idx_fp4: bool = False    # FP4 E2M1 indexer keys / queries (E4M3 scale per 16 channels)
    stream_compress: bool = False  # decode step compresses the newest block first
    D: int = D_HEAD
    W: int = WINDOW
    H_I: int = H_IDX
    d_I: int = D_IDX
    sink: bool = True
    seq_lens: Optional[tuple] = None  # ragged decode lengths (default: all L)
    span: int = 0            # raw tokens per compressed block (0: m, no overlap)
    batch_invariant: int = 0  # > 0: decode attention with fixed key splits of this size
    proj_groups: int = 0     # > 0: grouped output projection after the attention (G groups)
    proj_dim: int = 0        # output channels per projection group (d_g)
    kv_fp8: bool = False     # compressed K/V stored in FP8 (E4M3 + scale; K's RoPE half bf16)

    @property
    def cspan(self) -> int:
        """Tokens each compressed block is formed from (>= m; m: no overlap)."""
        return self.span or self.m

    @property
    def N_cap(self) -> int:
        if self.kind == "csa_prefill":
            return (self.L + self.T) // self.m
        return max(self.lens) // self.m

    @property
    def lens(self) -> tuple:
        return tuple(self.seq_lens) if self.seq_lens else (self.L,) * self.B


# The five workloads of the hot path.  Decode: L counts the current token.
# Prefill: L is the context already cached, T new tokens follow it.
WORKLOADS = {
    "csa_decode_tiny": Workload("csa_decode_tiny", "csa_decode", B=1, L=8192, m=4, H=16,
                                k=256),
    "csa_decode_128k": Workload("csa_decode_128k", "csa_decode", B=32, L=131072, m=4, H=64,
                                k=1024),
    "hca_decode_1m": Workload("hca_decode_1m", "hca_decode", B=16, L=1048576, m=128, H=64),
    "csa_prefill_4k": Workload("csa_prefill_4k", "csa_prefill", B=1, L=262144, m=4, H=64,
                               k=2048, T=4096),
    "csa_decode_1m_fp8": Workload("csa_decode_1m_fp8", "csa_decode", B=8, L=1048576, m=4,
                                  H=64, k=2048, idx_fp8=True, stream_compress=True),
    # the same with the FP4 indexer path
    "csa_decode_1m_fp4": Workload("csa_decode_1m_fp4", "csa_decode", B=8, L=1048576, m=4,
                                  H=64, k=2048, idx_fp4=True, stream_compress=True),
    # the 128K decode followed by the grouped output projection (8 groups of 8
    # heads, 512 output channels each: a 4096-wide output)
    "csa_decode_128k_proj": Workload("csa_decode_128k_proj", "csa_decode", B=32, L=131072, m=4,
                                     H=64, k=1024, proj_groups=8, proj_dim=512),
    # the 128K decode with batch-invariant attention (fixed 320-key splits)
    "csa_decode_128k_bi": Workload("csa_decode_128k_bi", "csa_decode", B=32, L=131072, m=4,
                                   H=64, k=1024, batch_invariant=320),
    # the 128K CSA decode and the 1M HCA decode over an FP8-stored compressed
    # KV cache (K: 64 E4M3 non-RoPE channels + scale, 64 bf16 RoPE channels;
    # V: 128 E4M3 channels + scale)
    "csa_decode_128k_fp8kv": Workload("csa_decode_128k_fp8kv", "csa_decode", B=32, L=131072,
                                      m=4, H=64, k=1024, kv_fp8=True),
    "hca_decode_1m_fp8kv": Workload("hca_decode_1m_fp8kv", "hca_decode", B=16, L=1048576,
                                    m=128, H=64, kv_fp8=True),
    # overlapping compression: each block formed from 2m tokens (its own and
    # the previous block's)
    "csa_prefill_4k_overlap": Workload("csa_prefill_4k_overlap", "csa_prefill", B=1, L=262144,
                                       m=4, H=64, k=2048, T=4096, span=8),
}


def _gen(seed: int, tid: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + tid)
    return g


def randn(shape, seed: int, tid: int, device="cpu", scale: float = 1.0,
          dtype=torch.bfloat16) -> torch.Tensor:
    x = torch.randn(shape, generator=_gen(seed, tid, device), device=device,
                    dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(dtype)


def randn_fp8_rows(shape, seed: int, tid: int, device="cpu"):
    """FP8 E4M3 codes (as uint8) and per-row fp32 scales for N(0,1) values."""
    x = torch.randn(shape, generator=_gen(seed, tid, device), device=device,
                    dtype=torch.float32)
    amax = x.abs().amax(dim=-1)
    s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (x / s.unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, s.contiguous()


def randn_kv8(B: int, N: int, seed: int, tid: int, device="cpu", n_rope: int = 64):
    """An FP8-stored compressed K/V cache of N(0,1) values: K's first
    D_HEAD - n_rope channels as E4M3 codes with per-entry scales
    (:func:`randn_fp8_rows`), its last n_rope channels bf16, V's D_HEAD
    channels as E4M3 codes with per-entry scales.
    Returns (k_nope u8 [B,N,D-n_rope], k_scale f32 [B,N], k_rope bf16
    [B,N,n_rope], v u8 [B,N,D], v_scale f32 [B,N])."""
    k_nope, k_scale = randn_fp8_rows((B, N, D_HEAD - n_rope), seed, tid, device)
    k_rope = randn((B, N, n_rope), seed, tid + 1, device)
    v, v_scale = randn_fp8_rows((B, N, D_HEAD), seed, tid + 2, device)
    return k_nope, k_scale, k_rope, v, v_scale


def rand_fp4_rows(shape, seed: int, tid: int, device="cpu"):
    """Random FP4-stored vectors of shape[-1] channels: uniformly drawn E2M1
    codes (two per byte, uint8 [..., d/2]) and E4M3 block-scale codes, one per
    16 channels (uint8 [..., d/16]), drawn from 0x28 .. 0x47 (scales 2^-2 ..
    2^1.9): random bytes, no arithmetic of the method."""
    *lead, d = shape
    g = _gen(seed, tid, device)
    codes = torch.randint(0, 256, (*lead, d // 2), generator=g, device=device,
                          dtype=torch.int32).to(torch.uint8)
    scales = torch.randint(0x28, 0x48, (*lead, d // 16), generator=g, device=device,
                           dtype=torch.int32).to(torch.uint8)
    return codes, scales


def make_inputs(wl: Workload, seed: int = 0, device="cpu") -> dict:
    """All inputs of one step of workload ``wl`` (see the module docstring).

    Decode keys: q [B,H,D]; k_cmp, v_cmp [B,N_cap,D] (FP8-stored KV instead:
    kc_nope, kc_scale, kc_rope, vc8, vc_scale, see :func:`randn_kv8`); q_idx [B,1,H_I,d_I];
    w [B,1,H_I]; k_idx [B,N_cap,d_I] (+ q_scale, k_scale for FP8); sink [H];
    seq_len, n_cmp [B]; k_win, v_win [B,W,D] = raw rows L_b-W .. L_b-1.
    Streaming compression adds raw_new_idx [B,m,d_I] (raw indexer-key rows of
    the newest block, whose K/V rows are the last m window rows) and gate
    parameters gate_{k,v,idx} = (W, pos_bias); the newest compressed entry
    (index N-1) is left for the step to compute.
    Prefill keys: q [B,T,H,D]; q_idx [B,T,H_I,d_I]; w [B,T,H_I]; q_pos [B,T];
    k_cmp, v_cmp, k_idx with the L/m cached entries (the T/m new ones are left
    for the compression step, zero here); raw_{k,v} [B,W-1+T,D] for positions
    L-W+1 .. L+T-1; raw_idx [B,span-m+T,d_I] for positions idx_base = L-(span-m)
    .. L+T-1 (span = m without overlap); gates (pos_bias [span, d]).
    """
    B, H, D, W, m = wl.B, wl.H, wl.D, wl.W, wl.m
    dev = device
    qs = 1.0 / math.sqrt(D)
    out: dict = {"workload": wl}
    if wl.sink:
        out["sink"] = randn((H,), seed, 1, dev, dtype=torch.float32)
    else:
        out["sink"] = None
    N_cap = wl.N_cap

    def gate(d, tid):
        return (randn((d, d), seed, tid, dev, scale=1.0 / math.sqrt(d)),
                randn((wl.cspan, d), seed, tid + 1, dev, dtype=torch.float32))

    if wl.kind in ("csa_decode", "hca_decode"):
        lens = torch.tensor(wl.lens, dtype=torch.int32)
        out["seq_len"] = lens.to(dev)
        out["n_cmp"] = (lens // m).to(dev)
        out["q"] = randn((B, H, D), seed, 2, dev, scale=qs)
        if wl.kv_fp8:
            assert not wl.stream_compress, "FP8 KV workloads read a cache filled beforehand"
            out["k_cmp"] = out["v_cmp"] = None
            (out["kc_nope"], out["kc_scale"], out["kc_rope"], out["vc8"],
             out["vc_scale"]) = randn_kv8(B, N_cap, seed, 40, dev)
        else:
            out["k_cmp"] = randn((B, N_cap, D), seed, 3, dev)
            out["v_cmp"] = randn((B, N_cap, D), seed, 4, dev)
        out["k_win"] = randn((B, W, D), seed, 5, dev)
        out["v_win"] = randn((B, W, D), seed, 6, dev)
        if wl.kind == "csa_decode":
            out["w"] = randn((B, 1, wl.H_I), seed, 7, dev, dtype=torch.float32)
            if wl.idx_fp4:
                out["q_idx"], out["q_scale"] = rand_fp4_rows((B, 1, wl.H_I, wl.d_I), seed, 8,
                                                             dev)
                out["k_idx"], out["k_scale"] = rand_fp4_rows((B, N_cap, wl.d_I), seed, 9, dev)
            elif wl.idx_fp8:
                out["q_idx"], out["q_scale"] = randn_fp8_rows((B, 1, wl.H_I, wl.d_I), seed, 8,
                                                              dev)
                out["k_idx"], out["k_scale"] = randn_fp8_rows((B, N_cap, wl.d_I), seed, 9, dev)
            else:
                out["q_idx"] = randn((B, 1, wl.H_I, wl.d_I), seed, 8, dev)
                out["k_idx"] = randn((B, N_cap, wl.d_I), seed, 9, dev)
                out["q_scale"] = out["k_scale"] = None
        if wl.proj_groups:
            K = (H // wl.proj_groups) * D
            out["W_o"] = randn((wl.proj_groups, wl.proj_dim, K), seed, 30, dev,
                               scale=1.0 / math.sqrt(K))
        if wl.stream_compress:
            assert wl.cspan == m, "streaming compression: non-overlapping blocks"
            # the newest block's raw K/V rows are the last m window rows;
            # its raw indexer-key rows have no other source
            out["raw_new_idx"] = randn((B, m, wl.d_I), seed, 12, dev)
            out["gate_k"] = gate(D, 20)
            out["gate_v"] = gate(D, 22)
            out["gate_idx"] = gate(wl.d_I, 24)
        return out

    assert wl.kind == "csa_prefill"
    T, L = wl.T, wl.L
    n_old = L // m
    out["q_pos"] = (L + torch.arange(T, dtype=torch.int32)).repeat(B, 1).to(dev)
    out["n_cmp"] = torch.full((B,), N_cap, dtype=torch.int32, device=dev)
    out["q"] = randn((B, T, H, D), seed, 2, dev, scale=qs)
    k_cmp = torch.zeros((B, N_cap, D), dtype=torch.bfloat16, device=dev)
    v_cmp = torch.zeros((B, N_cap, D), dtype=torch.bfloat16, device=dev)
    k_idx = torch.zeros((B, N_cap, wl.d_I), dtype=torch.bfloat16, device=dev)
    k_cmp[:, :n_old] = randn((B, n_old, D), seed, 3, dev)
    v_cmp[:, :n_old] = randn((B, n_old, D), seed, 4, dev)
    k_idx[:, :n_old] = randn((B, n_old, wl.d_I), seed, 9, dev)
    out["k_cmp"], out["v_cmp"], out["k_idx"] = k_cmp, v_cmp, k_idx
    out["raw_k"] = randn((B, W - 1 + T, D), seed, 5, dev)
    out["raw_v"] = randn((B, W - 1 + T, D), seed, 6, dev)
    pre = wl.cspan - m  # indexer-key rows before the first new block that its span reads
    out["raw_idx"] = randn((B, pre + T, wl.d_I), seed, 12, dev)
    out["idx_base"] = L - pre
    out["raw_base"] = L - (W - 1)
    out["q_idx"] = randn((B, T, wl.H_I, wl.d_I), seed, 8, dev)
    out["w"] = randn((B, T, wl.H_I), seed, 7, dev, dtype=torch.float32)
    out["q_scale"] = out["k_scale"] = None
    out["gate_k"] = gate(D, 20)
    out["gate_v"] = gate(D, 22)
    out["gate_idx"] = gate(wl.d_I, 24)
    return out
