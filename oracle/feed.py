"""Numpy views of synthetic workload inputs for the oracle (test infrastructure).

Converts the tensors that ``synth.make_inputs`` returns into the arrays the
oracle functions take -- bf16 as uint16 bit patterns, E4M3 as uint8 codes --
for a sample of a workload's queries.  Only data movement happens here; the
method's arithmetic stays in ``oracle.c``.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (BF16, FP4_E2M1, FP8_E4M3, compress, kv8_dequantize, quantize_bf16,
               quantize_e4m3_rows, quantize_fp4_rows)


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.uint8).numpy()


def f32(t):
    return None if t is None else t.detach().contiguous().cpu().float().numpy()


def i32(t):
    return t.detach().contiguous().cpu().to(torch.int32).numpy()


def window_arrays(win: torch.Tensor, lens):
    """Raw rows of the decode window: rows len-W .. len-1 of each sequence are
    win[b]; returns (uint16 [B, R, D], base) covering positions base ..
    base+R-1 (rows outside a sequence's window are zero and never read)."""
    B, W, D = win.shape
    base = max(0, min(lens) - W)
    R = max(lens) - base
    arr = np.zeros((B, R, D), np.uint16)
    w = u16(win)
    for b, n in enumerate(lens):
        lo = max(0, n - W)
        arr[b, lo - base:n - base] = w[b, W - (n - lo):]
    return arr, base


def oracle_inputs(wl, inp: dict, n_units: int, seqs=None, tokens=None) -> dict:
    """Arrays for ``n_units`` queries of workload ``wl``: the first n sequences
    (decode; or the listed ``seqs``), or n evenly spread new tokens (prefill; or
    the listed ``tokens``)."""
    a: dict = {"sink": f32(inp.get("sink"))}
    if wl.kind in ("csa_decode", "hca_decode"):
        sel = list(seqs) if seqs is not None else list(range(min(n_units, wl.B)))
        ix = torch.tensor(sel, dtype=torch.long, device=inp["q"].device)
        lens = [wl.lens[b] for b in sel]
        a["seqs"] = sel
        a["seq_len"] = np.array(lens, np.int32)
        a["n_cmp"] = np.array([n // wl.m for n in lens], np.int32)
        a["q"] = u16(inp["q"][ix])
        if getattr(wl, "kv_fp8", False):
            # FP8-stored entries: the oracle attends over their decoded values
            kn, ks, kr, v8, vs = (inp[k][ix] for k in ("kc_nope", "kc_scale", "kc_rope", "vc8",
                                                       "vc_scale"))
            a["k_cmp"] = kv8_dequantize(u8(kn), f32(ks), u16(kr))
            a["v_cmp"] = kv8_dequantize(u8(v8), f32(vs))
        else:
            a["k_cmp"] = u16(inp["k_cmp"][ix])
            a["v_cmp"] = u16(inp["v_cmp"][ix])
        a["k_win"], a["raw_base"] = window_arrays(inp["k_win"][ix].cpu(), lens)
        a["v_win"], _ = window_arrays(inp["v_win"][ix].cpu(), lens)
        if wl.kind == "csa_decode":
            a["q_pos"] = (a["seq_len"] - 1).reshape(-1, 1).astype(np.int32)
            a["w"] = f32(inp["w"][ix])
            if wl.idx_fp4:
                a["q_idx"], a["k_idx"] = u8(inp["q_idx"][ix]), u8(inp["k_idx"][ix])
                a["q_scale"], a["k_scale"] = u8(inp["q_scale"][ix]), u8(inp["k_scale"][ix])
            elif wl.idx_fp8:
                a["q_idx"], a["k_idx"] = u8(inp["q_idx"][ix]), u8(inp["k_idx"][ix])
                a["q_scale"], a["k_scale"] = f32(inp["q_scale"][ix]), f32(inp["k_scale"][ix])
            else:
                a["q_idx"], a["k_idx"] = u16(inp["q_idx"][ix]), u16(inp["k_idx"][ix])
        if getattr(wl, "proj_groups", 0):
            a["W_o"] = u16(inp["W_o"])
        if wl.stream_compress:
            m = wl.m
            a["raw_new_k"] = u16(inp["k_win"][ix][:, wl.W - m:])
            a["raw_new_v"] = u16(inp["v_win"][ix][:, wl.W - m:])
            a["raw_new_idx"] = u16(inp["raw_new_idx"][ix])
            for s in ("k", "v", "idx"):
                Wg, pb = inp["gate_" + s]
                a["gate_" + s] = (u16(Wg), f32(pb))
        return a

    # prefill
    T = wl.T
    toks = list(tokens) if tokens is not None else sorted(
        set(np.linspace(0, T - 1, n_units).round().astype(int).tolist()))
    tx = torch.tensor(toks, dtype=torch.long, device=inp["q"].device)
    a["tokens"] = toks
    a["q"] = u16(inp["q"][:, tx])
    a["q_idx"] = u16(inp["q_idx"][:, tx])
    a["w"] = f32(inp["w"][:, tx])
    a["q_pos"] = i32(inp["q_pos"][:, tx])
    a["n_cmp"] = i32(inp["n_cmp"])
    a["k_cmp"], a["v_cmp"], a["k_idx"] = u16(inp["k_cmp"]), u16(inp["v_cmp"]), u16(inp["k_idx"])
    a["k_raw"], a["v_raw"] = u16(inp["raw_k"]), u16(inp["raw_v"])
    a["raw_base"] = int(inp["raw_base"])
    nb = max(1, len(toks) // wl.m)
    a["n_blocks"] = nb
    # rows of the new blocks, plus the span - m older rows the first one reads
    # (a whole number of blocks here: block_begin = pre / m)
    pre = wl.cspan - wl.m
    assert pre % wl.m == 0
    a["block0"] = pre // wl.m
    first = wl.W - 1  # raw_k row of the first new token
    a["raw_new_k"] = a["k_raw"][:, first - pre:first + nb * wl.m]
    a["raw_new_v"] = a["v_raw"][:, first - pre:first + nb * wl.m]
    a["raw_new_idx"] = u16(inp["raw_idx"][:, : pre + nb * wl.m])
    for s in ("k", "v", "idx"):
        Wg, pb = inp["gate_" + s]
        a["gate_" + s] = (u16(Wg), f32(pb))
    return a


def fill_new_entries(wl, inp: dict, a: dict) -> dict:
    """Write the oracle's own compressed entries where a step compresses:
    the newest block (streaming decode) or all T/m new blocks (prefill).
    Returns the oracle's outputs of that compression for comparison."""
    m = wl.m
    res = {}
    if wl.kind == "csa_decode" and wl.stream_compress:
        j = a["n_cmp"][0] - 1
        for s, dst in (("k", "k_cmp"), ("v", "v_cmp")):
            y = compress(a["raw_new_" + s], *a["gate_" + s], m, 0, 1)
            a[dst] = a[dst].copy()
            a[dst][:, j] = quantize_bf16(y)[:, 0]
            res[s] = y
        y = compress(a["raw_new_idx"], *a["gate_idx"], m, 0, 1)
        res["idx"] = y
        a["k_idx"] = a["k_idx"].copy()
        if wl.idx_fp4:
            codes, scales = quantize_fp4_rows(y)
            a["k_scale"] = a["k_scale"].copy()
            a["k_idx"][:, j], a["k_scale"][:, j] = codes[:, 0], scales[:, 0]
        elif wl.idx_fp8:
            codes, scales = quantize_e4m3_rows(y)
            a["k_scale"] = a["k_scale"].copy()
            a["k_idx"][:, j], a["k_scale"][:, j] = codes[:, 0], scales[:, 0]
        else:
            a["k_idx"][:, j] = quantize_bf16(y)[:, 0]
        return res
    if wl.kind == "csa_prefill":
        n_old, n_new = wl.L // m, wl.T // m
        first = wl.W - 1
        pre = wl.cspan - m  # older rows the first new block's span reads
        assert pre % m == 0
        raws = {"k": a["k_raw"][:, first - pre:first + wl.T],
                "v": a["v_raw"][:, first - pre:first + wl.T], "idx": u16(inp["raw_idx"])}
        for s, dst in (("k", "k_cmp"), ("v", "v_cmp"), ("idx", "k_idx")):
            y = compress(raws[s], *a["gate_" + s], m, pre // m, n_new)
            a[dst] = a[dst].copy()
            a[dst][:, n_old:n_old + n_new] = quantize_bf16(y)
            res[s] = y
    return res


def idx_dtype(wl):
    return FP4_E2M1 if wl.idx_fp4 else FP8_E4M3 if wl.idx_fp8 else BF16
