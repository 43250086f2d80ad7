"""Shared test plumbing: tensor <-> numpy views, raw-cache placement, and the
parity criteria.  No step of the method is computed here."""
from __future__ import annotations

import numpy as np
import torch

# Parity bars for bf16 inputs with fp32 accumulation (attention outputs).
ATTN_MAX_ABS = 2e-2
ATTN_REL_L2 = 5e-3
LSE_ABS = 1e-3
NEAR_TIE_REL = 1e-6


# Compressed entries: one bf16 ulp of the exact value (rounding) plus the
# fp32 evaluation error of the gate logits and the weighted sum.  With
# |x| <~ 6, d = 128, and fp32 sums the absolute error stays below ~1e-6, which
# matters only where y is tiny (cancellation) and its ulp smaller than that.
COMPRESS_ABS = 2.0 ** -19


def bf16_bound(y):
    """Allowed |gpu - y| for a bf16 compressed entry with exact value y."""
    a = np.abs(np.asarray(y, np.float64))
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 7)
    return ulp + COMPRESS_ABS


# Quantised entries.  The GPU forms a compressed value y in fp32, the oracle
# in fp64; their difference stays below about 1e-6 of the entry's (or
# block's) largest magnitude, the agreement the fp32 scale amax/448 shows
# against the oracle's at rtol 1e-6.  A rounding decision may therefore
# differ only where the exact value lies that close to a rounding midpoint of
# the format; everywhere else the GPU's code must be the oracle's.
QUANT_REL = 1e-6


def _format_midpoints(decode, n_codes):
    v = decode(np.arange(n_codes, dtype=np.uint8))
    v = np.unique(np.abs(v[np.isfinite(v)]))
    return (v[1:] + v[:-1]) / 2


def _near(x, mids, window):
    """|x| within `window` (broadcast against x) of one of `mids`."""
    a = np.abs(np.asarray(x, np.float64))
    d = np.abs(a[..., None] - mids).min(axis=-1)
    return d <= window


def check_e4m3_rows(codes_gpu, scale_gpu, y, what=""):
    """FP8 storage of compressed entries (one fp32 scale per row, E4M3 codes):
    the scale equals the oracle's amax/448 within rtol 1e-6, and every code is
    the nearest E4M3 value of y / scale (the GPU's stored scale), except where
    that quotient lies within 1e-6 of the row's range (448) of an E4M3
    rounding midpoint."""
    import oracle
    y = np.asarray(y, np.float64)
    _, sc_ref = oracle.quantize_e4m3_rows(y)
    gs = np.asarray(scale_gpu, np.float64)
    np.testing.assert_allclose(gs, sc_ref, rtol=QUANT_REL, err_msg=f"{what}: scales")
    r = y / gs[..., None]
    want = oracle.e4m3_encode(r)
    mids = _format_midpoints(oracle.e4m3_decode, 256)
    tie = _near(r, mids, QUANT_REL * 448.0)
    bad = (np.asarray(codes_gpu) != want) & ~tie
    assert not bad.any(), f"{what}: {int(bad.sum())} E4M3 codes differ away from a midpoint"


def check_fp4_rows(codes_gpu, scales_gpu, y, what=""):
    """FP4 storage (E2M1 codes two per byte, one E4M3 scale per 16 channels):
    every scale byte equals the oracle's (nearest E4M3 of amax/6) unless
    amax/6 lies within 1e-6 relative of an E4M3 midpoint; every code is the
    nearest E2M1 value of y / scale on the GPU's scale (the oracle's, except at
    such a scale tie) unless the quotient lies within 1e-6 of the block's
    range (6) of an E2M1 midpoint.  Signs of zero count: -0 is its own code."""
    import oracle
    y = np.asarray(y, np.float64)
    codes_gpu = np.asarray(codes_gpu, np.uint8)
    scales_gpu = np.asarray(scales_gpu, np.uint8)
    d = y.shape[-1]
    _, ref_scales = oracle.quantize_fp4_rows(y)
    blk = y.reshape(y.shape[:-1] + (d // 16, 16))
    x = np.abs(blk).max(axis=-1) / 6.0
    scale_tie = _near(x, _format_midpoints(oracle.e4m3_decode, 256), QUANT_REL * x)
    bad_s = (scales_gpu != ref_scales) & ~scale_tie
    assert not bad_s.any(), f"{what}: {int(bad_s.sum())} E4M3 block scales differ"
    s = np.repeat(oracle.e4m3_decode(scales_gpu), 16, axis=-1)
    r = y / s
    want = oracle.e2m1_encode(r)
    got = np.empty(y.shape, np.uint8)
    got[..., 0::2] = codes_gpu & 0x0F
    got[..., 1::2] = codes_gpu >> 4
    tie = _near(r, _format_midpoints(oracle.e2m1_decode, 16), QUANT_REL * 6.0)
    bad = (got != want) & ~tie
    assert not bad.any(), f"{what}: {int(bad.sum())} E2M1 codes differ away from a midpoint"


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.uint8).numpy()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def poisoned(shape, dtype=torch.bfloat16, device="cuda"):
    """A tensor filled with NaN: any stray read shows up in the outputs."""
    return torch.full(shape, float("nan"), dtype=dtype, device=device)


def place_window(win: torch.Tensor, lens, L_cap: int, device="cuda") -> torch.Tensor:
    """Raw cache [B, L_cap, D], NaN everywhere except rows len-W .. len-1 of
    sequence b, which hold win[b] (rows before position 0 are dropped)."""
    B, W, D = win.shape
    raw = poisoned((B, L_cap, D), device=device)
    for b, n in enumerate(lens):
        lo = max(0, n - W)
        raw[b, lo:n] = win[b, W - (n - lo):].to(device)
    return raw


def window_arrays(win: torch.Tensor, lens):
    """The oracle's view of place_window: rows for positions base .. base+R-1
    of every sequence, with base = min over b of (len_b - W) clipped at 0.
    Returns (uint16 [B, R, D], base)."""
    B, W, D = win.shape
    base = max(0, min(lens) - W)
    R = max(lens) - base
    arr = np.zeros((B, R, D), np.uint16)
    w = u16(win)
    for b, n in enumerate(lens):
        lo = max(0, n - W)
        arr[b, lo - base:n - base] = w[b, W - (n - lo):]
    return arr, base


def check_attention(out_gpu, out_ref, lse_gpu=None, lse_ref=None, what="", lse_tol=None):
    """Attention parity: max-abs <= 2e-2, relative L2 <= 5e-3, lse within 1e-3
    (or lse_tol: a scalar or an array shaped like lse)."""
    o = f64(out_gpu).reshape(-1)
    r = np.asarray(out_ref, np.float64).reshape(-1)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output (stray read?)"
    max_abs = np.max(np.abs(o - r)) if o.size else 0.0
    rel_l2 = np.linalg.norm(o - r) / max(np.linalg.norm(r), 1e-30)
    assert max_abs <= ATTN_MAX_ABS, f"{what}: max-abs {max_abs:.3e}"
    assert rel_l2 <= ATTN_REL_L2, f"{what}: rel-L2 {rel_l2:.3e}"
    if lse_gpu is not None:
        lg = f64(lse_gpu).reshape(-1)
        lr = np.asarray(lse_ref, np.float64).reshape(-1)
        fin = np.isfinite(lr)
        np.testing.assert_array_equal(np.isfinite(lg), fin, err_msg=f"{what}: lse finiteness")
        if fin.any():
            tol = np.asarray(LSE_ABS if lse_tol is None else lse_tol, np.float64).reshape(-1)
            tol = (tol if tol.size == lr.size else np.full(lr.shape, tol.max()))[fin]
            d = np.abs(lg[fin] - lr[fin])
            assert np.all(d <= tol), f"{what}: lse max-abs {d.max():.3e} (worst excess " \
                f"{(d - tol).max():.3e})"
    return max_abs, rel_l2


def lse_tol(q, K, n_vis, scale=1.0):
    """lse tolerance for FP8-stored keys.  The kernel rounds each decoded key
    value to bf16 (relative error <= 2^-9) before the tensor cores use it, so
    a logit moves by at most 2^-9 * scale * sum_d |q_d| |k_d|, and the lse by
    at most the largest such move over the keys; on top of that the 1e-3 of
    the bf16 path.  q: bf16 [B, T, H, D] (torch) or fp64 values; K: decoded
    fp64 [B, N, D]; the max runs over each sequence's first n_vis[b] entries
    (a superset of its keys; the raw window rows are bf16 and exact).
    Returns [B, T, H]."""
    qa = np.abs(f64(q) if isinstance(q, torch.Tensor) else np.asarray(q, np.float64))
    B, T, H, _ = qa.shape
    tol = np.full((B, T, H), 1e-3)
    for b in range(B):
        if n_vis[b] > 0:
            m = np.einsum("thd,nd->thn", qa[b], np.abs(K[b, :n_vis[b]])).max(-1)
            tol[b] += 2.0 ** -9 * scale * m
    return tol


def check_topk(idx_gpu, idx_ref, scores_ref, n_vis, k: int, what=""):
    """Top-k parity: identical index sets except near-ties (an index in the
    symmetric difference must have an oracle score within 1e-6 relative of the
    oracle's k-th score); ascending order; -1 padding exactly where expected."""
    g = np.asarray(idx_gpu).reshape(-1, k)
    r = np.asarray(idx_ref).reshape(-1, k)
    s = np.asarray(scores_ref, np.float64).reshape(g.shape[0], -1)
    nv = np.asarray(n_vis).reshape(-1)
    mismatched = 0
    for qq in range(g.shape[0]):
        take = min(k, int(nv[qq]))
        gq, rq = g[qq], r[qq]
        assert np.all(gq[take:] == -1), f"{what}: query {qq} padding"
        gs = gq[:take]
        assert np.all(np.diff(gs) > 0), f"{what}: query {qq} not ascending"
        assert np.all((gs >= 0) & (gs < nv[qq])), f"{what}: query {qq} index range"
        diff = set(gs.tolist()) ^ set(rq[:take].tolist())
        if diff:
            kth = np.sort(s[qq, : nv[qq]])[::-1][take - 1]
            for i in diff:
                assert abs(s[qq, i] - kth) <= NEAR_TIE_REL * abs(kth), (
                    f"{what}: query {qq} index {i} score {s[qq, i]!r} vs k-th {kth!r}")
            mismatched += 1
    return mismatched
