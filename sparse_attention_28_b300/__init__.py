"""CSA / HCA hybrid-attention hot path on one B300 GPU.

A thin ctypes binding over ``libcsa.so`` (C ABI in ``include/csa.h``).  Every
step of the path runs in the library's CUDA kernels; this module only checks
tensors, allocates outputs / workspaces with torch on the tensors' device, and
passes pointers plus the current CUDA stream.  There is no CPU fallback: if
the library is missing, every call raises.

Calls (same names as the C ABI, without the prefix where it reads better):

* :func:`compress_kv`            -- csa_compress_kv (csa_compress_kv_span for overlap)
* :func:`indexer_scores`         -- csa_indexer_scores
* :func:`indexer_topk`           -- csa_indexer_topk
* :func:`sparse_attn_decode`     -- csa_sparse_attn_decode
* :func:`sparse_attn_prefill`    -- csa_sparse_attn_prefill
* :func:`sparse_attn_batch_invariant` -- csa_sparse_attn_batch_invariant
* :func:`hca_dense_attn_decode`  -- hca_dense_attn_decode
* :func:`grouped_out_proj`       -- csa_grouped_out_proj
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")

CSA_BF16 = 0
CSA_FP8_E4M3 = 1
CSA_FP4_E2M1 = 2
EW_BAD_INDEX = 1
EW_BAD_POSITION = 2
EW_TIMEOUT = 4

# exported symbols of the C ABI (include/csa.h)
ABI_SYMBOLS = (
    "csa_status_str", "csa_abi_version", "csa_compress_kv", "csa_indexer_topk_workspace",
    "csa_indexer_topk", "csa_attn_workspace", "csa_sparse_attn_decode",
    "csa_sparse_attn_prefill", "hca_dense_attn_decode", "csa_indexer_topk_static",
    "csa_indexer_scores", "csa_compress_kv_span", "csa_sparse_attn_batch_invariant",
    "csa_grouped_out_proj", "csa_compress_kv_mixed", "csa_attn_fp8kv",
    "csa_selftest_bounded_wait", "csa_probe_stream_read", "csa_probe_row_gather",
)

# capacity of the library-owned scratch behind indexer_topk_static (bytes)
INDEXER_STATIC_SCRATCH_BYTES = 16 << 20

_lock = threading.Lock()
_lib = None


class CsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {lib().csa_status_str(status).decode()} (status {status})")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libcsa.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libcsa.so not found at {LIB_PATH}; build it with "
                    "`python -m sparse_attention_28_b300._build` (there is no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            P, I, I64, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
            L.csa_status_str.argtypes = [I]
            L.csa_status_str.restype = ctypes.c_char_p
            L.csa_abi_version.restype = I
            L.csa_compress_kv.argtypes = [P, I64, I64, I, I, I, I, I, P, P, P, I64, I, P, I64, P,
                                          P]
            L.csa_compress_kv.restype = I
            L.csa_compress_kv_span.argtypes = [P, I64, I64, I, I, I, I, I, I, P, P, P, I64, I, P,
                                               I64, P, P]
            L.csa_compress_kv_span.restype = I
            L.csa_indexer_topk_workspace.argtypes = [I, I, I, I]
            L.csa_indexer_topk_workspace.restype = SZ
            L.csa_indexer_topk.argtypes = [P, P, P, P, I64, P, I64, I, P, P, I, I, I, I, I, I, I,
                                           P, P, P, SZ, P, P]
            L.csa_indexer_topk.restype = I
            L.csa_indexer_topk_static.argtypes = [P, P, P, P, I64, P, I64, I, P, P, I, I, I, I,
                                                  I, I, I, P, P, P, P]
            L.csa_indexer_topk_static.restype = I
            L.csa_indexer_scores.argtypes = [P, P, P, P, I64, P, I64, I, P, P, I, I, I, I, I, I,
                                             P, I64, P, P]
            L.csa_indexer_scores.restype = I
            L.csa_attn_workspace.argtypes = [I, I, I, I]
            L.csa_attn_workspace.restype = SZ
            L.csa_sparse_attn_decode.argtypes = [P, P, P, I64, I, P, I, P, P, I64, I64, P, I, P,
                                                 F, I, I, I, P, P, P, SZ, P, P]
            L.csa_sparse_attn_decode.restype = I
            L.csa_sparse_attn_prefill.argtypes = [P, P, P, I64, I, P, I, P, P, I64, I64, P, I, P,
                                                  F, I, I, I, I, P, P, P, SZ, P, P]
            L.csa_sparse_attn_prefill.restype = I
            L.csa_sparse_attn_batch_invariant.argtypes = [P, P, P, I64, I, P, I, P, P, I64, I64,
                                                          P, I, P, F, I, I, I, I, P, P, I, P, P]
            L.csa_sparse_attn_batch_invariant.restype = I
            L.csa_grouped_out_proj.argtypes = [P, P, P, I, I, I, I, I, P, P]
            L.csa_grouped_out_proj.restype = I
            L.hca_dense_attn_decode.argtypes = [P, P, P, I64, I, P, I, P, P, I64, I64, P, I, P, F,
                                                I, I, I, P, P, P, SZ, P, P]
            L.hca_dense_attn_decode.restype = I
            L.csa_compress_kv_mixed.argtypes = [P, I64, I64, I, I, I, I, I, I, P, P, P, I64, P,
                                                I64, P, I64, I, P, P]
            L.csa_compress_kv_mixed.restype = I
            L.csa_attn_fp8kv.argtypes = [P, P, P, P, P, P, I, P, I, P, I, P, P, I64, I64, P, I,
                                         P, F, I, I, I, I, P, P, P, SZ, P, P]
            L.csa_attn_fp8kv.restype = I
            L.csa_selftest_bounded_wait.argtypes = [I, ctypes.c_uint32, P, P]
            L.csa_selftest_bounded_wait.restype = I
            L.csa_probe_stream_read.argtypes = [P, I64, I, I, P, P]
            L.csa_probe_stream_read.restype = I
            L.csa_probe_row_gather.argtypes = [P, I64, P, I, I, I, I, P, P]
            L.csa_probe_row_gather.restype = I
            _lib = L
    return _lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(status: int, what: str):
    if status != 0:
        raise CsaError(status, what)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _cuda(t, name, dtype=None):
    _need(t is not None and t.is_cuda, f"{name} must be a CUDA tensor")
    if dtype is not None:
        _need(t.dtype == dtype, f"{name} must be {dtype}, got {t.dtype}")
    return t


def _bstride(t) -> int:
    """Elements between sequences of a [B, rows, d] tensor with contiguous rows."""
    _need(t.dim() == 3 and t.stride(2) == 1 and t.stride(1) == t.shape[2],
          "tensor rows must be contiguous")
    return t.stride(0)


def _ws(nbytes: int, device, ws):
    """Workspace for a call: `ws` itself, a new buffer when it is None, or no
    workspace when it is False (attention only: splits then merge on chip)."""
    if nbytes == 0 or ws is False:
        return None, 0
    if ws is not None:
        _need(ws.numel() * ws.element_size() >= nbytes, "workspace too small")
        return ws, ws.numel() * ws.element_size()
    return torch.empty(nbytes, dtype=torch.uint8, device=device), nbytes


# ---------------------------------------------------------------- a1

def compress_kv(raw, W, pos_bias, m: int, block_begin: int, n_blocks: int, out,
                out_scale=None, err_word=None):
    """Compress blocks [block_begin, block_begin+n_blocks) of every sequence.

    raw: bf16 [B, R, d], a ring of R rows (position p at row p mod R; a
    full-length cache is R > every position); W: bf16 [d, d]; pos_bias: fp32
    [span, d] with span >= m: block j is compressed from the span raw tokens
    ending at its last token (span == m: non-overlapping blocks, span > m:
    overlapping compression); out: bf16 [B, N_cap, d] or uint8 [B, N_cap, d]
    (E4M3 codes, then out_scale fp32 [B, N_cap] is required) or uint8
    [B, N_cap, d/2] (FP4: two E2M1 codes per byte, then out_scale uint8
    [B, N_cap, d/16] receives the E4M3 block scales).  Writes in place;
    returns out.
    """
    _cuda(raw, "raw", torch.bfloat16)
    _cuda(W, "W", torch.bfloat16)
    _cuda(pos_bias, "pos_bias", torch.float32)
    _cuda(out, "out")
    B, _, d = raw.shape
    coded = out.dtype in (torch.uint8, torch.float8_e4m3fn)
    _need(coded or out.dtype == torch.bfloat16, "out must be bf16, E4M3 or FP4 bytes")
    fp4 = coded and out.shape[-1] * 2 == d  # two E2M1 codes per byte
    _need(W.is_contiguous() and pos_bias.is_contiguous(), "W, pos_bias must be contiguous")
    if fp4:
        _cuda(out_scale, "out_scale", torch.uint8)
        _need(out_scale.dim() == 3 and out_scale.shape[2] == d // 16 and out_scale.stride(2) == 1
              and out_scale.stride(1) == d // 16, "FP4 out_scale: uint8 [B, N_cap, d/16]")
        dtype, obs, sbs = CSA_FP4_E2M1, 2 * _bstride(out), out_scale.stride(0) // (d // 16)
    elif coded:
        _cuda(out_scale, "out_scale", torch.float32)
        _need(out_scale.dim() == 2 and out_scale.stride(1) == 1, "out_scale [B, N_cap]")
        dtype, obs, sbs = CSA_FP8_E4M3, _bstride(out), out_scale.stride(0)
    else:
        dtype, obs, sbs = CSA_BF16, _bstride(out), 0
    _need(pos_bias.dim() == 2 and pos_bias.shape[1] == d, "pos_bias [span, d]")
    span = pos_bias.shape[0]
    common = (_p(W), _p(pos_bias), _p(out), obs, dtype, _p(out_scale) if coded else None, sbs,
              _p(err_word), _stream(raw.device))
    if span == m:
        st = lib().csa_compress_kv(_p(raw), _bstride(raw), raw.shape[1], B, d, m, block_begin,
                                   n_blocks, *common)
        _check(st, "csa_compress_kv")
    else:
        st = lib().csa_compress_kv_span(_p(raw), _bstride(raw), raw.shape[1], B, d, m, span,
                                        block_begin, n_blocks, *common)
        _check(st, "csa_compress_kv_span")
    return out


def compress_kv_mixed(raw, W, pos_bias, m: int, block_begin: int, n_blocks: int, out_codes,
                      out_scale, out_rope, err_word=None):
    """Compress blocks into mixed-precision storage: the first d - n_rope
    channels as E4M3 codes (out_codes uint8 [B, N_cap, d - n_rope]) with a
    per-entry fp32 scale over them (out_scale [B, N_cap]), the last n_rope
    (RoPE) channels as bf16 (out_rope [B, N_cap, n_rope]).  Other arguments as
    :func:`compress_kv`.  Writes in place; returns (out_codes, out_scale,
    out_rope)."""
    _cuda(raw, "raw", torch.bfloat16)
    _cuda(W, "W", torch.bfloat16)
    _cuda(pos_bias, "pos_bias", torch.float32)
    _cuda(out_codes, "out_codes", torch.uint8)
    _cuda(out_scale, "out_scale", torch.float32)
    _cuda(out_rope, "out_rope", torch.bfloat16)
    B, _, d = raw.shape
    n_rope = out_rope.shape[-1]
    _need(out_codes.shape[-1] + n_rope == d, "codes and RoPE channels must add up to d")
    _need(W.is_contiguous() and pos_bias.is_contiguous(), "W, pos_bias must be contiguous")
    _need(out_scale.dim() == 2 and out_scale.stride(1) == 1, "out_scale [B, N_cap]")
    _need(pos_bias.dim() == 2 and pos_bias.shape[1] == d, "pos_bias [span, d]")
    st = lib().csa_compress_kv_mixed(
        _p(raw), _bstride(raw), raw.shape[1], B, d, m, pos_bias.shape[0], block_begin, n_blocks,
        _p(W), _p(pos_bias), _p(out_codes), _bstride(out_codes), _p(out_scale),
        out_scale.stride(0), _p(out_rope), _bstride(out_rope), n_rope, _p(err_word),
        _stream(raw.device))
    _check(st, "csa_compress_kv_mixed")
    return out_codes, out_scale, out_rope


# ---------------------------------------------------------------- a2 + a3

def _indexer_common(q_idx, w, k_idx, q_pos, n_cmp, m, q_scale, k_scale):
    """Checks and the shared leading C arguments of the indexer calls.

    bf16: q_idx [B, T, 4, 64], k_idx [B, N_cap, 64] bf16.  E4M3: the same as
    uint8 codes with q_scale fp32 [B, T, 4], k_scale fp32 [B, N_cap].  FP4:
    q_idx [B, T, 4, 32], k_idx [B, N_cap, 32] uint8 (two E2M1 codes per byte)
    with q_scale uint8 [B, T, 4, 4], k_scale uint8 [B, N_cap, 4] (E4M3 scale
    per 16 channels)."""
    _cuda(q_idx, "q_idx")
    _cuda(k_idx, "k_idx")
    _cuda(w, "w", torch.float32)
    _cuda(q_pos, "q_pos", torch.int32)
    _cuda(n_cmp, "n_cmp", torch.int32)
    coded = q_idx.dtype in (torch.uint8, torch.float8_e4m3fn)
    _need(coded == (k_idx.dtype in (torch.uint8, torch.float8_e4m3fn)), "q/k dtypes differ")
    if not coded:
        _need(q_idx.dtype == torch.bfloat16 and k_idx.dtype == torch.bfloat16, "bf16 expected")
    fp4 = coded and q_scale is not None and q_scale.dtype == torch.uint8
    _need(q_idx.is_contiguous() and w.is_contiguous() and q_pos.is_contiguous(),
          "q_idx, w, q_pos must be contiguous")
    B, T, H_I, d_I = q_idx.shape
    N_cap = k_idx.shape[1]
    if coded:
        _cuda(q_scale, "q_scale")
        _cuda(k_scale, "k_scale")
        _need(q_scale.is_contiguous(), "q_scale layout")
    if fp4:
        d_I *= 2
        _need(k_scale.dtype == torch.uint8 and k_scale.dim() == 3 and k_scale.shape[2] == d_I // 16
              and k_scale.stride(2) == 1 and k_scale.stride(1) == k_scale.shape[2],
              "FP4 k_scale: uint8 [B, N_cap, d_I/16]")
        dtype, kbs, ksbs = CSA_FP4_E2M1, 2 * _bstride(k_idx), k_scale.stride(0) // (d_I // 16)
    elif coded:
        _need(q_scale.dtype == torch.float32 and k_scale.dtype == torch.float32
              and k_scale.stride(1) == 1, "E4M3 scales: fp32")
        dtype, kbs, ksbs = CSA_FP8_E4M3, _bstride(k_idx), k_scale.stride(0)
    else:
        dtype, kbs, ksbs = CSA_BF16, _bstride(k_idx), 0
    args = (_p(q_idx), _p(q_scale) if coded else None, _p(w), _p(k_idx), kbs,
            _p(k_scale) if coded else None, ksbs, dtype, _p(q_pos), _p(n_cmp), B, T, H_I, d_I,
            N_cap, m)
    return args, (B, T, N_cap)


def indexer_scores(q_idx, w, k_idx, q_pos, n_cmp, m: int, q_scale=None, k_scale=None, out=None,
                   err_word=None):
    """Lightning-Indexer scores I(t, s) for every query token (no selection).

    Arguments as :func:`indexer_topk`.  Returns fp32 [B, T, N_cap]; column s of
    token t is defined for s < n_vis(t) only (the rest is unspecified).
    """
    args, (B, T, N_cap) = _indexer_common(q_idx, w, k_idx, q_pos, n_cmp, m, q_scale, k_scale)
    sc = out if out is not None else torch.empty((B, T, N_cap), dtype=torch.float32,
                                                 device=q_idx.device)
    _need(sc.dtype == torch.float32 and sc.shape[:2] == (B, T) and sc.shape[2] >= N_cap
          and sc.stride(2) == 1 and sc.stride(1) == sc.shape[2]
          and sc.stride(0) == T * sc.shape[2], "out: contiguous fp32 [B, T, >= N_cap]")
    st = lib().csa_indexer_scores(*args, _p(sc), sc.shape[2], _p(err_word),
                                  _stream(q_idx.device))
    _check(st, "csa_indexer_scores")
    return sc


def indexer_topk(q_idx, w, k_idx, q_pos, n_cmp, m: int, k: int, q_scale=None, k_scale=None,
                 return_scores: bool = False, out=None, ws=None, err_word=None):
    """Top-k compressed entries per query token by Lightning-Indexer score.

    q_idx: [B, T, 4, 64] bf16 (or uint8 E4M3 codes with q_scale fp32 [B, T, 4];
    or uint8 [B, T, 4, 32] FP4 codes with q_scale uint8 [B, T, 4, 4]);
    w: fp32 [B, T, 4]; k_idx: [B, N_cap, 64] bf16 (or uint8 with k_scale fp32
    [B, N_cap]; or uint8 [B, N_cap, 32] FP4 codes with k_scale uint8
    [B, N_cap, 4]); q_pos: int32 [B, T]; n_cmp: int32 [B].
    Returns int32 [B, T, k] (ascending, -1 padded) [, fp32 scores [B, T, k]].
    """
    args, (B, T, N_cap) = _indexer_common(q_idx, w, k_idx, q_pos, n_cmp, m, q_scale, k_scale)
    dev = q_idx.device
    idx = out if out is not None else torch.empty((B, T, k), dtype=torch.int32, device=dev)
    scores = torch.empty((B, T, k), dtype=torch.float32, device=dev) if return_scores else None
    nbytes = lib().csa_indexer_topk_workspace(B, T, N_cap, k)
    wsb, wsn = _ws(nbytes, dev, ws)
    st = lib().csa_indexer_topk(*args, k, _p(idx), _p(scores), _p(wsb), wsn, _p(err_word),
                                _stream(dev))
    _check(st, "csa_indexer_topk")
    return (idx, scores) if return_scores else idx


def indexer_topk_static(q_idx, w, k_idx, q_pos, n_cmp, m: int, k: int, q_scale=None,
                        k_scale=None, return_scores: bool = False, out=None, err_word=None,
                        scores_out=None):
    """indexer_topk with the library's fixed scratch instead of a caller
    workspace: the C call allocates no device memory (the output tensors here
    are still allocated by torch unless `out` and, with return_scores,
    `scores_out` are given).  Problems whose workspace would exceed
    INDEXER_STATIC_SCRATCH_BYTES are refused.  Calls that may run at the same
    time share the scratch and race."""
    args, (B, T, N_cap) = _indexer_common(q_idx, w, k_idx, q_pos, n_cmp, m, q_scale, k_scale)
    dev = q_idx.device
    idx = out if out is not None else torch.empty((B, T, k), dtype=torch.int32, device=dev)
    scores = None
    if return_scores:
        scores = scores_out if scores_out is not None else torch.empty(
            (B, T, k), dtype=torch.float32, device=dev)
    st = lib().csa_indexer_topk_static(*args, k, _p(idx), _p(scores), _p(err_word), _stream(dev))
    _check(st, "csa_indexer_topk_static")
    return (idx, scores) if return_scores else idx


def indexer_topk_workspace(B: int, T: int, N_cap: int, k: int) -> int:
    return int(lib().csa_indexer_topk_workspace(B, T, N_cap, k))


# ---------------------------------------------------------------- a4 / a5 / a6

def attn_workspace(B: int, T: int, H: int, n_keys_max: int) -> int:
    return int(lib().csa_attn_workspace(B, T, H, n_keys_max))


def _attn_common(q, k_cmp, v_cmp, k_raw, v_raw, sink):
    _cuda(q, "q", torch.bfloat16)
    _need(q.is_contiguous(), "q must be contiguous")
    _cuda(k_cmp, "k_cmp", torch.bfloat16)
    _cuda(v_cmp, "v_cmp", torch.bfloat16)
    _need(k_cmp.stride() == v_cmp.stride() and k_cmp.shape == v_cmp.shape,
          "k_cmp and v_cmp must share shape and strides")
    if k_raw is not None:
        _cuda(k_raw, "k_raw", torch.bfloat16)
        _cuda(v_raw, "v_raw", torch.bfloat16)
        _need(k_raw.stride() == v_raw.stride() and k_raw.shape == v_raw.shape,
              "k_raw and v_raw must share shape and strides")
    if sink is not None:
        _cuda(sink, "sink", torch.float32)


def sparse_attn_decode(q, k_cmp, v_cmp, topk_idx, k_raw, v_raw, seq_len, window: int, sink,
                       softmax_scale: float = 1.0, return_lse: bool = False, out=None, ws=None,
                       err_word=None):
    """CSA decode attention.  q: bf16 [B, H, 128]; k_cmp/v_cmp: bf16 [B, N_cap, 128];
    topk_idx: int32 [B, k]; k_raw/v_raw: bf16 [B, R, 128], a ring of R rows
    (position p at row p mod R, R >= window); seq_len: int32 [B];
    sink: fp32 [H] or None.  Returns bf16 [B, H, 128] [, lse fp32 [B, H]]."""
    _attn_common(q, k_cmp, v_cmp, k_raw, v_raw, sink)
    _cuda(topk_idx, "topk_idx", torch.int32)
    _cuda(seq_len, "seq_len", torch.int32)
    topk_idx = topk_idx.reshape(q.shape[0], -1)
    _need(topk_idx.is_contiguous(), "topk_idx must be contiguous")
    B, H, D = q.shape
    k = topk_idx.shape[1]
    dev = q.device
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev) if return_lse else None
    wsb, wsn = _ws(attn_workspace(B, 1, H, k + window), dev, ws)
    st = lib().csa_sparse_attn_decode(
        _p(q), _p(k_cmp), _p(v_cmp), _bstride(k_cmp), k_cmp.shape[1], _p(topk_idx), k,
        _p(k_raw), _p(v_raw), _bstride(k_raw) if k_raw is not None else 0,
        k_raw.shape[1] if k_raw is not None else 0, _p(seq_len), window, _p(sink),
        softmax_scale, B, H, D, _p(o), _p(lse), _p(wsb), wsn, _p(err_word), _stream(dev))
    _check(st, "csa_sparse_attn_decode")
    return (o, lse) if return_lse else o


def sparse_attn_prefill(q, k_cmp, v_cmp, topk_idx, k_raw, v_raw, q_pos, window: int, sink,
                        softmax_scale: float = 1.0, return_lse: bool = False, out=None, ws=None,
                        err_word=None):
    """CSA prefill attention.  q: bf16 [B, T, H, 128]; topk_idx: int32 [B, T, k];
    q_pos: int32 [B, T].  Returns bf16 [B, T, H, 128] [, lse fp32 [B, T, H]]."""
    _attn_common(q, k_cmp, v_cmp, k_raw, v_raw, sink)
    _cuda(topk_idx, "topk_idx", torch.int32)
    _cuda(q_pos, "q_pos", torch.int32)
    _need(topk_idx.is_contiguous() and q_pos.is_contiguous(), "contiguous index tensors")
    B, T, H, D = q.shape
    k = topk_idx.shape[-1]
    dev = q.device
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=dev) if return_lse else None
    wsb, wsn = _ws(attn_workspace(B, T, H, k + window), dev, ws)
    st = lib().csa_sparse_attn_prefill(
        _p(q), _p(k_cmp), _p(v_cmp), _bstride(k_cmp), k_cmp.shape[1], _p(topk_idx), k,
        _p(k_raw), _p(v_raw), _bstride(k_raw) if k_raw is not None else 0,
        k_raw.shape[1] if k_raw is not None else 0, _p(q_pos), window, _p(sink), softmax_scale,
        B, T, H, D, _p(o), _p(lse), _p(wsb), wsn, _p(err_word), _stream(dev))
    _check(st, "csa_sparse_attn_prefill")
    return (o, lse) if return_lse else o


def sparse_attn_batch_invariant(q, k_cmp, v_cmp, topk_idx, k_raw, v_raw, q_pos, window: int,
                                sink, keys_per_split: int = 256, softmax_scale: float = 1.0,
                                return_lse: bool = False, out=None, err_word=None):
    """CSA attention whose result for a query does not depend on the rest of
    the batch (bitwise): keys split in fixed ranges of keys_per_split slots.
    Shapes as :func:`sparse_attn_prefill` (T = 1: decode at q_pos = seq_len - 1;
    T = 2: a two-token step)."""
    _attn_common(q, k_cmp, v_cmp, k_raw, v_raw, sink)
    _cuda(topk_idx, "topk_idx", torch.int32)
    _cuda(q_pos, "q_pos", torch.int32)
    _need(topk_idx.is_contiguous() and q_pos.is_contiguous(), "contiguous index tensors")
    B, T, H, D = q.shape
    k = topk_idx.shape[-1]
    dev = q.device
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=dev) if return_lse else None
    st = lib().csa_sparse_attn_batch_invariant(
        _p(q), _p(k_cmp), _p(v_cmp), _bstride(k_cmp), k_cmp.shape[1], _p(topk_idx), k,
        _p(k_raw), _p(v_raw), _bstride(k_raw) if k_raw is not None else 0,
        k_raw.shape[1] if k_raw is not None else 0, _p(q_pos), window, _p(sink), softmax_scale,
        B, T, H, D, _p(o), _p(lse), keys_per_split, _p(err_word), _stream(dev))
    _check(st, "csa_sparse_attn_batch_invariant")
    return (o, lse) if return_lse else o


def hca_dense_attn_decode(q, k_cmp, v_cmp, n_cmp, m_prime: int, k_raw, v_raw, seq_len,
                          window: int, sink, softmax_scale: float = 1.0,
                          return_lse: bool = False, out=None, ws=None, err_word=None):
    """HCA decode attention over compressed entries 0 .. n_vis-1 plus the window."""
    _attn_common(q, k_cmp, v_cmp, k_raw, v_raw, sink)
    _cuda(n_cmp, "n_cmp", torch.int32)
    _cuda(seq_len, "seq_len", torch.int32)
    B, H, D = q.shape
    N_cap = k_cmp.shape[1]
    dev = q.device
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev) if return_lse else None
    wsb, wsn = _ws(attn_workspace(B, 1, H, N_cap + window), dev, ws)
    st = lib().hca_dense_attn_decode(
        _p(q), _p(k_cmp), _p(v_cmp), _bstride(k_cmp), N_cap, _p(n_cmp), m_prime, _p(k_raw),
        _p(v_raw), _bstride(k_raw) if k_raw is not None else 0,
        k_raw.shape[1] if k_raw is not None else 0, _p(seq_len), window, _p(sink),
        softmax_scale, B, H, D, _p(o), _p(lse), _p(wsb), wsn, _p(err_word), _stream(dev))
    _check(st, "hca_dense_attn_decode")
    return (o, lse) if return_lse else o


def attn_fp8kv(q, k_nope, k_scale, k_rope, v, v_scale, topk_idx, k_raw, v_raw, q_pos,
               window: int, sink, n_cmp=None, m_prime: int = 1, softmax_scale: float = 1.0,
               return_lse: bool = False, out=None, ws=None, err_word=None):
    """Attention over FP8-stored compressed entries (K: 64 E4M3 non-RoPE
    channels + k_scale, 64 bf16 RoPE channels; V: 128 E4M3 channels +
    v_scale).  q: bf16 [B, T, H, 128]; k_nope uint8 [B, N_cap, 64]; k_scale,
    v_scale fp32 [B, N_cap]; k_rope bf16 [B, N_cap, 64]; v uint8
    [B, N_cap, 128]; q_pos int32 [B, T].  topk_idx int32 [B, T, k] (CSA) or
    None (HCA: every visible entry, n_cmp int32 [B] and m_prime required).
    Returns bf16 [B, T, H, 128] [, lse fp32 [B, T, H]]."""
    _cuda(q, "q", torch.bfloat16)
    _need(q.is_contiguous() and q.dim() == 4, "q: contiguous [B, T, H, 128]")
    B, T, H, D = q.shape
    N_cap = k_nope.shape[1]
    for t, n, dt, w in ((k_nope, "k_nope", torch.uint8, 64), (k_rope, "k_rope", torch.bfloat16, 64),
                        (v, "v", torch.uint8, 128)):
        _cuda(t, n, dt)
        _need(t.is_contiguous() and tuple(t.shape) == (B, N_cap, w), f"{n}: [B, N_cap, {w}]")
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _cuda(t, n, torch.float32)
        _need(t.is_contiguous() and tuple(t.shape) == (B, N_cap), f"{n}: [B, N_cap]")
    if k_raw is not None:
        _cuda(k_raw, "k_raw", torch.bfloat16)
        _cuda(v_raw, "v_raw", torch.bfloat16)
        _need(k_raw.stride() == v_raw.stride() and k_raw.shape == v_raw.shape,
              "k_raw and v_raw must share shape and strides")
    if sink is not None:
        _cuda(sink, "sink", torch.float32)
    _cuda(q_pos, "q_pos", torch.int32)
    _need(q_pos.is_contiguous(), "q_pos must be contiguous")
    if topk_idx is not None:
        _cuda(topk_idx, "topk_idx", torch.int32)
        _need(topk_idx.is_contiguous(), "topk_idx must be contiguous")
        k = topk_idx.shape[-1]
        n_keys = k + window
    else:
        _cuda(n_cmp, "n_cmp", torch.int32)
        k = 0
        n_keys = N_cap + window
    dev = q.device
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=dev) if return_lse else None
    wsb, wsn = _ws(attn_workspace(B, T, H, n_keys), dev, ws)
    st = lib().csa_attn_fp8kv(
        _p(q), _p(k_nope), _p(k_scale), _p(k_rope), _p(v), _p(v_scale), N_cap, _p(topk_idx), k,
        _p(n_cmp), m_prime, _p(k_raw), _p(v_raw), _bstride(k_raw) if k_raw is not None else 0,
        k_raw.shape[1] if k_raw is not None else 0, _p(q_pos), window, _p(sink), softmax_scale,
        B, T, H, D, _p(o), _p(lse), _p(wsb), wsn, _p(err_word), _stream(dev))
    _check(st, "csa_attn_fp8kv")
    return (o, lse) if return_lse else o


# ---------------------------------------------------------------- output projection

def selftest_bounded_wait(err_word, arrive: bool = False, limit: int = 1000):
    """Run the library's bounded mbarrier wait on a barrier in a one-thread
    kernel: without `arrive` nobody completes it, so the wait gives up after
    `limit` polls and ORs CSA_EW_TIMEOUT into err_word (an int32 CUDA
    tensor); with `arrive` the wait succeeds and err_word is untouched."""
    _cuda(err_word, "err_word", torch.int32)
    st = lib().csa_selftest_bounded_wait(int(bool(arrive)), int(limit), _p(err_word),
                                         _stream(err_word.device))
    _check(st, "csa_selftest_bounded_wait")


def grouped_out_proj(o, W, out=None, err_word=None):
    """Grouped output projection: o bf16 [n, H, D] (the attention output), W
    bf16 [G, d_g, (H/G)*D] (group g's rows); returns bf16 [n, G*d_g] with
    y[q, g*d_g + r] = sum_j W[g, r, j] * o[q, heads of group g flattened][j]."""
    _cuda(o, "o", torch.bfloat16)
    _cuda(W, "W", torch.bfloat16)
    _need(o.is_contiguous() and W.is_contiguous(), "o, W must be contiguous")
    n, H, D = o.shape
    G, d_g, K = W.shape
    _need(K * G == H * D, "W must be [G, d_g, (H/G)*D]")
    y = out if out is not None else torch.empty((n, G * d_g), dtype=torch.bfloat16,
                                               device=o.device)
    _need(y.dtype == torch.bfloat16 and y.is_contiguous() and tuple(y.shape) == (n, G * d_g),
          "out: contiguous bf16 [n, G*d_g]")
    st = lib().csa_grouped_out_proj(_p(o), _p(W), _p(y), n, H, D, G, d_g, _p(err_word),
                                    _stream(o.device))
    _check(st, "csa_grouped_out_proj")
    return y



# ---------------------------------------------------------------- feed probes

def probe_stream_read(src, sink, ctas_per_sm: int = 2, in_flight: int = 4):
    """Stream-read every byte of the CUDA tensor src (16-byte loads, in_flight
    per thread before any is used, 148 * ctas_per_sm CTAs).  sink: a float32
    CUDA tensor of one element.  Asynchronous on the current stream."""
    _need(src.is_cuda and src.is_contiguous(), "src: contiguous CUDA tensor")
    _cuda(sink, "sink", torch.float32)
    st = lib().csa_probe_stream_read(_p(src), src.numel() * src.element_size(), int(ctas_per_sm),
                                     int(in_flight), _p(sink), _stream(src.device))
    _check(st, "csa_probe_stream_read")


def _gather_mode(tma: bool, wide: bool, issuers: int) -> int:
    if not tma:
        _need(issuers == 0, "issuers: TMA gathers only")
        return 2 if wide else 0
    n = issuers if issuers else (4 if wide else 1)
    _need(n in (1, 4, 8), "issuers: 1, 4 or 8")
    return {1: 1, 4: 3, 8: 4}[n]


def probe_row_gather(table, idx, n_ctas: int, stages: int, ring: int, sink, tma: bool = False,
                     wide: bool = False, issuers: int = 0):
    """Gather 512-byte rows of table (uint8 CUDA tensor [n_rows, 512]) into
    shared memory: CTA c reads idx[c * stages * 64: (c + 1) * stages * 64]
    (int32, 64 rows per stage) through a ring of `ring` 32 KB stages, with
    16-byte cp.async copies by 256 threads (512 when `wide`), or TMA
    tile::gather4 when `tma`, issued by `issuers` warps (1, 4 or 8; when 0:
    four if `wide`, else one)."""
    _need(table.is_cuda and table.is_contiguous() and table.dim() == 2 and table.shape[1] == 512,
          "table: contiguous CUDA [n_rows, 512]")
    _cuda(idx, "idx", torch.int32)
    _need(idx.is_contiguous() and idx.numel() >= n_ctas * stages * 64, "idx: n_ctas * stages * 64")
    _cuda(sink, "sink", torch.float32)
    st = lib().csa_probe_row_gather(_p(table), table.shape[0], _p(idx), int(n_ctas), int(stages),
                                    int(ring), _gather_mode(tma, wide, issuers), _p(sink),
                                    _stream(table.device))
    _check(st, "csa_probe_row_gather")
