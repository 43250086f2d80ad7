"""CPU oracle for the CSA / HCA hot path (test infrastructure only).

This package wraps ``oracle.c`` -- a plain fp64 C implementation of every step
of the path -- with numpy marshalling.  Only the tests, the smoke entry and the
benchmark's CPU-baseline leg may import it.  It does not import, link or call
anything from the CUDA library, and the CUDA library does not use it.

Arrays are numpy: bf16 data travels as ``uint16`` bit patterns, E4M3 data as
``uint8`` codes.  Steps (page: "DeepSeek-V4: Towards Highly Efficient
Million-Token Context Intelligence", hyper.ai, Method; aiboss88 news page,
Technical Principles):

* :func:`compress`         -- a1, softmax-gated block compression (fp64 out)
* :func:`quantize_bf16`, :func:`quantize_e4m3_rows` -- storage formats of a1
* :func:`indexer_scores`   -- a2, Lightning-Indexer scores
* :func:`topk`             -- a3, exact top-k with the lower-index tie rule
* :func:`attend`           -- a4 / a5, attention over the selected compressed
  entries plus the raw sliding window plus the sink logit
* :func:`kv8_dequantize`   -- decoded values of FP8-stored compressed K / V
  entries (E4M3 non-RoPE channels with a per-entry scale, bf16 RoPE channels)
* :func:`csa_decode`, :func:`hca_decode`, :func:`csa_prefill` -- the steps
  chained per call of the CUDA library's boundary.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
FP8_E4M3 = 1
FP4_E2M1 = 2


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc -O2, OpenMP, no fast-math)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-Wno-unused-parameter", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB)
    except subprocess.CalledProcessError as e:  # pragma: no cover - build failure is fatal
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed:\n{e.stderr}") from e
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.orc_num_threads.restype = I
            lib.orc_f64_to_bf16.argtypes = [D]
            lib.orc_f64_to_bf16.restype = ctypes.c_uint16
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f64.restype = D
            lib.orc_f64_to_e4m3.argtypes = [D]
            lib.orc_f64_to_e4m3.restype = ctypes.c_uint8
            lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_to_f64.restype = D
            lib.orc_f64_to_e2m1.argtypes = [D]
            lib.orc_f64_to_e2m1.restype = ctypes.c_uint8
            lib.orc_e2m1_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_e2m1_to_f64.restype = D
            for f in ("orc_bf16_decode_array", "orc_bf16_encode_array",
                      "orc_e4m3_decode_array", "orc_e4m3_encode_array",
                      "orc_e2m1_decode_array"):
                getattr(lib, f).argtypes = [P, P, L]
                getattr(lib, f).restype = None
            lib.orc_quantize_e4m3_rows.argtypes = [P, L, I, P, P]
            lib.orc_quantize_e4m3_rows.restype = None
            lib.orc_quantize_fp4_rows.argtypes = [P, L, I, P, P]
            lib.orc_quantize_fp4_rows.restype = None
            lib.orc_fp4_dequantize_rows.argtypes = [P, P, L, I, P]
            lib.orc_fp4_dequantize_rows.restype = None
            lib.orc_compress.argtypes = [P, L, I, I, I, I, I, P, P, P]
            lib.orc_compress.restype = I
            lib.orc_compress_span.argtypes = [P, L, I, I, I, I, I, I, P, P, P]
            lib.orc_compress_span.restype = I
            lib.orc_grouped_out_proj.argtypes = [P, P, L, I, I, I, I, P]
            lib.orc_grouped_out_proj.restype = I
            lib.orc_indexer_scores.argtypes = [P, P, P, P, L, P, L, I, P, P, I, I, I, I, I, L,
                                               P, P]
            lib.orc_indexer_scores.restype = I
            lib.orc_topk.argtypes = [P, L, P, L, I, P]
            lib.orc_topk.restype = I
            lib.orc_attend.argtypes = [P, P, P, L, I, I, P, P, L, L, P, L, I, P, P, L, L, L, I,
                                       P, D, P, P]
            lib.orc_attend.restype = I
            lib.orc_attend_f64cmp.argtypes = lib.orc_attend.argtypes
            lib.orc_attend_f64cmp.restype = I
            lib.orc_kv8_dequantize.argtypes = [P, P, P, L, I, I, P]
            lib.orc_kv8_dequantize.restype = I
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle uses (the CPU-baseline core count)."""
    return int(_load().orc_num_threads())


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def bf16_decode(bits) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    _load().orc_bf16_decode_array(_ptr(bits), _ptr(out), bits.size)
    return out


def bf16_encode(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().orc_bf16_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_decode(codes) -> np.ndarray:
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().orc_e4m3_decode_array(_ptr(codes), _ptr(out), codes.size)
    return out


def e4m3_encode(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint8)
    _load().orc_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e2m1_decode(codes) -> np.ndarray:
    """Values of FP4 E2M1 codes (one code per uint8, low 4 bits)."""
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().orc_e2m1_decode_array(_ptr(codes), _ptr(out), codes.size)
    return out


def e2m1_encode(x) -> np.ndarray:
    """Nearest E2M1 codes (ties to even, saturating at 6), one per uint8."""
    x = np.asarray(x, np.float64)
    f = _load().orc_f64_to_e2m1
    return np.array([f(float(v)) for v in x.ravel()], np.uint8).reshape(x.shape)


def quantize_fp4_rows(y):
    """FP4 storage of indexer vectors: per 16 channels one E4M3 scale (nearest
    to amax / 6), E2M1 codes of y / scale packed two per byte (channel 2i in
    the low nibble).  Returns (codes uint8 [..., d/2], scales uint8 [..., d/16])."""
    y = _c(y, np.float64)
    d = y.shape[-1]
    assert d % 16 == 0
    rows = y.size // d
    codes = np.zeros(y.shape[:-1] + (d // 2,), np.uint8)
    scales = np.empty(y.shape[:-1] + (d // 16,), np.uint8)
    _load().orc_quantize_fp4_rows(_ptr(y), rows, d, _ptr(codes), _ptr(scales))
    return codes, scales


def fp4_dequantize(codes, scales) -> np.ndarray:
    """Values of FP4-stored vectors (layout of quantize_fp4_rows)."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    d = codes.shape[-1] * 2
    rows = codes.size // (d // 2)
    out = np.empty(codes.shape[:-1] + (d,), np.float64)
    _load().orc_fp4_dequantize_rows(_ptr(codes), _ptr(scales), rows, d, _ptr(out))
    return out


def quantize_bf16(y) -> np.ndarray:
    """bf16 storage of a1's output: nearest bf16, ties to even."""
    return bf16_encode(y)


def quantize_e4m3_rows(y):
    """FP8 storage of a1's output: per-row scale amax/448 (fp32), E4M3 codes."""
    y = _c(y, np.float64)
    d = y.shape[-1]
    rows = y.size // d
    codes = np.empty(y.shape, np.uint8)
    scales = np.empty(y.shape[:-1], np.float32)
    _load().orc_quantize_e4m3_rows(_ptr(y), rows, d, _ptr(codes), _ptr(scales))
    return codes, scales


# --------------------------------------------------------------------------
# a1: compression
# --------------------------------------------------------------------------

def compress(raw, W, pos_bias, m: int, block_begin: int, n_blocks: int) -> np.ndarray:
    """a1 in fp64.  raw: uint16 [B, L, d]; W: uint16 [d, d]; pos_bias: f32 [span, d].

    Block j (stride m) is compressed from the span = pos_bias.shape[0] raw
    tokens ending at its last token, j*m + m - span .. j*m + m - 1 (the
    non-negative ones): span = m is the non-overlapping operator, span > m
    overlapping compression.  Returns fp64 [B, n_blocks, d] for blocks
    [block_begin, block_begin+n_blocks).
    """
    raw = _c(raw, np.uint16)
    W = _c(W, np.uint16)
    pos_bias = _c(pos_bias, np.float32)
    B, L, d = raw.shape
    span = pos_bias.shape[0]
    assert W.shape == (d, d) and pos_bias.shape == (span, d) and span >= m
    y = np.empty((B, n_blocks, d), np.float64)
    rc = _load().orc_compress_span(_ptr(raw), L * d, B, d, m, span, block_begin, n_blocks,
                                   _ptr(W), _ptr(pos_bias), _ptr(y))
    _check(rc, "compress")
    return y


# --------------------------------------------------------------------------
# a2 / a3: indexer and top-k
# --------------------------------------------------------------------------

def indexer_scores(q, w, k, q_pos, n_cmp, m: int, dtype: int = BF16, q_scale=None,
                   k_scale=None):
    """a2 in fp64.

    q: [B, T, H, dI] (uint16 bf16 bits, or uint8 E4M3 codes); w: f32 [B, T, H];
    k: [B, N, dI] same format as q; q_scale: f32 [B, T, H]; k_scale: f32 [B, N];
    FP4: q [B, T, H, dI/2] and k [B, N, dI/2] packed E2M1 codes, q_scale
    uint8 [B, T, H, dI/16] and k_scale uint8 [B, N, dI/16] E4M3 block scales.
    q_pos: int32 [B, T] absolute positions; n_cmp: int32 [B] entries present.
    Returns (scores fp64 [B, T, N] with -inf beyond n_vis, n_vis int32 [B, T]).
    """
    code = np.uint16 if dtype == BF16 else np.uint8
    q = _c(q, code)
    k = _c(k, code)
    w = _c(w, np.float32)
    q_pos = _c(q_pos, np.int32)
    n_cmp = _c(n_cmp, np.int32)
    sc_t = np.uint8 if dtype == FP4_E2M1 else np.float32
    q_scale = _c(q_scale, sc_t)
    k_scale = _c(k_scale, sc_t)
    B, T, H, dI = q.shape
    if dtype == FP4_E2M1:
        dI *= 2
    N = k.shape[1]
    scores = np.empty((B, T, N), np.float64)
    n_vis = np.empty((B, T), np.int32)
    rc = _load().orc_indexer_scores(_ptr(q), _ptr(q_scale), _ptr(w), _ptr(k), N * dI,
                                    _ptr(k_scale), N, dtype, _ptr(q_pos), _ptr(n_cmp), B, T,
                                    H, dI, m, N, _ptr(scores), _ptr(n_vis))
    _check(rc, "indexer_scores")
    return scores, n_vis


def topk(scores, n_vis, k: int) -> np.ndarray:
    """a3: indices of the min(k, n_vis) best scores, ascending, -1 padded."""
    scores = _c(scores, np.float64)
    n_vis = _c(n_vis, np.int32)
    N = scores.shape[-1]
    Q = scores.size // N if N else int(np.prod(scores.shape[:-1]))
    assert n_vis.size == Q
    out = np.empty(scores.shape[:-1] + (k,), np.int32)
    rc = _load().orc_topk(_ptr(scores), N, _ptr(n_vis), Q, k, _ptr(out))
    _check(rc, "topk")
    return out


# --------------------------------------------------------------------------
# a4 / a5: attention
# --------------------------------------------------------------------------

def kv8_dequantize(codes, scale, rope=None) -> np.ndarray:
    """Decoded fp64 values of FP8-stored compressed entries.

    codes: uint8 E4M3 [..., d - n_rope] (the non-RoPE channels); scale: f32
    [...] (one per entry); rope: uint16 bf16 bits [..., n_rope] or None (V
    entries have no RoPE channels).  Returns fp64 [..., d]: code * scale, then
    the RoPE channels' bf16 values.
    """
    codes = _c(codes, np.uint8)
    scale = _c(scale, np.float32)
    dn = codes.shape[-1]
    n_rope = 0 if rope is None else np.asarray(rope).shape[-1]
    rope = _c(rope, np.uint16)
    rows = codes.size // dn
    assert scale.size == rows and (rope is None or rope.size == rows * n_rope)
    out = np.empty(codes.shape[:-1] + (dn + n_rope,), np.float64)
    rc = _load().orc_kv8_dequantize(_ptr(codes), _ptr(scale), _ptr(rope), rows, dn + n_rope,
                                    n_rope, _ptr(out))
    _check(rc, "kv8_dequantize")
    return out


def attend(q, qb, qt, k_cmp, v_cmp, sel, k_raw, v_raw, window: int, sink, scale: float,
           raw_base: int = 0):
    """a4 / a5 in fp64.

    q: uint16 [Q, H, D]; qb, qt: int32 [Q] (sequence, absolute position);
    k_cmp, v_cmp: uint16 bf16 bits [B, N, D], or fp64 [B, N, D] decoded values
    of FP8-stored entries (:func:`kv8_dequantize`); sel: int32 [Q, n_sel]
    compressed rows (-1 = none) or None; k_raw, v_raw: uint16 [B, R, D]
    holding absolute positions raw_base .. raw_base+R-1 (or None when
    window == 0); sink: f32 [H] or None.
    Returns (out fp64 [Q, H, D], lse fp64 [Q, H]).
    """
    q = _c(q, np.uint16)
    Q, H, D = q.shape
    qb = _c(qb, np.int32)
    qt = _c(qt, np.int32)
    f64 = k_cmp is not None and np.asarray(k_cmp).dtype == np.float64
    if sel is None or k_cmp is None:
        sel_a, n_sel, kc, vc, cmp_bstride, n_rows = None, 0, None, None, 0, 0
    else:
        sel_a = _c(sel, np.int32)
        n_sel = sel_a.shape[-1]
        ct = np.float64 if f64 else np.uint16
        kc, vc = _c(k_cmp, ct), _c(v_cmp, ct)
        cmp_bstride, n_rows = kc.shape[1] * D, kc.shape[1]
    if window > 0:
        kr, vr = _c(k_raw, np.uint16), _c(v_raw, np.uint16)
        raw_bstride, raw_rows = kr.shape[1] * D, kr.shape[1]
    else:
        kr = vr = None
        raw_bstride = raw_rows = 0
    sink = _c(sink, np.float32)
    out = np.empty((Q, H, D), np.float64)
    lse = np.empty((Q, H), np.float64)
    fn = _load().orc_attend_f64cmp if f64 else _load().orc_attend
    rc = fn(_ptr(q), _ptr(qb), _ptr(qt), Q, H, D, _ptr(kc), _ptr(vc),
                            cmp_bstride, n_rows, _ptr(sel_a), n_sel, n_sel, _ptr(kr), _ptr(vr),
                            raw_bstride, raw_base, raw_rows, window, _ptr(sink), scale,
                            _ptr(out), _ptr(lse))
    _check(rc, "attend")
    return out, lse


def hca_select(n_cmp, q_pos, m_prime: int) -> np.ndarray:
    """a5's key set: every visible compressed entry 0 .. n_vis-1 (-1 padded)."""
    n_cmp = np.asarray(n_cmp, np.int64)
    q_pos = np.asarray(q_pos, np.int64)
    n_vis = np.minimum(n_cmp[:, None], (q_pos + 1) // m_prime)
    width = int(n_vis.max()) if n_vis.size else 0
    sel = np.full(q_pos.shape + (width,), -1, np.int32)
    for idx in np.ndindex(*q_pos.shape):
        sel[idx][: n_vis[idx]] = np.arange(n_vis[idx], dtype=np.int32)
    return sel


# --------------------------------------------------------------------------
# chained steps, one per call of the CUDA library's boundary
# --------------------------------------------------------------------------

def csa_decode(q, k_cmp, v_cmp, topk_idx, k_raw, v_raw, seq_len, window, sink, scale,
               raw_base: int = 0):
    """CSA sparse attention for one decode token per sequence (t = seq_len-1)."""
    B = q.shape[0]
    qb = np.arange(B, dtype=np.int32)
    qt = np.asarray(seq_len, np.int32) - 1
    return attend(q, qb, qt, k_cmp, v_cmp, topk_idx, k_raw, v_raw, window, sink, scale,
                  raw_base)


def hca_decode(q, k_cmp, v_cmp, n_cmp, m_prime, k_raw, v_raw, seq_len, window, sink, scale,
               raw_base: int = 0):
    """HCA dense attention for one decode token per sequence."""
    B = q.shape[0]
    qb = np.arange(B, dtype=np.int32)
    qt = np.asarray(seq_len, np.int32) - 1
    sel = hca_select(n_cmp, qt[:, None], m_prime)[:, 0, :]
    return attend(q, qb, qt, k_cmp, v_cmp, sel, k_raw, v_raw, window, sink, scale, raw_base)


def csa_prefill(q, k_cmp, v_cmp, topk_idx, k_raw, v_raw, q_pos, window, sink, scale,
                raw_base: int = 0):
    """CSA sparse attention for T query tokens per sequence: q [B, T, H, D]."""
    B, T, H, D = q.shape
    qb = np.repeat(np.arange(B, dtype=np.int32), T)
    qt = np.asarray(q_pos, np.int32).reshape(-1)
    out, lse = attend(q.reshape(B * T, H, D), qb, qt, k_cmp, v_cmp,
                      np.asarray(topk_idx).reshape(B * T, -1), k_raw, v_raw, window, sink,
                      scale, raw_base)
    return out.reshape(B, T, H, D), lse.reshape(B, T, H)


# --------------------------------------------------------------------------
# grouped output projection
# --------------------------------------------------------------------------

def grouped_out_proj(o, W) -> np.ndarray:
    """y[q][g*d_g + r] = sum_j W[g][r][j] * o[q][g*K + j] in fp64, K = (H/G)*D.

    o: uint16 bf16 bits [n, H, D] (or [n, H*D]); W: uint16 [G, d_g, K].
    Returns fp64 [n, G*d_g].
    """
    o = _c(o, np.uint16)
    W = _c(W, np.uint16)
    G, d_g, K = W.shape
    n = o.shape[0]
    HD = o.size // n
    assert HD == G * K
    D = o.shape[-1] if o.ndim == 3 else K
    H = HD // D
    y = np.empty((n, G * d_g), np.float64)
    rc = _load().orc_grouped_out_proj(_ptr(o), _ptr(W), n, H, D, G, d_g, _ptr(y))
    _check(rc, "grouped_out_proj")
    return y

