"""Pins for the CPU oracle: each test checks it against something that is not
the oracle itself -- hand-derived worked examples (tests/golden), closed forms,
library routines on special cases (torch casts, numpy lexsort, torch SDPA in
fp64), invariants, and exhaustive checks on tiny inputs.  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _golden(name):
    e = math.e
    consts = {"ln3": math.log(3), "ln4": math.log(4), "ln5": math.log(5),
              "2/(e+1)": 2 / (e + 1), "(e+9e^3)/(e+3e^3)": (e + 9 * e**3) / (e + 3 * e**3)}
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = (s.strip() for s in line.split("=", 1))
        rows = [[consts[t] if t in consts else float(t) for t in r.split()]
                for r in val.split(";")]
        arr = np.array(rows if len(rows) > 1 else rows[0], np.float64)
        out[key] = arr.reshape(()) if arr.size == 1 else arr
    return out


def bf16_bits(x):
    """bf16 bit patterns of a float array (torch's RNE cast, via float32)."""
    t = torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16)).view(
        torch.bfloat16).double().numpy()


# ---------------------------------------------------------------- codecs

def test_bf16_decode_all_codes_match_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_decode(codes)
    ref = bits_to_f64(codes)
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])


def test_bf16_encode_matches_torch_on_float32_values():
    # float32-representable inputs: torch's float->bf16 cast rounds once
    x = np.concatenate([
        RNG.standard_normal(20000) * 10.0 ** RNG.integers(-40, 38, 20000),
        RNG.standard_normal(2000) * 1e-39,  # subnormal range
        [0.0, -0.0, 3.3895313892515355e38, -3.3895313892515355e38, 1e-45],
    ]).astype(np.float32)
    # exact ties: float32 bit patterns whose low 16 bits are 0x8000
    u = RNG.integers(0, 2 ** 31, 5000, dtype=np.uint32) & np.uint32(0x7F7F0000) | np.uint32(0x8000)
    ties = u.view(np.float32)
    x = np.concatenate([x, ties, -ties])
    x = x[np.isfinite(x)]
    np.testing.assert_array_equal(oracle.bf16_encode(x.astype(np.float64)), bf16_bits(x))


def test_bf16_encode_rounds_once_from_double():
    # 1 + 2^-8 + 2^-40 lies just above the midpoint of 1 and 1 + 2^-7:
    # direct rounding gives 1 + 2^-7 (0x3F81); rounding through float32 first
    # would land on the midpoint and tie to 1.0 (0x3F80).
    assert oracle.bf16_encode(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    assert oracle.bf16_encode(np.array([1 + 2.0 ** -8]))[0] == 0x3F80  # tie -> even
    assert oracle.bf16_encode(np.array([1 + 3 * 2.0 ** -8]))[0] == 0x3F82  # tie -> even
    assert oracle.bf16_encode(np.array([3.5e38]))[0] == 0x7F80  # overflow -> inf
    assert oracle.bf16_encode(np.array([-np.inf]))[0] == 0xFF80


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_in_range_and_ties():
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # 0 .. 448
    mids = (vals[:-1] + vals[1:]) / 2  # exact ties between neighbours
    x = np.concatenate([RNG.uniform(-448, 448, 20000), RNG.standard_normal(5000) * 1e-2,
                        vals, -vals, mids, -mids]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(x.astype(np.float64)), ref)


def test_e4m3_saturates():
    got = oracle.e4m3_encode(np.array([448.0, 449.0, 464.0, 1e9, -1e9, -500.0]))
    np.testing.assert_array_equal(got, [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE])


# ---------------------------------------------------------------- a1 compression

def _rand_bf16(shape, scale=1.0):
    return bf16_bits(RNG.standard_normal(shape) * scale)


def test_compress_hand_example():
    g = _golden("compress_hand.txt")
    raw = bf16_bits(g["x"])[None]  # [1, 2, 2]
    y = oracle.compress(raw, bf16_bits(g["W"]), g["pos_bias"].astype(np.float32), m=2,
                        block_begin=0, n_blocks=1)
    # pos_bias ln3 is rounded to fp32 on input: tolerance covers that
    np.testing.assert_allclose(y[0, 0], g["y"], rtol=1e-7)


def test_compress_zero_gate_is_block_mean():
    B, L, d, m = 2, 32, 16, 4
    raw = _rand_bf16((B, L, d))
    y = oracle.compress(raw, np.zeros((d, d), np.uint16), np.zeros((m, d), np.float32), m, 1, 6)
    x = bits_to_f64(raw)
    ref = x[:, 4:28].reshape(B, 6, m, d).mean(axis=2)
    np.testing.assert_allclose(y, ref, rtol=1e-14, atol=1e-15)


def test_compress_overlap_hand_example():
    g = _golden("compress_overlap_hand.txt")
    raw = bf16_bits(g["x"]).reshape(1, 2, 1)
    bias = g["pos_bias"].astype(np.float32).reshape(2, 1)
    for key, w in (("y_W0", 0.0), ("y_W1", 1.0)):
        y = oracle.compress(raw, bf16_bits(np.array([[w]])), bias, m=1, block_begin=0,
                            n_blocks=2)
        np.testing.assert_allclose(y[0, :, 0], g[key], rtol=1e-7)


def test_compress_overlap_zero_gate_is_span_mean_clipped_at_zero():
    # m = 4, span = 10: block j averages positions max(0, 4j-6) .. 4j+3
    B, L, d, m, span = 2, 32, 8, 4, 10
    raw = _rand_bf16((B, L, d))
    y = oracle.compress(raw, np.zeros((d, d), np.uint16), np.zeros((span, d), np.float32), m,
                        0, 8)
    x = bits_to_f64(raw)
    for j in range(8):
        lo, hi = max(0, 4 * j - 6), 4 * j + 4
        np.testing.assert_allclose(y[:, j], x[:, lo:hi].mean(axis=1), rtol=1e-14, atol=1e-15)


def test_compress_overlap_one_hot_bias_reaches_into_the_previous_block():
    # bias row i belongs to position j*m + m - span + i: rows below span - m
    # pick tokens of the previous block
    B, d, m, span = 2, 8, 4, 8
    raw = _rand_bf16((B, 4 * m, d))
    pick = RNG.integers(0, span, d)
    bias = np.zeros((span, d), np.float32)
    bias[pick, np.arange(d)] = 1e4
    y = oracle.compress(raw, _rand_bf16((d, d), 0.3), bias, m, 1, 3)
    x = bits_to_f64(raw)
    for jj, j in enumerate(range(1, 4)):
        pos = j * m + m - span + pick
        np.testing.assert_array_equal(y[:, jj], x[:, pos, np.arange(d)])


def test_compress_overlap_is_convex_over_its_span():
    B, d, m, span = 3, 16, 4, 12
    raw = _rand_bf16((B, 40, d), 2.0)
    bias = RNG.standard_normal((span, d)).astype(np.float32) * 3
    y = oracle.compress(raw, _rand_bf16((d, d), 0.5), bias, m, 0, 10)
    x = bits_to_f64(raw)
    for j in range(10):
        win = x[:, max(0, j * m + m - span):j * m + m]
        assert np.all(y[:, j] >= win.min(axis=1) - 1e-12)
        assert np.all(y[:, j] <= win.max(axis=1) + 1e-12)


# ---------------------------------------------------------------- FP4 (E2M1)

def test_e2m1_values_are_the_format_definition():
    g = _golden("indexer_fp4_hand.txt")
    mags = g["e2m1_magnitudes"]
    vals = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    np.testing.assert_array_equal(vals[:8], mags)
    np.testing.assert_array_equal(vals[8:], -mags)
    assert np.signbit(vals[8])  # code 8 is -0


def test_e2m1_encode_nearest_ties_to_even_saturating():
    # midpoints go to the code with mantissa bit 0; beyond 6 saturates
    x = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 100.0, 0.26, 4.99, -0.75, -5.0]
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, 0.5, 4.0, -1.0, -4.0]
    np.testing.assert_array_equal(oracle.e2m1_decode(oracle.e2m1_encode(x)), want)
    codes = np.arange(16, dtype=np.uint8)
    np.testing.assert_array_equal(oracle.e2m1_encode(oracle.e2m1_decode(codes)), codes)


def test_fp4_block_quantization_scale_rule_and_error_bound():
    y = RNG.standard_normal((7, 64)) * np.exp(RNG.uniform(-6, 6, (7, 1)))
    y[3, 16:32] = 0.0  # an all-zero block: scale 1, codes 0
    codes, scales = oracle.quantize_fp4_rows(y)
    sc = oracle.e4m3_decode(scales)
    amax = np.abs(y.reshape(7, 4, 16)).max(axis=2)
    want = np.where(amax > 0, oracle.e4m3_decode(oracle.e4m3_encode(amax / 6)), 1.0)
    np.testing.assert_array_equal(sc, want)
    assert sc[3, 1] == 1.0 and not codes[3, 8:16].any()
    d = oracle.fp4_dequantize(codes, scales)
    r = np.abs(y) / np.repeat(sc, 16, axis=1)  # magnitude in units of the scale
    half = np.where(r < 2, 0.25, np.where(r < 4, 0.5, 1.0)) * np.repeat(sc, 16, axis=1)
    over = np.maximum(np.abs(y) - 6 * np.repeat(sc, 16, axis=1), 0)
    assert np.all(np.abs(d - y) <= np.maximum(half, over) * (1 + 1e-12))


def test_fp4_exact_values_round_trip():
    # values = E2M1 value x a power-of-two scale whose block amax is 6 x scale
    # are stored exactly
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    v = RNG.choice(np.concatenate([mags, -mags]), (5, 64))
    v[:, ::16] = 6.0
    y = v * np.repeat(2.0 ** RNG.integers(-5, 6, (5, 4)), 16, axis=1)
    codes, scales = oracle.quantize_fp4_rows(y)
    np.testing.assert_array_equal(oracle.fp4_dequantize(codes, scales), y)


def _fp4_pack(vals_codes):
    c = np.asarray(vals_codes, np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def test_indexer_scores_fp4_hand_example():
    g = _golden("indexer_fp4_hand.txt")
    qc = np.zeros((1, 1, 4, 64), np.uint8)
    qc[0, 0, 0, 0], qc[0, 0, 0, 17] = 0x2, 0xB
    qs = np.full((1, 1, 4, 4), 0x38, np.uint8)  # E4M3 1.0
    qs[0, 0, 0, 0], qs[0, 0, 0, 1] = 0x40, 0x30  # 2.0, 0.5
    kc = np.zeros((1, 1, 64), np.uint8)
    kc[0, 0, 0], kc[0, 0, 17] = 0x3, 0x6
    ks = np.full((1, 1, 4), 0x38, np.uint8)
    ks[0, 0, 0] = 0x40
    w = np.array([[[0.5, 1, 1, 1]]], np.float32)
    sc, nv = oracle.indexer_scores(_fp4_pack(qc), w, _fp4_pack(kc), np.array([[7]], np.int32),
                                   np.array([1], np.int32), 4, oracle.FP4_E2M1, qs, ks)
    assert nv[0, 0] == 1 and sc[0, 0, 0] == g["I"]


def test_indexer_scores_fp4_is_the_dot_of_the_stored_values():
    B, T, N, m = 2, 3, 50, 4
    qc, qs = oracle.quantize_fp4_rows(RNG.standard_normal((B, T, 4, 64)))
    kc, ks = oracle.quantize_fp4_rows(RNG.standard_normal((B, N, 64)) * 3)
    w = RNG.standard_normal((B, T, 4)).astype(np.float32)
    qp = np.full((B, T), 4 * N - 1, np.int32)
    sc, nv = oracle.indexer_scores(qc, w, kc, qp, np.array([N, N - 7], np.int32), m,
                                   oracle.FP4_E2M1, qs, ks)
    qv, kv = oracle.fp4_dequantize(qc, qs), oracle.fp4_dequantize(kc, ks)
    dots = np.einsum("bthd,bnd->bthn", qv, kv)
    want = np.einsum("bth,bthn->btn", w.astype(np.float64), np.maximum(dots, 0))
    for b in range(B):
        np.testing.assert_allclose(sc[b, :, :nv[b, 0]], want[b, :, :nv[b, 0]], rtol=1e-13,
                                   atol=1e-12)
    assert nv[1, 0] == N - 7 and np.all(np.isneginf(sc[1, :, N - 7:]))


def test_compress_m1_is_identity():
    raw = _rand_bf16((2, 9, 8))
    W = _rand_bf16((8, 8))
    y = oracle.compress(raw, W, RNG.standard_normal((1, 8)).astype(np.float32), 1, 0, 9)
    np.testing.assert_array_equal(y, bits_to_f64(raw))


def test_compress_one_hot_bias_picks_token_per_channel():
    B, d, m = 2, 8, 4
    raw = _rand_bf16((B, 2 * m, d))
    pick = RNG.integers(0, m, d)
    bias = np.zeros((m, d), np.float32)
    bias[pick, np.arange(d)] = 1e4
    y = oracle.compress(raw, _rand_bf16((d, d), 0.3), bias, m, 0, 2)
    x = bits_to_f64(raw).reshape(B, 2, m, d)
    np.testing.assert_array_equal(y, x[:, :, pick, np.arange(d)])


def test_compress_weight_orientation_row_is_output_channel():
    # only W[c0][e0] is non-zero and large: channel c0 follows token argmax_i x[i][e0];
    # every other channel keeps uniform weights (block mean)
    d, m, c0, e0 = 8, 4, 5, 2
    raw = _rand_bf16((1, m, d))
    W = np.zeros((d, d), np.float64)
    W[c0, e0] = 2.0 ** 20
    y = oracle.compress(raw, bf16_bits(W), np.zeros((m, d), np.float32), m, 0, 1)[0, 0]
    x = bits_to_f64(raw)[0]
    np.testing.assert_allclose(y[c0], x[np.argmax(x[:, e0]), c0], rtol=1e-12)
    others = [c for c in range(d) if c != c0]
    np.testing.assert_allclose(y[others], x[:, others].mean(axis=0), rtol=1e-14)


def test_compress_softmax_is_over_positions():
    # adding a per-channel constant to the positional bias is invisible to a
    # softmax over the m positions (it would not be to one over channels)
    d, m = 16, 4
    raw = _rand_bf16((1, 3 * m, d))
    W = _rand_bf16((d, d), 0.25)
    # multiples of 2^-10 plus small integers: the shifted bias is exact in fp32
    bias = (np.round(RNG.standard_normal((m, d)) * 1024) / 1024).astype(np.float32)
    shift = np.round(RNG.standard_normal(d) * 4).astype(np.float32)
    y0 = oracle.compress(raw, W, bias, m, 0, 3)
    y1 = oracle.compress(raw, W, bias + shift[None, :], m, 0, 3)
    np.testing.assert_allclose(y0, y1, rtol=1e-12, atol=1e-13)


def test_compress_output_is_convex_combination():
    d, m = 32, 128
    raw = _rand_bf16((1, 2 * m, d))
    y = oracle.compress(raw, _rand_bf16((d, d), 1 / math.sqrt(d)),
                        RNG.standard_normal((m, d)).astype(np.float32), m, 0, 2)
    x = bits_to_f64(raw).reshape(2, m, d)
    assert np.all(y[0] >= x.min(axis=1) - 1e-12) and np.all(y[0] <= x.max(axis=1) + 1e-12)


def test_quantize_e4m3_rows_scale_rule_and_error_bound():
    y = RNG.standard_normal((50, 64)) * np.exp(RNG.standard_normal((50, 1)) * 3)
    y[7] = 0.0
    codes, scales = oracle.quantize_e4m3_rows(y)
    assert scales[7] == 1.0 and np.all(codes[7] == 0)
    dec = oracle.e4m3_decode(codes)
    for r in range(50):
        if r == 7:
            continue
        amax = np.abs(y[r]).max()
        assert scales[r] == np.float32(amax / 448.0)
        assert np.abs(dec[r]).max() == 448.0  # the amax channel maps to the top code
        # nearest-code error bound: half the E4M3 spacing at each magnitude
        v = np.abs(y[r] / np.float64(scales[r]))
        e = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
        half_ulp = 2.0 ** (e - 4)
        assert np.all(np.abs(dec[r] - y[r] / np.float64(scales[r])) <= half_ulp * (1 + 1e-12))


# ---------------------------------------------------------------- a2 indexer

def test_indexer_hand_example_and_topk():
    g = _golden("indexer_hand.txt")
    q = bf16_bits(g["q"])[None, None]            # [1,1,2,2]
    k = bf16_bits(g["k"])[None]                  # [1,3,2]
    w = g["w"].astype(np.float32)[None, None]
    s, nv = oracle.indexer_scores(q, w, k, np.array([[2]]), np.array([3]), m=1)
    np.testing.assert_array_equal(s[0, 0], g["scores"])
    assert nv[0, 0] == 3
    np.testing.assert_array_equal(oracle.topk(s, nv, 2)[0, 0], g["top2"])


def test_indexer_unit_query_is_relu_of_key_channel():
    B, N, dI = 2, 50, 64
    k = _rand_bf16((B, N, dI))
    q = np.zeros((B, 1, 1, dI))
    q[0, 0, 0, 5] = 1.0
    q[1, 0, 0, 17] = 1.0
    s, _ = oracle.indexer_scores(bf16_bits(q), np.ones((B, 1, 1), np.float32), k,
                                 np.array([[N * 4], [N * 4]]), np.array([N, N]), m=4)
    kk = bits_to_f64(k)
    np.testing.assert_array_equal(s[0, 0], np.maximum(kk[0, :, 5], 0))
    np.testing.assert_array_equal(s[1, 0], np.maximum(kk[1, :, 17], 0))


def test_indexer_weight_sign_and_linearity():
    q = _rand_bf16((1, 1, 4, 64))
    k = _rand_bf16((1, 40, 64))
    w = RNG.standard_normal((1, 1, 4)).astype(np.float32)
    pos, n = np.array([[159]]), np.array([40])
    s1, _ = oracle.indexer_scores(q, w, k, pos, n, m=4)
    s2, _ = oracle.indexer_scores(q, -2 * w, k, pos, n, m=4)
    np.testing.assert_allclose(s2, -2 * s1, rtol=1e-15)
    # one head at a time sums to the total
    parts = 0
    for h in range(4):
        wh = np.zeros_like(w)
        wh[..., h] = w[..., h]
        parts = parts + oracle.indexer_scores(q, wh, k, pos, n, m=4)[0]
    np.testing.assert_allclose(parts, s1, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("m", [1, 4, 128])
def test_indexer_block_causal_visibility(m):
    N = 40
    k = _rand_bf16((1, N, 64))
    q = _rand_bf16((1, 6, 4, 64))
    pos = np.array([[0, m - 2, m - 1, 3 * m + 1, N * m - 1, N * m + 5 * m]]).clip(0)
    s, nv = oracle.indexer_scores(q, np.ones((1, 6, 4), np.float32), k, pos, np.array([N]), m)
    want = np.minimum(N, (pos + 1) // m)
    np.testing.assert_array_equal(nv, want)
    for t in range(6):
        assert np.all(np.isfinite(s[0, t, : want[0, t]]))
        assert np.all(s[0, t, want[0, t]:] == -np.inf)


def test_indexer_fp8_matches_bf16_on_shared_values_and_scales():
    # small integers are exact in both formats; power-of-two scales are exact
    qv = RNG.integers(-6, 7, (1, 1, 4, 64)).astype(np.float64)
    kv = RNG.integers(-6, 7, (1, 30, 64)).astype(np.float64)
    sq = (2.0 ** RNG.integers(-3, 4, (1, 1, 4))).astype(np.float32)
    sk = (2.0 ** RNG.integers(-3, 4, (1, 30))).astype(np.float32)
    w = RNG.standard_normal((1, 1, 4)).astype(np.float32)
    pos, n = np.array([[119]]), np.array([30])
    s8, _ = oracle.indexer_scores(oracle.e4m3_encode(qv), w, oracle.e4m3_encode(kv), pos, n,
                                  m=4, dtype=oracle.FP8_E4M3, q_scale=sq, k_scale=sk)
    sb, _ = oracle.indexer_scores(bf16_bits(qv * sq[..., None]), w,
                                  bf16_bits(kv * sk[..., None]), pos, n, m=4)
    np.testing.assert_allclose(s8, sb, rtol=1e-15)


# ---------------------------------------------------------------- a3 top-k

def test_topk_matches_lexsort_with_ties():
    Q, N, k = 40, 300, 37
    scores = RNG.integers(-5, 6, (Q, N)).astype(np.float64)  # heavy ties
    n_vis = RNG.integers(0, N + 1, Q).astype(np.int32)
    n_vis[:3] = [0, 5, k]
    got = oracle.topk(scores, n_vis, k)
    for qq in range(Q):
        nv = n_vis[qq]
        order = np.lexsort((np.arange(nv), -scores[qq, :nv]))[: min(k, nv)]
        want = np.full(k, -1, np.int32)
        want[: len(order)] = np.sort(order)
        np.testing.assert_array_equal(got[qq], want)


def test_topk_exhaustive_dominance_tiny():
    for trial in range(200):
        N = int(RNG.integers(1, 9))
        k = int(RNG.integers(1, 9))
        s = RNG.integers(0, 3, N).astype(np.float64)
        sel = oracle.topk(s[None], np.array([N]), k)[0]
        chosen = set(int(i) for i in sel if i >= 0)
        assert len(chosen) == min(k, N)
        assert list(sel[: len(chosen)]) == sorted(chosen)
        for i in chosen:
            for j in set(range(N)) - chosen:
                assert s[i] > s[j] or (s[i] == s[j] and i < j)


# ---------------------------------------------------------------- a4 / a5 attention

def _sdpa(qv, keys, vals, scale, bias=None):
    """torch SDPA in fp64: qv [H, D], keys/vals [S, D] shared by all heads."""
    H, D = qv.shape
    q = torch.from_numpy(qv)[None, :, None, :]
    kk = torch.from_numpy(keys)[None, None].expand(1, H, -1, D)
    vv = torch.from_numpy(vals)[None, None].expand(1, H, -1, D)
    mask = None if bias is None else torch.from_numpy(bias)[None, :, None, :]
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask, scale=scale)
    return o[0, :, 0].numpy()


def test_attention_hand_example():
    g = _golden("attention_hand.txt")
    q = bf16_bits(g["q"])[None, None]
    K = bf16_bits(g["K"])[None]
    V = bf16_bits(g["V"])[None]
    sel = np.array([[0, 1]], np.int32)
    for sink, o_key, l_key in ((None, "nosink_o", "nosink_lse"),
                               (np.array([g["sink"]], np.float32), "sink_o",
                                "sink_lse")):
        o, lse = oracle.attend(q, [0], [10], K, V, sel, None, None, 0, sink, float(g["scale"]))
        np.testing.assert_allclose(o[0, 0], g[o_key], rtol=1e-14)
        np.testing.assert_allclose(lse[0, 0], g[l_key], rtol=1e-14)


def test_hca_m1_no_window_no_sink_is_textbook_attention():
    # m' = 1: each compressed entry is one raw token, so HCA over n_vis = t+1
    # entries is plain causal MQA softmax attention
    B, N, H, D = 2, 70, 8, 32
    q = _rand_bf16((B, H, D), 0.3)
    K, V = _rand_bf16((B, N, D)), _rand_bf16((B, N, D))
    seq_len = np.array([45, 70], np.int32)
    o, lse = oracle.hca_decode(q, K, V, np.array([N, N]), 1, None, None, seq_len, 0, None, 0.7)
    for b in range(B):
        t = seq_len[b]
        keys, vals = bits_to_f64(K[b, :t]), bits_to_f64(V[b, :t])
        ref = _sdpa(bits_to_f64(q[b]), keys, vals, 0.7)
        np.testing.assert_allclose(o[b], ref, rtol=1e-12, atol=1e-13)
        logits = 0.7 * bits_to_f64(q[b]) @ keys.T
        np.testing.assert_allclose(lse[b], torch.logsumexp(torch.from_numpy(logits), -1).numpy(),
                                   rtol=1e-13)


def test_sink_is_an_extra_zero_value_key():
    B, N, H, D = 1, 33, 4, 16
    q = _rand_bf16((B, H, D))
    K, V = _rand_bf16((B, N, D)), _rand_bf16((B, N, D))
    sink = (RNG.standard_normal(H) * 3).astype(np.float32)
    o, lse = oracle.hca_decode(q, K, V, np.array([N]), 1, None, None, np.array([N]), 0, sink, 0.5)
    keys = np.concatenate([bits_to_f64(K[0]), np.zeros((1, D))])
    vals = np.concatenate([bits_to_f64(V[0]), np.zeros((1, D))])
    bias = np.zeros((H, N + 1))
    bias[:, N] = sink
    ref = _sdpa(bits_to_f64(q[0]), keys, vals, 0.5, bias)
    np.testing.assert_allclose(o[0], ref, rtol=1e-12, atol=1e-13)


def test_window_only_is_attention_over_recent_raw_tokens():
    B, L, H, D, Wn = 3, 300, 4, 16, 128
    q = _rand_bf16((B, H, D))
    Kr, Vr = _rand_bf16((B, L, D)), _rand_bf16((B, L, D))
    seq_len = np.array([300, 60, 1], np.int32)  # full window, clipped at 0, single token
    sel = np.full((B, 8), -1, np.int32)
    o, _ = oracle.csa_decode(q, Kr, Vr, sel, Kr, Vr, seq_len, Wn, None, 0.9)
    for b in range(B):
        t = seq_len[b] - 1
        lo = max(0, t - Wn + 1)
        ref = _sdpa(bits_to_f64(q[b]), bits_to_f64(Kr[b, lo:t + 1]), bits_to_f64(Vr[b, lo:t + 1]),
                    0.9)
        np.testing.assert_allclose(o[b], ref, rtol=1e-12, atol=1e-13)


def test_csa_with_all_entries_selected_equals_hca():
    B, L, m, H, D, Wn = 2, 400, 4, 8, 32, 16
    N = L // m
    q = _rand_bf16((B, H, D), 0.2)
    K, V = _rand_bf16((B, N, D)), _rand_bf16((B, N, D))
    Kr, Vr = _rand_bf16((B, L, D)), _rand_bf16((B, L, D))
    sink = RNG.standard_normal(H).astype(np.float32)
    seq_len = np.array([400, 203], np.int32)
    n_vis = seq_len // m
    sel = np.full((B, N + 7), -1, np.int32)
    for b in range(B):
        sel[b, : n_vis[b]] = np.arange(n_vis[b])
    o1, l1 = oracle.csa_decode(q, K, V, sel, Kr, Vr, seq_len, Wn, sink, 1.0)
    o2, l2 = oracle.hca_decode(q, K, V, np.array([N, N]), m, Kr, Vr, seq_len, Wn, sink, 1.0)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-13)


def test_weights_and_sink_mass_sum_to_one():
    # with every value row equal to ones, o_h = (total key mass) = 1 - sink mass
    B, N, H, D = 2, 64, 16, 8
    q = _rand_bf16((B, H, D))
    K = _rand_bf16((B, N, D))
    ones = bf16_bits(np.ones((B, N, D)))
    sink = (RNG.standard_normal(H) * 2).astype(np.float32)
    sel = np.stack([RNG.permutation(N)[:20] for _ in range(B)]).astype(np.int32)
    o, lse = oracle.csa_decode(q, K, ones, sel, K, ones, np.array([N, 40]), 16, sink, 1.0)
    np.testing.assert_allclose(o, (1 - np.exp(sink[None, :] - lse))[..., None].repeat(D, -1),
                               rtol=1e-13, atol=1e-14)


def test_split_merge_of_two_key_subsets_equals_one_pass():
    # lse-weighted merge of the compressed-only and window-only results (no
    # sink) reproduces the joint result: checks lse and the normalisation
    B, N, L, H, D = 1, 50, 200, 8, 32
    q = _rand_bf16((B, H, D), 0.3)
    K, V = _rand_bf16((B, N, D)), _rand_bf16((B, N, D))
    Kr, Vr = _rand_bf16((B, L, D)), _rand_bf16((B, L, D))
    sel = RNG.permutation(N)[None, :17].astype(np.int32)
    sl = np.array([L], np.int32)
    o, lse = oracle.csa_decode(q, K, V, sel, Kr, Vr, sl, 32, None, 1.0)
    oa, la = oracle.csa_decode(q, K, V, sel, None, None, sl, 0, None, 1.0)
    ob, lb = oracle.csa_decode(q, K, V, np.full_like(sel, -1), Kr, Vr, sl, 32, None, 1.0)
    Mx = np.maximum(la, lb)
    wa, wb = np.exp(la - Mx), np.exp(lb - Mx)
    merged = (wa[..., None] * oa + wb[..., None] * ob) / (wa + wb)[..., None]
    np.testing.assert_allclose(o, merged, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, Mx + np.log(wa + wb), rtol=1e-13)


def test_empty_key_set():
    q = _rand_bf16((1, 2, 8))
    K = _rand_bf16((1, 4, 8))
    sel = np.full((1, 3), -1, np.int32)
    o, lse = oracle.csa_decode(q, K, K, sel, None, None, np.array([4]), 0, None, 1.0)
    assert np.all(o == 0) and np.all(lse == -np.inf)
    sink = np.array([0.25, -1.5], np.float32)
    o, lse = oracle.csa_decode(q, K, K, sel, None, None, np.array([4]), 0, sink, 1.0)
    assert np.all(o == 0)
    np.testing.assert_array_equal(lse[0], sink.astype(np.float64))


def test_attention_rejects_out_of_range_indices():
    q = _rand_bf16((1, 2, 8))
    K = _rand_bf16((1, 4, 8))
    with pytest.raises(ValueError):
        oracle.csa_decode(q, K, K, np.array([[0, 4]], np.int32), None, None, np.array([16]), 0,
                          None, 1.0)
    with pytest.raises(ValueError):  # window reaches rows the raw buffer does not hold
        oracle.csa_decode(q, K, K, np.array([[0]], np.int32), K, K, np.array([16]), 4, None,
                          1.0)


# ---------------------------------------------------------------- grouped output projection

def test_out_proj_hand_example():
    g = _golden("out_proj_hand.txt")
    o = bf16_bits(g["o"]).reshape(1, 2, 2)
    W = bf16_bits(np.stack([g["W0"], g["W1"]]))
    np.testing.assert_array_equal(oracle.grouped_out_proj(o, W)[0], g["y"])


def test_out_proj_one_group_is_a_matmul():
    n, H, D, d = 5, 4, 8, 12
    o = _rand_bf16((n, H, D))
    W = _rand_bf16((1, d, H * D))
    want = bits_to_f64(o).reshape(n, H * D) @ bits_to_f64(W)[0].T
    np.testing.assert_allclose(oracle.grouped_out_proj(o, W), want, rtol=1e-13, atol=1e-13)


def test_out_proj_is_block_diagonal():
    # group g's outputs depend on group g's heads only: a block-diagonal
    # matrix (numpy) over all heads gives the same result
    n, H, D, G, d_g = 3, 8, 4, 4, 5
    K = (H // G) * D
    o = _rand_bf16((n, H, D))
    W = _rand_bf16((G, d_g, K))
    big = np.zeros((G * d_g, H * D))
    for g in range(G):
        big[g * d_g:(g + 1) * d_g, g * K:(g + 1) * K] = bits_to_f64(W)[g]
    want = bits_to_f64(o).reshape(n, H * D) @ big.T
    np.testing.assert_allclose(oracle.grouped_out_proj(o, W), want, rtol=1e-13, atol=1e-13)



# ---------------------------------------------------------------- FP8 KV storage

def test_kv8_dequantize_hand_example():
    g = _golden("kv8_hand.txt")
    codes = g["deq_codes"].astype(np.uint8)[None]
    out = oracle.kv8_dequantize(codes, np.array([g["deq_scale"]], np.float32),
                                bf16_bits(g["deq_rope"])[None])
    np.testing.assert_array_equal(out[0], g["deq_out"])


def test_kv8_dequantize_matches_torch_float8_times_scale():
    rows, dn, nr = 37, 64, 64
    codes = RNG.integers(0, 256, (rows, dn)).astype(np.uint8)
    codes[codes == 0x7F] = 0x7E  # leave out the NaN codes
    codes[codes == 0xFF] = 0xFE
    scale = (RNG.random(rows) * 0.02 + 1e-3).astype(np.float32)
    rope = bf16_bits(RNG.standard_normal((rows, nr)))
    out = oracle.kv8_dequantize(codes, scale, rope)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(out[:, :dn], dec * scale.astype(np.float64)[:, None])
    np.testing.assert_array_equal(out[:, dn:], bits_to_f64(rope))
    v = oracle.kv8_dequantize(codes, scale)  # V entries: no RoPE channels
    np.testing.assert_array_equal(v, out[:, :dn])


def test_attention_over_fp8_entries_hand_example():
    g = _golden("kv8_hand.txt")
    K = oracle.kv8_dequantize(g["k_codes"].astype(np.uint8).reshape(2, 1),
                              g["k_scale"].astype(np.float32),
                              bf16_bits(g["k_rope"]).reshape(2, 1))
    V = oracle.kv8_dequantize(g["v_codes"].astype(np.uint8), g["v_scale"].astype(np.float32))
    q = bf16_bits(g["q"])[None, None]
    o, lse = oracle.attend(q, [0], [10], K[None], V[None], np.array([[0, 1]], np.int32), None,
                           None, 0, None, float(g["scale"]))
    np.testing.assert_allclose(o[0, 0], g["o"], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], g["lse"], rtol=1e-14)


def test_attention_fp64_rows_equal_bf16_rows_on_shared_values():
    # FP8 codes with power-of-two scales decode to values that bf16 holds
    # exactly, so attention over the decoded rows must equal attention over
    # the same values stored as bf16 (the bf16 path is pinned above by SDPA)
    B, N, H, D, W = 2, 40, 4, 16, 8
    codes_k = RNG.integers(0, 0x7E, (B, N, D // 2)).astype(np.uint8)
    codes_k |= (RNG.integers(0, 2, codes_k.shape) << 7).astype(np.uint8)
    codes_v = RNG.integers(0, 0x7E, (B, N, D)).astype(np.uint8)
    sk = np.exp2(RNG.integers(-6, 3, (B, N))).astype(np.float32)
    sv = np.exp2(RNG.integers(-6, 3, (B, N))).astype(np.float32)
    rope = bf16_bits(RNG.standard_normal((B, N, D // 2)))
    K = oracle.kv8_dequantize(codes_k, sk, rope)
    V = oracle.kv8_dequantize(codes_v, sv)
    Kb, Vb = bf16_bits(K), bf16_bits(V)
    np.testing.assert_array_equal(bits_to_f64(Kb), K)
    np.testing.assert_array_equal(bits_to_f64(Vb), V)
    q = bf16_bits(RNG.standard_normal((B, H, D)) * 0.25)
    sel = np.stack([RNG.permutation(30)[:12] for _ in range(B)]).astype(np.int32)
    sel[1, 3] = -1
    kr, vr = bf16_bits(RNG.standard_normal((B, W, D))), bf16_bits(RNG.standard_normal((B, W, D)))
    sink = RNG.standard_normal(H).astype(np.float32)
    seq_len = np.array([128, 128], np.int32)
    a = oracle.csa_decode(q, K, V, sel, kr, vr, seq_len, W, sink, 0.3, raw_base=120)
    b = oracle.csa_decode(q, Kb, Vb, sel, kr, vr, seq_len, W, sink, 0.3, raw_base=120)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
