"""CUDA path vs the CPU oracle, element by element, on seeded inputs at sizes
the oracle finishes in seconds: several tiles, several splits, ragged tails,
edge cases.  All calls go through the C ABI (via the thin binding)."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_28_b300 as csa
import synth
from _util import (bf16_bound, check_attention, check_e4m3_rows, check_fp4_rows, check_topk, f64,
                   place_window, poisoned, u8, u16, window_arrays)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def rnd(shape, tid, scale=1.0, dtype=torch.bfloat16, seed=11):
    return synth.randn(shape, seed, tid, "cpu", scale=scale, dtype=dtype)


# ---------------------------------------------------------------- a1 compression

@pytest.mark.parametrize("d,m,fp8", [(128, 4, False), (64, 4, False), (128, 1, False),
                                     (128, 128, False), (64, 4, True), (128, 4, True),
                                     (64, 256, True), (128, 7, False)])
def test_compress_parity(cuda_device, d, m, fp8):
    B, bb, nb = 3, 2, 5
    N_cap = bb + nb + 2
    L = N_cap * m
    raw = rnd((B, L, d), 1)
    W = rnd((d, d), 2, 1 / math.sqrt(d))
    pb = rnd((m, d), 3, dtype=torch.float32)
    if fp8:
        out = torch.full((B, N_cap, d), 0x7F, dtype=torch.uint8, device=DEV)
        sc = torch.full((B, N_cap), float("nan"), device=DEV)
    else:
        out = poisoned((B, N_cap, d))
        sc = None
    csa.compress_kv(raw.to(DEV), W.to(DEV), pb.to(DEV), m, bb, nb, out, sc)
    torch.cuda.synchronize()
    y = oracle.compress(u16(raw), u16(W), pb.numpy(), m, bb, nb)
    if not fp8:
        g = f64(out[:, bb:bb + nb])
        assert np.all(np.abs(g - y) <= bf16_bound(y)), "beyond 1 bf16 ulp + fp32 error"
        exact = np.mean(u16(out[:, bb:bb + nb]) == oracle.quantize_bf16(y))
        assert exact > 0.99
        assert torch.isnan(out[:, :bb]).all() and torch.isnan(out[:, bb + nb:]).all()
        return
    check_e4m3_rows(u8(out[:, bb:bb + nb]), sc[:, bb:bb + nb].cpu().numpy(), y, "compress fp8")
    assert (out[:, :bb] == 0x7F).all() and (out[:, bb + nb:] == 0x7F).all()


@pytest.mark.parametrize("d,m,span,fp8,ring", [(128, 4, 8, False, False), (64, 4, 12, True, False),
                                                (128, 4, 16, True, True), (128, 1, 5, False, True)])
def test_compress_overlap_parity(cuda_device, d, m, span, fp8, ring):
    # blocks 0 .. 6: the first ones reach below position 0 (left out); ring:
    # the raw rows sit in a ring just long enough for the blocks' spans
    B, bb, nb = 3, 0, 7
    N_cap = nb + 1
    L = N_cap * m
    raw = rnd((B, L, d), 11)
    W = rnd((d, d), 12, 1 / math.sqrt(d))
    pb = rnd((span, d), 13, dtype=torch.float32)
    if ring:
        R = nb * m + span - m + 1
        src = torch.full((B, R, d), float("nan"), dtype=torch.bfloat16)
        for p in range(max(0, bb * m + m - span), (bb + nb) * m):
            src[:, p % R] = raw[:, p]
    else:
        src = raw
    if fp8:
        out = torch.full((B, N_cap, d), 0x7F, dtype=torch.uint8, device=DEV)
        sc = torch.full((B, N_cap), float("nan"), device=DEV)
    else:
        out = poisoned((B, N_cap, d))
        sc = None
    csa.compress_kv(src.to(DEV), W.to(DEV), pb.to(DEV), m, bb, nb, out, sc)
    torch.cuda.synchronize()
    y = oracle.compress(u16(raw), u16(W), pb.numpy(), m, bb, nb)
    if not fp8:
        g = f64(out[:, bb:bb + nb])
        assert np.all(np.abs(g - y) <= bf16_bound(y)), "beyond 1 bf16 ulp + fp32 error"
        assert torch.isnan(out[:, bb + nb:]).all()
        return
    check_e4m3_rows(u8(out[:, bb:bb + nb]), sc[:, bb:bb + nb].cpu().numpy(), y,
                    "compress fp8 overlap")


@pytest.mark.parametrize("d", [64, 128])
def test_compress_fp4_parity(cuda_device, d):
    # FP4 output: per 16 channels the nearest E4M3 scale to amax / 6 and the
    # nearest E2M1 codes of y / scale, against the oracle's fp64 entries:
    # every scale and code equal, except exact values within 1e-6 of a
    # rounding midpoint (check_fp4_rows)
    B, bb, nb, m = 3, 1, 6, 4
    N_cap = bb + nb + 1
    raw = rnd((B, N_cap * m, d), 21)
    W = rnd((d, d), 22, 1 / math.sqrt(d))
    pb = rnd((m, d), 23, dtype=torch.float32)
    out = torch.full((B, N_cap, d // 2), 0x77, dtype=torch.uint8, device=DEV)
    sc = torch.full((B, N_cap, d // 16), 0xFF, dtype=torch.uint8, device=DEV)
    csa.compress_kv(raw.to(DEV), W.to(DEV), pb.to(DEV), m, bb, nb, out, sc)
    torch.cuda.synchronize()
    y = oracle.compress(u16(raw), u16(W), pb.numpy(), m, bb, nb)
    check_fp4_rows(u8(out[:, bb:bb + nb]), u8(sc[:, bb:bb + nb]), y, f"compress fp4 d={d}")
    assert (u8(out[:, :bb]) == 0x77).all() and (u8(out[:, bb + nb:]) == 0x77).all()
    assert (u8(sc[:, :bb]) == 0xFF).all() and (u8(sc[:, bb + nb:]) == 0xFF).all()


# ---------------------------------------------------------------- a2 + a3 indexer top-k

@pytest.mark.parametrize("T", [1, 5, 12])
def test_indexer_fp4_parity(cuda_device, T):
    # FP4 indexer vectors (E2M1 codes + E4M3 scale per 16 channels): scores
    # element by element and the top-k set against the oracle
    B, N_cap, m, k = 3, 3000, 4, 200
    n_cmp = [3000, 2100, 150]
    q_pos = [[(4 * n_cmp[b] + 3) - 37 * (T - 1 - t) for t in range(T)] for b in range(B)]
    qc, qs = synth.rand_fp4_rows((B, T, 4, 64), 31, 1)
    kc, ks = synth.rand_fp4_rows((B, N_cap, 64), 31, 2)
    for b in range(B):  # entries beyond n_cmp are never read: poison them
        kc[b, n_cmp[b]:] = 0x77
        ks[b, n_cmp[b]:] = 0x7F
    w = synth.randn((B, T, 4), 31, 3, dtype=torch.float32)
    qp = torch.tensor(q_pos, dtype=torch.int32)
    nc = torch.tensor(n_cmp, dtype=torch.int32)
    args = (qc.to(DEV), w.to(DEV), kc.to(DEV), qp.to(DEV), nc.to(DEV), m)
    got = csa.indexer_scores(*args, q_scale=qs.to(DEV), k_scale=ks.to(DEV))
    idx, sc = csa.indexer_topk(*args, k, q_scale=qs.to(DEV), k_scale=ks.to(DEV),
                               return_scores=True)
    torch.cuda.synchronize()
    want, nv = oracle.indexer_scores(u8(qc), w.numpy(), u8(kc), qp.numpy(), nc.numpy(), m,
                                     oracle.FP4_E2M1, u8(qs), u8(ks))
    got = got.cpu().numpy().astype(np.float64)
    for b in range(B):
        for t in range(T):
            n = int(nv[b, t])
            np.testing.assert_allclose(got[b, t, :n], want[b, t, :n], rtol=2e-5, atol=2e-4)
    ref = oracle.topk(want, nv, k)
    check_topk(idx.cpu().numpy(), ref, want, nv, k, "indexer fp4")




def _indexer_case(B, T, N_cap, n_cmp, q_pos, fp8, seed=5):
    if fp8:
        qi, qs = synth.randn_fp8_rows((B, T, 4, 64), seed, 1)
        ki, ks = synth.randn_fp8_rows((B, N_cap, 64), seed, 2)
    else:
        qi, qs = synth.randn((B, T, 4, 64), seed, 1), None
        ki, ks = synth.randn((B, N_cap, 64), seed, 2), None
    w = synth.randn((B, T, 4), seed, 3, dtype=torch.float32)
    # entries beyond n_cmp must never be read: poison them
    for b in range(B):
        if fp8:
            ki[b, n_cmp[b]:] = 0x7F
        else:
            ki[b, n_cmp[b]:] = float("nan")
    return qi, qs, ki, ks, w, torch.tensor(q_pos, dtype=torch.int32), torch.tensor(
        n_cmp, dtype=torch.int32)


def _run_indexer(qi, qs, ki, ks, w, qp, nc, m, k):
    idx, sc = csa.indexer_topk(qi.to(DEV), w.to(DEV), ki.to(DEV), qp.to(DEV), nc.to(DEV), m, k,
                               q_scale=None if qs is None else qs.to(DEV),
                               k_scale=None if ks is None else ks.to(DEV), return_scores=True)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), sc.cpu().numpy()


def _oracle_indexer(qi, qs, ki, ks, w, qp, nc, m, k, fp8):
    conv = u8 if fp8 else u16
    s, nv = oracle.indexer_scores(conv(qi), w.numpy(), conv(ki), qp.numpy(), nc.numpy(), m,
                                  oracle.FP8_E4M3 if fp8 else oracle.BF16,
                                  None if qs is None else qs.numpy(),
                                  None if ks is None else ks.numpy())
    return s, nv, oracle.topk(s, nv, k)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("T", [1, 5, 12])  # up to 8 tokens per sequence: fused path
def test_indexer_topk_parity(cuda_device, fp8, T):
    B, N_cap, m, k = 3, 3000, 4, 200
    n_cmp = [3000, 2100, 150]
    base = [12003, 8401, 601]
    q_pos = [[base[b] - 37 * (T - 1 - t) for t in range(T)] for b in range(B)]
    case = _indexer_case(B, T, N_cap, n_cmp, q_pos, fp8)
    idx, sc = _run_indexer(*case, m, k)
    s, nv, ref = _oracle_indexer(*case, m, k, fp8)
    check_topk(idx, ref, s, nv, k, "indexer")
    # reported scores agree with the oracle's
    for b in range(B):
        for t in range(T):
            take = min(k, nv[b, t])
            got = sc[b, t, :take].astype(np.float64)
            want = s[b, t, idx[b, t, :take]]
            np.testing.assert_allclose(got, want, rtol=2e-5, atol=2e-4)
            assert np.all(np.isneginf(sc[b, t, take:]))


@pytest.mark.parametrize("fp8,T", [(False, 1), (True, 1), (False, 3), (True, 5),
                                    (False, 64), (False, 128)])
def test_indexer_scores_parity(cuda_device, fp8, T):
    # the a2 scores alone, element by element on the visible entries; T = 64
    # and 128 take the tensor-core scorer (whole 64-token blocks)
    B, N_cap, m = 2, 2500, 4
    n_cmp = [2500, 1303]
    q_pos = [[(n_cmp[b] * m + 1) * (t + 1) // T - 1 for t in range(T)] for b in range(B)]
    qi, qs, ki, ks, w, qp, nc = _indexer_case(B, T, N_cap, n_cmp, q_pos, fp8, seed=17)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = csa.indexer_scores(qi.to(DEV), w.to(DEV), ki.to(DEV), qp.to(DEV), nc.to(DEV), m,
                             q_scale=None if qs is None else qs.to(DEV),
                             k_scale=None if ks is None else ks.to(DEV), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = got.cpu().numpy().astype(np.float64)
    conv = u8 if fp8 else u16
    want, nv = oracle.indexer_scores(conv(qi), w.numpy(), conv(ki), qp.numpy(), nc.numpy(), m,
                                     oracle.FP8_E4M3 if fp8 else oracle.BF16,
                                     None if qs is None else qs.numpy(),
                                     None if ks is None else ks.numpy())
    for b in range(B):
        for t in range(T):
            n = int(nv[b, t])
            np.testing.assert_allclose(got[b, t, :n], want[b, t, :n], rtol=2e-5, atol=2e-4)


@pytest.mark.parametrize("B,T,N_cap,k", [(2, 64, 3000, 200), (2, 320, 3000, 256),
                                         (1, 256, 40000, 2048)])
def test_indexer_topk_parity_many_tokens(cuda_device, B, T, N_cap, k):
    # whole 64-token blocks of one sequence (chunked prefill): the scores come
    # from the tensor-core scorer; 320 tokens cross a 256-query chunk, 40000
    # entries give each CTA several key tiles (ring and TMEM buffers wrap)
    m = 4
    n_cmp = [N_cap, N_cap * 2 // 5 + 7][:B]
    q_pos = [[(n_cmp[b] * m + 2) * (t + 1) // T - 1 for t in range(T)] for b in range(B)]
    q_pos[0][0] = 1  # sees no entry
    case = _indexer_case(B, T, N_cap, n_cmp, q_pos, False)
    idx, sc = _run_indexer(*case, m, k)
    s, nv, ref = _oracle_indexer(*case, m, k, False)
    assert nv[0, 0] == 0 and (nv < k).any() and (nv > k).any()
    check_topk(idx, ref, s, nv, k, "indexer, many tokens")
    for b in range(B):
        for t in range(T):
            take = min(k, nv[b, t])
            got = sc[b, t, :take].astype(np.float64)
            want = s[b, t, idx[b, t, :take]]
            np.testing.assert_allclose(got, want, rtol=2e-5, atol=2e-4)
            assert np.all(np.isneginf(sc[b, t, take:]))


@pytest.mark.parametrize("N_cap,k", [(20000, 300), (200000, 5000)])
def test_topk_ties_take_lowest_indices(cuda_device, N_cap, k):
    # identical keys: every score ties, so the k lowest indices win, and they
    # come from the lowest-ranked CTAs of the select cluster; at 200000
    # entries one CTA's slice holds more threshold-bin entries than it keeps
    # in shared memory (the passes re-read the scores)
    B, m = 2, 4
    qi = synth.randn((B, 1, 4, 64), 3, 1)
    ki = synth.randn((1, 1, 64), 3, 2).expand(B, N_cap, 64).contiguous()
    w = torch.ones((B, 1, 4))
    w[1] = -1.0  # second query: all scores equal and <= 0
    qp = torch.tensor([[N_cap * m - 1], [N_cap * m - 1]], dtype=torch.int32)
    nc = torch.tensor([N_cap, N_cap], dtype=torch.int32)
    idx, _ = _run_indexer(qi, None, ki, None, w, qp, nc, m, k)
    np.testing.assert_array_equal(idx[:, 0], np.tile(np.arange(k), (B, 1)))


def test_topk_ties_many_queries(cuda_device):
    # 512 tokens of one sequence (several waves of select CTAs: the 512-thread
    # shape) over 20000 identical keys: every visible score ties, so each
    # token keeps the k lowest visible indices
    T, N_cap, m, k = 512, 20000, 4, 700
    qi = synth.randn((1, T, 4, 64), 5, 1)
    ki = synth.randn((1, 1, 64), 5, 2).expand(1, N_cap, 64).contiguous()
    w = torch.ones((1, T, 4))
    qp = torch.tensor([[N_cap * m - 1 - 37 * (T - 1 - t) for t in range(T)]], dtype=torch.int32)
    nc = torch.tensor([N_cap], dtype=torch.int32)
    idx, _ = _run_indexer(qi, None, ki, None, w, qp, nc, m, k)
    nv = np.minimum(N_cap, (qp.numpy() + 1) // m)
    want = np.stack([np.where(np.arange(k) < nv[0, t], np.arange(k), -1) for t in range(T)])
    np.testing.assert_array_equal(idx[0], want)


def test_topk_dense_threshold_bin_slow_path(cuda_device):
    # a one-hot query makes the score the key's first channel; those take 16
    # bf16 values in [1, 1.125): one histogram bin holds all 12000 entries
    B, N_cap, m, k = 2, 12000, 4, 777
    qi = torch.zeros((B, 1, 4, 64), dtype=torch.bfloat16)
    qi[:, :, 0, 0] = 1.0
    g = torch.Generator().manual_seed(9)
    ki = synth.randn((B, N_cap, 64), 4, 2)
    ki[:, :, 0] = (1.0 + torch.randint(0, 16, (B, N_cap), generator=g) / 128.0).to(torch.bfloat16)
    w = torch.tensor([1.0, 0.0, 0.0, 0.0]).repeat(B, 1, 1)
    qp = torch.tensor([[N_cap * m - 1], [N_cap * m - 3]], dtype=torch.int32)
    nc = torch.tensor([N_cap, N_cap], dtype=torch.int32)
    case = (qi, None, ki, None, w, qp, nc)
    idx, _ = _run_indexer(*case, m, k)
    s, nv, ref = _oracle_indexer(*case, m, k, False)
    np.testing.assert_array_equal(idx, ref)  # exact: ties resolved by index


@pytest.mark.parametrize("n_levels", [16, 128])
def test_topk_dense_threshold_bin_many_queries(cuda_device, n_levels):
    # 160 queries in one call (the one-CTA-per-query select), scores drawn
    # from n_levels bf16 values 1 + j/128: with 16 every entry falls in one
    # level-1 bin (12000 keys: levels 2 and 3 streamed from the scores
    # again); with 128 eight bins of about 1500 tied keys each (levels 2 and 3
    # on the candidate list in shared memory)
    T, N_cap, m, k = 160, 12000, 4, 777
    qi = torch.zeros((1, T, 4, 64), dtype=torch.bfloat16)
    qi[:, :, 0, 0] = 1.0
    g = torch.Generator().manual_seed(10)
    ki = synth.randn((1, N_cap, 64), 4, 3)
    ki[:, :, 0] = (1.0 + torch.randint(0, n_levels, (1, N_cap), generator=g) / 128.0
                   ).to(torch.bfloat16)
    w = torch.tensor([1.0, 0.0, 0.0, 0.0]).repeat(1, T, 1)
    qp = torch.tensor([[N_cap * m - 1 - 61 * (T - 1 - t) for t in range(T)]], dtype=torch.int32)
    nc = torch.tensor([N_cap], dtype=torch.int32)
    case = (qi, None, ki, None, w, qp, nc)
    idx, _ = _run_indexer(*case, m, k)
    s, nv, ref = _oracle_indexer(*case, m, k, False)
    np.testing.assert_array_equal(idx, ref)  # exact: ties resolved by index


@pytest.mark.parametrize("sampled", ["low", "high"])
def test_topk_stream_skewed_sample(cuda_device, sampled):
    # the one-CTA-per-query select first bounds the list from an evenly spaced
    # sample of 16-byte score vectors (entries 16 i .. 16 i + 3 at 20000
    # visible entries).  Scores that give the sampled entries the smallest
    # ("low": far more than the list holds lie above the sample's bound) or
    # the largest values ("high": fewer than k lie above it) send every query
    # to the histogram passes; the selection stays exact
    T, N_cap, m, k = 160, 20000, 4, 1500
    qi = torch.zeros((1, T, 4, 64), dtype=torch.bfloat16)
    qi[:, :, 0, 0] = 1.0
    g = torch.Generator().manual_seed(21)
    ki = synth.randn((1, N_cap, 64), 6, 3)
    val = 1.0 + torch.rand((1, N_cap), generator=g)
    in_sample = (torch.arange(N_cap) % 16) < 4  # 5000 entries, about 4100 of them sampled
    low = 0.25 + torch.rand((1, N_cap), generator=g) / 8
    high = 3.0 + torch.rand((1, N_cap), generator=g)
    val[:, in_sample] = (low if sampled == "low" else high)[:, in_sample]
    ki[:, :, 0] = val.to(torch.bfloat16)
    w = torch.tensor([1.0, 0.0, 0.0, 0.0]).repeat(1, T, 1)
    qp = torch.tensor([[N_cap * m - 1 - 3 * (T - 1 - t) for t in range(T)]], dtype=torch.int32)
    nc = torch.tensor([N_cap], dtype=torch.int32)
    case = (qi, None, ki, None, w, qp, nc)
    idx, _ = _run_indexer(*case, m, k)
    s, nv, ref = _oracle_indexer(*case, m, k, False)
    np.testing.assert_array_equal(idx, ref)  # exact: ties resolved by index


def test_topk_stream_large_k_histogram_path(cuda_device):
    # 2k above the 4096-entry list: the one-CTA-per-query select skips the
    # sampled bound and runs the histogram passes (pass 1, then the list of
    # the threshold bin and above through the per-warp buckets, or the
    # candidate passes when that list would not fit)
    T, N_cap, m, k = 160, 24000, 4, 2100
    qi = synth.randn((1, T, 4, 64), 8, 1)
    ki = synth.randn((1, N_cap, 64), 8, 2)
    w = synth.randn((1, T, 4), 8, 3, dtype=torch.float32)
    qp = torch.tensor([[N_cap * m - 1 - 50 * (T - 1 - t) for t in range(T)]], dtype=torch.int32)
    nc = torch.tensor([N_cap], dtype=torch.int32)
    case = (qi, None, ki, None, w, qp, nc)
    idx, _ = _run_indexer(*case, m, k)
    s, nv, ref = _oracle_indexer(*case, m, k, False)
    check_topk(idx, ref, s, nv, k, "stream select, k = 2100")


def test_topk_zero_scores_and_short_lists(cuda_device):
    # n_vis below k (every visible entry, -1 padded), n_vis == 0, and a query
    # whose scores are mostly exactly zero (negative dot products)
    B, N_cap, m, k = 4, 600, 4, 64
    case = list(_indexer_case(B, 1, N_cap, [600, 600, 10, 600], [[2399], [3], [2399], [2399]],
                              False))
    case[2][:, :, :] = case[2].abs()  # positive keys ...
    case[0][3] = -case[0][3].abs()  # ... and a negative query: every score of query 3 is 0
    idx, _ = _run_indexer(*case, m, k)
    s, nv, ref = _oracle_indexer(*case, m, k, False)
    assert nv.ravel().tolist() == [600, 1, 10, 600]
    check_topk(idx, ref, s, nv, k, "short lists")
    np.testing.assert_array_equal(idx[1, 0], [0] + [-1] * (k - 1))
    np.testing.assert_array_equal(idx[3, 0], np.arange(k))


# ---------------------------------------------------------------- a4 / a5 attention

def _attn_inputs(B, H, N_cap, lens, seed=21, W=128):
    q = synth.randn((B, H, 128), seed, 1, scale=1 / math.sqrt(128))
    kc, vc = synth.randn((B, N_cap, 128), seed, 2), synth.randn((B, N_cap, 128), seed, 3)
    kw, vw = synth.randn((B, W, 128), seed, 4), synth.randn((B, W, 128), seed, 5)
    sink = synth.randn((H,), seed, 6, dtype=torch.float32)
    return q, kc, vc, kw, vw, sink


def _random_topk(B, k, n_vis, seed=3):
    g = np.random.default_rng(seed)
    sel = np.full((B, k), -1, np.int32)
    for b in range(B):
        take = min(k, n_vis[b])
        sel[b, :take] = np.sort(g.choice(n_vis[b], take, replace=False))
    return sel


@pytest.mark.parametrize("H", [16, 64, 128])
@pytest.mark.parametrize("with_sink", [True, False])
def test_sparse_decode_parity(cuda_device, H, with_sink):
    B, N_cap, k, W = 3, 300, 48, 128
    lens = [700, 129, 37]
    q, kc, vc, kw, vw, sink = _attn_inputs(B, H, N_cap, lens)
    sink = sink if with_sink else None
    n_vis = [min(N_cap, n // 4) for n in lens]
    sel = _random_topk(B, k, n_vis)
    kc_d = kc.to(DEV)
    vc_d = vc.to(DEV)
    for b in range(B):  # entries beyond n_vis are never selected: poison them
        kc_d[b, n_vis[b]:] = float("nan")
        vc_d[b, n_vis[b]:] = float("nan")
    out, lse = csa.sparse_attn_decode(
        q.to(DEV), kc_d, vc_d, torch.from_numpy(sel).to(DEV), place_window(kw, lens, 800),
        place_window(vw, lens, 800), torch.tensor(lens, dtype=torch.int32, device=DEV), W,
        None if sink is None else sink.to(DEV), return_lse=True)
    torch.cuda.synchronize()
    kr, base = window_arrays(kw, lens)
    vr, _ = window_arrays(vw, lens)
    ro, rl = oracle.csa_decode(u16(q), u16(kc), u16(vc), sel, kr, vr, np.array(lens), W,
                               None if sink is None else sink.numpy(), 1.0, base)
    check_attention(out, ro, lse, rl, f"csa decode H={H}")


def test_sparse_decode_many_splits_multi_tile(cuda_device):
    # 40 queries x 640 keys: 8 splits of 128 keys (two 64-key tiles each)
    B, H, N_cap, k, W = 40, 64, 900, 512, 128
    lens = [3600 - 37 * b for b in range(B)]
    q, kc, vc, kw, vw, sink = _attn_inputs(B, H, N_cap, lens, seed=33)
    n_vis = [min(N_cap, n // 4) for n in lens]
    sel = _random_topk(B, k, n_vis, seed=8)
    out, lse = csa.sparse_attn_decode(
        q.to(DEV), kc.to(DEV), vc.to(DEV), torch.from_numpy(sel).to(DEV),
        place_window(kw, lens, 3600), place_window(vw, lens, 3600),
        torch.tensor(lens, dtype=torch.int32, device=DEV), W, sink.to(DEV), return_lse=True)
    torch.cuda.synchronize()
    kr, base = window_arrays(kw, lens)
    vr, _ = window_arrays(vw, lens)
    ro, rl = oracle.csa_decode(u16(q), u16(kc), u16(vc), sel, kr, vr, np.array(lens), W,
                               sink.numpy(), 1.0, base)
    check_attention(out, ro, lse, rl, "csa decode splits")


@pytest.mark.parametrize("ws", [None, False])
def test_many_keys_few_queries_split_modes(cuda_device, ws):
    # 25 tiles of keys for each of 1-2 queries: clusters of 16 splits would
    # leave most SMs idle, so with a workspace (ws=None: the binding sizes one)
    # the keys are split 25 ways without a cluster and merged by a second
    # kernel; ws=False forces the in-cluster merge.  Both against the oracle.
    H, m = 64, 8
    lens = [24000, 23001]
    N_cap = 3000
    n_cmp = [3000, 2875]
    q, kc, vc, kw, vw, sink = _attn_inputs(2, H, N_cap, lens, seed=61)
    out, lse = csa.hca_dense_attn_decode(
        q.to(DEV), kc.to(DEV), vc.to(DEV), torch.tensor(n_cmp, dtype=torch.int32, device=DEV), m,
        place_window(kw, lens, 24000), place_window(vw, lens, 24000),
        torch.tensor(lens, dtype=torch.int32, device=DEV), 128, sink.to(DEV), return_lse=True,
        ws=ws)
    torch.cuda.synchronize()
    kr, base = window_arrays(kw, lens)
    vr, _ = window_arrays(vw, lens)
    ro, rl = oracle.hca_decode(u16(q), u16(kc), u16(vc), np.array(n_cmp), m, kr, vr,
                               np.array(lens), 128, sink.numpy(), 1.0, base)
    check_attention(out, ro, lse, rl, f"hca many keys ws={ws}")
    # one CSA query with 3000 selected entries (+128 window)
    lens1 = [16004]
    q1, kc1, vc1, kw1, vw1, sink1 = _attn_inputs(1, H, 4001, lens1, seed=62)
    sel = _random_topk(1, 3000, [4001], seed=9)
    out1, lse1 = csa.sparse_attn_decode(
        q1.to(DEV), kc1.to(DEV), vc1.to(DEV), torch.from_numpy(sel).to(DEV),
        place_window(kw1, lens1, 16004), place_window(vw1, lens1, 16004),
        torch.tensor(lens1, dtype=torch.int32, device=DEV), 128, sink1.to(DEV), return_lse=True,
        ws=ws)
    torch.cuda.synchronize()
    kr1, base1 = window_arrays(kw1, lens1)
    vr1, _ = window_arrays(vw1, lens1)
    ro1, rl1 = oracle.csa_decode(u16(q1), u16(kc1), u16(vc1), sel, kr1, vr1, np.array(lens1),
                                 128, sink1.numpy(), 1.0, base1)
    check_attention(out1, ro1, lse1, rl1, f"csa 3000 entries ws={ws}")


def test_decode_window_only_and_compressed_only(cuda_device):
    B, H, N_cap, k = 2, 64, 100, 32
    lens = [400, 90]
    q, kc, vc, kw, vw, sink = _attn_inputs(B, H, N_cap, lens, seed=44)
    n_vis = [min(N_cap, n // 4) for n in lens]
    sel = _random_topk(B, k, n_vis, seed=1)
    L = torch.tensor(lens, dtype=torch.int32, device=DEV)
    kr, base = window_arrays(kw, lens)
    vr, _ = window_arrays(vw, lens)
    # compressed entries only (window 0, no raw cache)
    out = csa.sparse_attn_decode(q.to(DEV), kc.to(DEV), vc.to(DEV),
                                 torch.from_numpy(sel).to(DEV), None, None, L, 0, sink.to(DEV))
    ro, _ = oracle.csa_decode(u16(q), u16(kc), u16(vc), sel, None, None, np.array(lens), 0,
                              sink.numpy(), 1.0)
    check_attention(out, ro, what="compressed only")
    # window only (every top-k slot is padding)
    pad = np.full_like(sel, -1)
    out = csa.sparse_attn_decode(q.to(DEV), kc.to(DEV), vc.to(DEV),
                                 torch.from_numpy(pad).to(DEV), place_window(kw, lens, 400),
                                 place_window(vw, lens, 400), L, 128, sink.to(DEV))
    ro, _ = oracle.csa_decode(u16(q), u16(kc), u16(vc), pad, kr, vr, np.array(lens), 128,
                              sink.numpy(), 1.0, base)
    check_attention(out, ro, what="window only")


@pytest.mark.parametrize("window", [128, 0])
def test_hca_decode_parity(cuda_device, window):
    B, H, m = 4, 64, 8
    lens = [1000, 517, 64, 5]
    N_cap = 130
    n_cmp = [125, 64, 8, 0]
    q, kc, vc, kw, vw, sink = _attn_inputs(B, H, N_cap, lens, seed=55)
    kc_d, vc_d = kc.to(DEV), vc.to(DEV)
    for b in range(B):
        nv = min(n_cmp[b], lens[b] // m)
        kc_d[b, nv:] = float("nan")
        vc_d[b, nv:] = float("nan")
    out, lse = csa.hca_dense_attn_decode(
        q.to(DEV), kc_d, vc_d, torch.tensor(n_cmp, dtype=torch.int32, device=DEV), m,
        place_window(kw, lens, 1000) if window else None,
        place_window(vw, lens, 1000) if window else None,
        torch.tensor(lens, dtype=torch.int32, device=DEV), window, sink.to(DEV), return_lse=True)
    torch.cuda.synchronize()
    kr, base = window_arrays(kw, lens)
    vr, _ = window_arrays(vw, lens)
    ro, rl = oracle.hca_decode(u16(q), u16(kc), u16(vc), np.array(n_cmp), m,
                               kr if window else None, vr if window else None, np.array(lens),
                               window, sink.numpy(), 1.0, base)
    check_attention(out, ro, lse, rl, f"hca window={window}")
    if window == 0:  # sequence 3 sees nothing: output 0, lse = sink
        assert torch.all(out[3] == 0)
        np.testing.assert_allclose(lse[3].cpu().numpy(), sink.numpy(), rtol=1e-6)


def test_prefill_parity(cuda_device):
    B, T, H, N_cap, k, W, m = 2, 37, 64, 140, 48, 128, 4
    q_pos = np.array([[500 + t for t in range(T)], [100 + 3 * t for t in range(T)]], np.int32)
    L_cap = 700
    q = synth.randn((B, T, H, 128), 61, 1, scale=1 / math.sqrt(128))
    kc, vc = synth.randn((B, N_cap, 128), 61, 2), synth.randn((B, N_cap, 128), 61, 3)
    kr, vr = synth.randn((B, L_cap, 128), 61, 4), synth.randn((B, L_cap, 128), 61, 5)
    sink = synth.randn((H,), 61, 6, dtype=torch.float32)
    n_vis = np.minimum(N_cap, (q_pos + 1) // m)
    g = np.random.default_rng(4)
    sel = np.full((B, T, k), -1, np.int32)
    for b in range(B):
        for t in range(T):
            take = min(k, n_vis[b, t])
            sel[b, t, :take] = np.sort(g.choice(n_vis[b, t], take, replace=False))
    kr_d, vr_d = kr.to(DEV), vr.to(DEV)
    kr_d[:, 611:] = float("nan")  # beyond the last query position
    vr_d[:, 611:] = float("nan")
    out, lse = csa.sparse_attn_prefill(
        q.to(DEV), kc.to(DEV), vc.to(DEV), torch.from_numpy(sel).to(DEV), kr_d, vr_d,
        torch.from_numpy(q_pos).to(DEV), W, sink.to(DEV), return_lse=True)
    torch.cuda.synchronize()
    ro, rl = oracle.csa_prefill(u16(q), u16(kc), u16(vc), sel, u16(kr), u16(vr), q_pos, W,
                                sink.numpy(), 1.0)
    check_attention(out, ro, lse, rl, "prefill")


def _bi_case(B, T, seed, N_cap=1500, k=1024, L_cap=6100, m=4):
    q = synth.randn((B, T, 64, 128), seed, 1, scale=1 / math.sqrt(128))
    kc, vc = synth.randn((B, N_cap, 128), seed, 2), synth.randn((B, N_cap, 128), seed, 3)
    kr, vr = synth.randn((B, L_cap, 128), seed, 4), synth.randn((B, L_cap, 128), seed, 5)
    sink = synth.randn((64,), seed, 6, dtype=torch.float32)
    g = np.random.default_rng(seed)
    q_pos = np.stack([6000 - 3 * b + np.arange(T) for b in range(B)]).astype(np.int32)
    n_vis = np.minimum(N_cap, (q_pos + 1) // m)
    sel = np.full((B, T, k), -1, np.int32)
    for b in range(B):
        for t in range(T):
            take = min(k, n_vis[b, t])
            sel[b, t, :take] = np.sort(g.choice(n_vis[b, t], take, replace=False))
    return q, kc, vc, kr, vr, sink, q_pos, sel


def _bi_run(case, kps, rows=None):
    q, kc, vc, kr, vr, sink, q_pos, sel = case
    if rows is not None:  # a sub-batch of the same sequences
        q, kc, vc, kr, vr = q[rows], kc[rows], vc[rows], kr[rows], vr[rows]
        q_pos, sel = q_pos[rows], sel[rows]
    out, lse = csa.sparse_attn_batch_invariant(
        q.to(DEV), kc.to(DEV), vc.to(DEV), torch.from_numpy(np.ascontiguousarray(sel)).to(DEV),
        kr.to(DEV), vr.to(DEV), torch.from_numpy(np.ascontiguousarray(q_pos)).to(DEV), 128,
        sink.to(DEV), keys_per_split=kps, return_lse=True)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


@pytest.mark.parametrize("T", [1, 2])  # decode, and a two-token (multi-token) step
def test_batch_invariant_attention_parity(cuda_device, T):
    case = _bi_case(3, T, 71)
    out, lse = _bi_run(case, 256)
    q, kc, vc, kr, vr, sink, q_pos, sel = case
    ro, rl = oracle.csa_prefill(u16(q), u16(kc), u16(vc), sel, u16(kr), u16(vr), q_pos, 128,
                                sink.numpy(), 1.0)
    check_attention(out, ro, lse, rl, f"batch-invariant T={T}")


def test_batch_invariant_attention_is_bitwise_independent_of_the_batch(cuda_device):
    # the same sequences alone, in a batch of 24, and a token alone vs in a
    # two-token step: bitwise equal outputs and lse
    big = _bi_case(24, 2, 72)
    out_b, lse_b = _bi_run(big, 320)
    for rows in ([5], [0, 17], list(range(24))[::-1][:9]):
        out_s, lse_s = _bi_run(big, 320, rows)
        assert torch.equal(out_s, out_b[rows]) and torch.equal(lse_s, lse_b[rows])
    q, kc, vc, kr, vr, sink, q_pos, sel = big
    one = (q[:, 1:], kc, vc, kr, vr, sink, q_pos[:, 1:], sel[:, 1:])
    out_1, lse_1 = _bi_run(one, 320)
    assert torch.equal(out_1[:, 0], out_b[:, 1]) and torch.equal(lse_1[:, 0], lse_b[:, 1])
    # the automatic plan (split count from the batch) agrees within rounding
    out_a, lse_a = csa.sparse_attn_prefill(
        q.to(DEV), kc.to(DEV), vc.to(DEV), torch.from_numpy(sel).to(DEV), kr.to(DEV),
        vr.to(DEV), torch.from_numpy(q_pos).to(DEV), 128, sink.to(DEV), return_lse=True)
    torch.cuda.synchronize()
    assert (out_a.cpu().float() - out_b.float()).abs().max().item() < 2e-2
    assert (lse_a.cpu() - lse_b).abs().max().item() < 1e-3


@pytest.mark.parametrize("n,G,d_g", [(1, 8, 128), (32, 8, 512), (300, 4, 256), (77, 16, 128),
                                     (5, 32, 128), (600, 8, 512)])
def test_grouped_out_proj_parity(cuda_device, n, G, d_g):
    # 300 queries: two tiles (256 + a ragged 44); K = (64 / G) * 128; few
    # queries split K over a cluster (G = 32: K = 256, 4 slabs, 4 splits of
    # one); 600 queries: three tiles, no split
    H, D = 64, 128
    K = (H // G) * D
    o = synth.randn((n, H, D), 81, 1)
    W = synth.randn((G, d_g, K), 81, 2, scale=1 / math.sqrt(K))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = csa.grouped_out_proj(o.to(DEV), W.to(DEV), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.grouped_out_proj(u16(o), u16(W))
    g = f64(y)
    # bf16 rounding of the result plus fp32 accumulation over K products
    mag = np.abs(oracle.grouped_out_proj(u16(o.abs()), u16(W.abs())))
    assert np.all(np.abs(g - ref) <= bf16_bound(ref) + K * 2.0 ** -23 * mag)


def test_softmax_scale_is_applied(cuda_device):
    B, H, N_cap, k = 2, 32, 64, 16
    lens = [256, 256]
    q, kc, vc, kw, vw, sink = _attn_inputs(B, H, N_cap, lens, seed=77)
    q = (q.float() * math.sqrt(128)).to(torch.bfloat16)  # unscaled query
    sel = _random_topk(B, k, [64, 64], seed=2)
    L = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out = csa.sparse_attn_decode(q.to(DEV), kc.to(DEV), vc.to(DEV),
                                 torch.from_numpy(sel).to(DEV), place_window(kw, lens, 256),
                                 place_window(vw, lens, 256), L, 128, sink.to(DEV),
                                 softmax_scale=1 / math.sqrt(128))
    kr, base = window_arrays(kw, lens)
    vr, _ = window_arrays(vw, lens)
    ro, _ = oracle.csa_decode(u16(q), u16(kc), u16(vc), sel, kr, vr, np.array(lens), 128,
                              sink.numpy(), 1 / math.sqrt(128), base)
    check_attention(out, ro, what="softmax scale")


# ---------------------------------------------------------------- errors, determinism

def test_bad_indices_and_positions_set_the_error_word(cuda_device):
    B, H, N_cap, k = 2, 64, 64, 8
    lens = [200, 200]
    q, kc, vc, kw, vw, sink = _attn_inputs(B, H, N_cap, lens, seed=88)
    sel = _random_topk(B, k, [50, 50], seed=3)
    bad = sel.copy()
    bad[0, 2] = N_cap + 5  # out of range: skipped and flagged
    bad[1, 3] = -7
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    L = torch.tensor(lens, dtype=torch.int32, device=DEV)
    kr_d, vr_d = place_window(kw, lens, 256), place_window(vw, lens, 256)
    out = csa.sparse_attn_decode(q.to(DEV), kc.to(DEV), vc.to(DEV),
                                 torch.from_numpy(bad).to(DEV), kr_d, vr_d, L, 128,
                                 sink.to(DEV), err_word=err)
    torch.cuda.synchronize()
    assert err.item() & csa.EW_BAD_INDEX
    assert torch.isfinite(out.float()).all()
    # the flagged entries are skipped, exactly as if they were padding
    skip = bad.copy()
    skip[0, 2] = -1
    skip[1, 3] = -1
    kr, base = window_arrays(kw, lens)
    vr, _ = window_arrays(vw, lens)
    ro, _ = oracle.csa_decode(u16(q), u16(kc), u16(vc), skip, kr, vr, np.array(lens), 128,
                              sink.numpy(), 1.0, base)
    check_attention(out, ro, what="skipped bad indices")
    # an empty sequence (length 0, position -1): flagged, its window dropped,
    # no fault; only the compressed entries and the sink remain
    err.zero_()
    L2 = torch.tensor([200, 0], dtype=torch.int32, device=DEV)
    out2 = csa.sparse_attn_decode(q.to(DEV), kc.to(DEV), vc.to(DEV),
                                  torch.from_numpy(sel).to(DEV), kr_d, vr_d, L2, 128,
                                  sink.to(DEV), err_word=err)
    torch.cuda.synchronize()
    assert err.item() & csa.EW_BAD_POSITION
    assert torch.isfinite(out2.float()).all()


def test_determinism_bitwise(cuda_device):
    wl = synth.Workload("det", "csa_decode", B=4, L=16384, m=4, H=64, k=512)
    from sparse_attention_28_b300.steps import make_step
    step = make_step(synth.make_inputs(wl, seed=3, device=DEV), DEV)
    a = step().clone()
    ia = step.idx.clone()
    b = step().clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(ia, step.idx)


def test_decode_with_window_ring_cache(cuda_device):
    # raw caches as rings of exactly W rows: position p lives at row p mod W
    B, H, N_cap, k, W = 3, 64, 200, 40, 128
    lens = [5000, 777, 90]
    q, kc, vc, kw, vw, sink = _attn_inputs(B, H, N_cap, lens, seed=99)
    n_vis = [min(N_cap, n // 4) for n in lens]
    sel = _random_topk(B, k, n_vis, seed=5)
    kr_ring, vr_ring = poisoned((B, W, 128)), poisoned((B, W, 128))
    for b, n in enumerate(lens):
        lo = max(0, n - W)
        rows = torch.arange(lo, n) % W
        kr_ring[b, rows] = kw[b, W - (n - lo):].to(DEV)
        vr_ring[b, rows] = vw[b, W - (n - lo):].to(DEV)
    out, lse = csa.sparse_attn_decode(
        q.to(DEV), kc.to(DEV), vc.to(DEV), torch.from_numpy(sel).to(DEV), kr_ring, vr_ring,
        torch.tensor(lens, dtype=torch.int32, device=DEV), W, sink.to(DEV), return_lse=True)
    torch.cuda.synchronize()
    kr, base = window_arrays(kw, lens)
    vr, _ = window_arrays(vw, lens)
    ro, rl = oracle.csa_decode(u16(q), u16(kc), u16(vc), sel, kr, vr, np.array(lens), W,
                               sink.numpy(), 1.0, base)
    check_attention(out, ro, lse, rl, "ring cache")
