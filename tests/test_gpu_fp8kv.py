"""FP8-stored compressed KV (E4M3 non-RoPE channels with a per-entry scale,
bf16 RoPE channels; V all E4M3): the mixed-storage compression and the
attention over such entries, against the CPU oracle on seeded inputs.  All
calls go through the C ABI (via the thin binding)."""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_28_b300 as csa
import synth
from _util import (bf16_bound, check_attention, check_e4m3_rows, f64, lse_tol, place_window, u8,
                   u16, window_arrays)

pytestmark = pytest.mark.gpu
DEV = "cuda"


# ---------------------------------------------------------------- compression

@pytest.mark.parametrize("d,n_rope,m,span", [(128, 64, 4, 4), (64, 16, 4, 4), (128, 64, 4, 8),
                                             (128, 32, 128, 128)])
def test_compress_mixed_parity(cuda_device, d, n_rope, m, span):
    B, bb, nb = 3, 2, 5
    N_cap = bb + nb + 2
    L = N_cap * m
    dn = d - n_rope
    raw = synth.randn((B, L, d), 12, 1)
    W = synth.randn((d, d), 12, 2, scale=1 / math.sqrt(d))
    pb = synth.randn((span, d), 12, 3, dtype=torch.float32)
    codes = torch.full((B, N_cap, dn), 0x7F, dtype=torch.uint8, device=DEV)
    sc = torch.full((B, N_cap), float("nan"), device=DEV)
    rope = torch.full((B, N_cap, n_rope), float("nan"), dtype=torch.bfloat16, device=DEV)
    csa.compress_kv_mixed(raw.to(DEV), W.to(DEV), pb.to(DEV), m, bb, nb, codes, sc, rope)
    torch.cuda.synchronize()
    y = oracle.compress(u16(raw), u16(W), pb.numpy(), m, bb, nb)
    check_e4m3_rows(u8(codes[:, bb:bb + nb]), sc[:, bb:bb + nb].cpu().numpy(), y[..., :dn],
                    "mixed compression")
    g = f64(rope[:, bb:bb + nb])
    assert np.all(np.abs(g - y[..., dn:]) <= bf16_bound(y[..., dn:])), "RoPE channels"
    # nothing outside the written blocks
    assert (codes[:, :bb] == 0x7F).all() and (codes[:, bb + nb:] == 0x7F).all()
    assert torch.isnan(sc[:, :bb]).all() and torch.isnan(sc[:, bb + nb:]).all()
    assert torch.isnan(rope[:, :bb]).all() and torch.isnan(rope[:, bb + nb:]).all()


# ---------------------------------------------------------------- attention

def _kv8(B, N_cap, n_vis, seed):
    """FP8 cache on the device with entries >= n_vis[b] poisoned (NaN codes
    and scales), and the oracle's decoded fp64 K and V."""
    kn, ks, kr, v, vs = synth.randn_kv8(B, N_cap, seed, 10)
    K = oracle.kv8_dequantize(u8(kn), ks.numpy(), u16(kr))
    V = oracle.kv8_dequantize(u8(v), vs.numpy())
    dev = [t.to(DEV) for t in (kn, ks, kr, v, vs)]
    for b in range(B):
        dev[0][b, n_vis[b]:] = 0x7F
        dev[1][b, n_vis[b]:] = float("nan")
        dev[2][b, n_vis[b]:] = float("nan")
        dev[3][b, n_vis[b]:] = 0x7F
        dev[4][b, n_vis[b]:] = float("nan")
    return dev, K, V


def _random_topk(B, k, n_vis, seed=3):
    g = np.random.default_rng(seed)
    sel = np.full((B, k), -1, np.int32)
    for b in range(B):
        take = min(k, n_vis[b])
        sel[b, :take] = np.sort(g.choice(n_vis[b], take, replace=False))
    return sel


@pytest.mark.parametrize("H", [16, 64])
@pytest.mark.parametrize("with_sink", [True, False])
def test_fp8kv_sparse_decode_parity(cuda_device, H, with_sink):
    B, N_cap, k, W = 3, 300, 48, 128
    lens = [700, 129, 37]
    n_vis = [min(N_cap, n // 4) for n in lens]
    (kn, ks, kr, v, vs), K, V = _kv8(B, N_cap, n_vis, 31)
    q = synth.randn((B, 1, H, 128), 31, 1, scale=1 / math.sqrt(128))
    kw, vw = synth.randn((B, W, 128), 31, 4), synth.randn((B, W, 128), 31, 5)
    sink = synth.randn((H,), 31, 6, dtype=torch.float32) if with_sink else None
    sel = _random_topk(B, k, n_vis)
    q_pos = torch.tensor(lens, dtype=torch.int32).view(B, 1) - 1
    out, lse = csa.attn_fp8kv(
        q.to(DEV), kn, ks, kr, v, vs, torch.from_numpy(sel).view(B, 1, k).to(DEV),
        place_window(kw, lens, 800), place_window(vw, lens, 800), q_pos.to(DEV), W,
        None if sink is None else sink.to(DEV), return_lse=True)
    torch.cuda.synchronize()
    rkw, base = window_arrays(kw, lens)
    rvw, _ = window_arrays(vw, lens)
    ro, rl = oracle.csa_decode(u16(q[:, 0]), K, V, sel, rkw, rvw, np.array(lens), W,
                               None if sink is None else sink.numpy(), 1.0, base)
    check_attention(out[:, 0], ro, lse[:, 0], rl, f"fp8kv csa decode H={H}",
                    lse_tol(q, K, n_vis)[:, 0])


@pytest.mark.parametrize("ws", [None, False])
def test_fp8kv_many_splits(cuda_device, ws):
    # 40 queries x 640 keys (8 splits), and one query with 3000 entries (free
    # splits merged by the second kernel when a workspace is given)
    B, H, N_cap, k, W = 40, 64, 900, 512, 128
    lens = [3600 - 37 * b for b in range(B)]
    n_vis = [min(N_cap, n // 4) for n in lens]
    (kn, ks, kr, v, vs), K, V = _kv8(B, N_cap, n_vis, 32)
    q = synth.randn((B, 1, H, 128), 32, 1, scale=1 / math.sqrt(128))
    kw, vw = synth.randn((B, W, 128), 32, 4), synth.randn((B, W, 128), 32, 5)
    sink = synth.randn((H,), 32, 6, dtype=torch.float32)
    sel = _random_topk(B, k, n_vis, seed=8)
    q_pos = torch.tensor(lens, dtype=torch.int32).view(B, 1) - 1
    out, lse = csa.attn_fp8kv(
        q.to(DEV), kn, ks, kr, v, vs, torch.from_numpy(sel).view(B, 1, k).to(DEV),
        place_window(kw, lens, 3600), place_window(vw, lens, 3600), q_pos.to(DEV), W,
        sink.to(DEV), return_lse=True, ws=ws)
    torch.cuda.synchronize()
    rkw, base = window_arrays(kw, lens)
    rvw, _ = window_arrays(vw, lens)
    ro, rl = oracle.csa_decode(u16(q[:, 0]), K, V, sel, rkw, rvw, np.array(lens), W,
                               sink.numpy(), 1.0, base)
    check_attention(out[:, 0], ro, lse[:, 0], rl, f"fp8kv splits ws={ws}",
                    lse_tol(q, K, n_vis)[:, 0])
    lens1 = [16004]
    (kn1, ks1, kr1, v1, vs1), K1, V1 = _kv8(1, 4001, [4001], 33)
    q1 = synth.randn((1, 1, H, 128), 33, 1, scale=1 / math.sqrt(128))
    kw1, vw1 = synth.randn((1, W, 128), 33, 4), synth.randn((1, W, 128), 33, 5)
    sel1 = _random_topk(1, 3000, [4001], seed=9)
    out1, lse1 = csa.attn_fp8kv(
        q1.to(DEV), kn1, ks1, kr1, v1, vs1, torch.from_numpy(sel1).view(1, 1, 3000).to(DEV),
        place_window(kw1, lens1, 16004), place_window(vw1, lens1, 16004),
        torch.tensor([[16003]], dtype=torch.int32, device=DEV), W, sink.to(DEV),
        return_lse=True, ws=ws)
    torch.cuda.synchronize()
    rkw1, base1 = window_arrays(kw1, lens1)
    rvw1, _ = window_arrays(vw1, lens1)
    ro1, rl1 = oracle.csa_decode(u16(q1[:, 0]), K1, V1, sel1, rkw1, rvw1, np.array(lens1), W,
                                 sink.numpy(), 1.0, base1)
    check_attention(out1[:, 0], ro1, lse1[:, 0], rl1, f"fp8kv 3000 entries ws={ws}",
                    lse_tol(q1, K1, [4001])[:, 0])


@pytest.mark.parametrize("window,ws", [(128, None), (128, False), (0, None)])
def test_fp8kv_hca_parity(cuda_device, window, ws):
    # dense HCA over FP8 entries (contiguous stages go by bulk copies); a
    # sequence with no visible entries; long key ranges (25 tiles) for the
    # split modes
    B, H, m = 4, 64, 8
    lens = [24000, 517, 64, 5]
    N_cap = 3000
    n_cmp = [3000, 64, 8, 0]
    n_vis = [min(n_cmp[b], lens[b] // m) for b in range(B)]
    (kn, ks, kr, v, vs), K, V = _kv8(B, N_cap, n_vis, 34)
    q = synth.randn((B, 1, H, 128), 34, 1, scale=1 / math.sqrt(128))
    kw, vw = synth.randn((B, 128, 128), 34, 4), synth.randn((B, 128, 128), 34, 5)
    sink = synth.randn((H,), 34, 6, dtype=torch.float32)
    q_pos = torch.tensor(lens, dtype=torch.int32).view(B, 1) - 1
    out, lse = csa.attn_fp8kv(
        q.to(DEV), kn, ks, kr, v, vs, None,
        place_window(kw, lens, 24000) if window else None,
        place_window(vw, lens, 24000) if window else None, q_pos.to(DEV), window, sink.to(DEV),
        n_cmp=torch.tensor(n_cmp, dtype=torch.int32, device=DEV), m_prime=m, return_lse=True,
        ws=ws)
    torch.cuda.synchronize()
    rkw, base = window_arrays(kw, lens)
    rvw, _ = window_arrays(vw, lens)
    ro, rl = oracle.hca_decode(u16(q[:, 0]), K, V, np.array(n_cmp), m,
                               rkw if window else None, rvw if window else None, np.array(lens),
                               window, sink.numpy(), 1.0, base)
    check_attention(out[:, 0], ro, lse[:, 0], rl, f"fp8kv hca window={window} ws={ws}",
                    lse_tol(q, K, n_vis)[:, 0])
    if window == 0:  # sequence 3 sees nothing: output 0, lse = sink
        assert torch.all(out[3] == 0)
        np.testing.assert_allclose(lse[3, 0].cpu().numpy(), sink.numpy(), rtol=1e-6)


def test_fp8kv_prefill_parity(cuda_device):
    # T query tokens per sequence with block-causal top-k rows and a causal
    # window over the raw rows of the chunk
    B, T, H, N_cap, k, W, m = 2, 37, 64, 140, 48, 128, 4
    q_pos = np.array([[500 + t for t in range(T)], [100 + 3 * t for t in range(T)]], np.int32)
    L_cap = 700
    n_vis = [N_cap, N_cap]
    (kn, ks, kr, v, vs), K, V = _kv8(B, N_cap, n_vis, 35)
    q = synth.randn((B, T, H, 128), 35, 1, scale=1 / math.sqrt(128))
    rk, rv = synth.randn((B, L_cap, 128), 35, 4), synth.randn((B, L_cap, 128), 35, 5)
    sink = synth.randn((H,), 35, 6, dtype=torch.float32)
    g = np.random.default_rng(4)
    sel = np.full((B, T, k), -1, np.int32)
    for b in range(B):
        for t in range(T):
            nv = min(N_cap, (q_pos[b, t] + 1) // m)
            take = min(k, nv)
            sel[b, t, :take] = np.sort(g.choice(nv, take, replace=False))
    out, lse = csa.attn_fp8kv(
        q.to(DEV), kn, ks, kr, v, vs, torch.from_numpy(sel).to(DEV), rk.to(DEV), rv.to(DEV),
        torch.from_numpy(q_pos).to(DEV), W, sink.to(DEV), return_lse=True)
    torch.cuda.synchronize()
    ro, rl = oracle.csa_prefill(u16(q), K, V, sel, u16(rk), u16(rv), q_pos, W, sink.numpy(), 1.0)
    check_attention(out, ro, lse, rl, "fp8kv prefill", lse_tol(q, K, n_vis))


def test_fp8kv_rejects(cuda_device):
    B, N_cap = 1, 64
    (kn, ks, kr, v, vs), _, _ = _kv8(B, N_cap, [N_cap], 36)
    q = torch.zeros((B, 1, 128, 128), dtype=torch.bfloat16, device=DEV)  # H = 128 > 64
    sel = torch.zeros((B, 1, 8), dtype=torch.int32, device=DEV)
    qp = torch.full((B, 1), 300, dtype=torch.int32, device=DEV)
    with pytest.raises(csa.CsaError) as e:
        csa.attn_fp8kv(q, kn, ks, kr, v, vs, sel, None, None, qp, 0, None)
    assert e.value.status == 2  # CSA_ERR_UNSUPPORTED
