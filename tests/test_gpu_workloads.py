"""The five workloads at full size, in the launch configuration the benchmark
times (one step object per workload), checked against the CPU oracle on
sampled queries: sequences for decode, new tokens for prefill."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_28_b300 as csa
import synth
from _util import (bf16_bound, check_attention, check_e4m3_rows, check_fp4_rows, check_topk, f64,
                   lse_tol, u8, u16)
from oracle.feed import fill_new_entries, idx_dtype, oracle_inputs
from sparse_attention_28_b300.steps import make_step

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(name):
    wl = synth.WORKLOADS[name]
    inp = synth.make_inputs(wl, seed=0, device=DEV)
    step = make_step(inp, DEV)
    out = step().clone()
    torch.cuda.synchronize()
    return wl, inp, step, out


def _check_bf16_entries(gpu, y, what):
    g = f64(gpu)
    assert np.all(np.abs(g - y) <= bf16_bound(y)), f"{what}: beyond 1 bf16 ulp + fp32 error"


def _check_decode(name, seqs):
    wl, inp, step, out = _run(name)
    a = oracle_inputs(wl, inp, 0, seqs=seqs)
    if wl.stream_compress:
        y = fill_new_entries(wl, inp, a)
        j = wl.N_cap - 1
        ix = torch.tensor(seqs, device=DEV)
        _check_bf16_entries(step.k_cmp[ix, j], y["k"][:, 0], "compressed K")
        _check_bf16_entries(step.v_cmp[ix, j], y["v"][:, 0], "compressed V")
        if wl.idx_fp4:
            check_fp4_rows(u8(step.k_idx[ix, j]), u8(step.k_scale[ix, j]), y["idx"][:, 0],
                           "streamed FP4 index key")
        else:
            check_e4m3_rows(u8(step.k_idx[ix, j]), step.k_scale[ix, j].cpu().numpy(),
                            y["idx"][:, 0], "streamed FP8 index key")
    if wl.kind == "hca_decode":
        ro, rl = oracle.hca_decode(a["q"], a["k_cmp"], a["v_cmp"], a["n_cmp"], wl.m, a["k_win"],
                                   a["v_win"], a["seq_len"], wl.W, a["sink"], 1.0, a["raw_base"])
        check_attention(out[seqs], ro, what=name)
        return
    sc, nv = oracle.indexer_scores(a["q_idx"], a["w"], a["k_idx"], a["q_pos"], a["n_cmp"], wl.m,
                                   idx_dtype(wl), a.get("q_scale"), a.get("k_scale"))
    ref = oracle.topk(sc, nv, wl.k)
    gidx = step.idx[seqs].cpu().numpy()
    check_topk(gidx, ref, sc, nv, wl.k, name)
    ro, rl = oracle.csa_decode(a["q"], a["k_cmp"], a["v_cmp"], ref[:, 0], a["k_win"], a["v_win"],
                               a["seq_len"], wl.W, a["sink"], 1.0, a["raw_base"])
    # the same attention call as the step, fed the oracle's top-k
    full_ref = step.idx[:, 0].clone()
    full_ref[seqs] = torch.from_numpy(ref[:, 0]).to(DEV)
    if wl.kv_fp8:
        B, H, D = step.q.shape
        o2, l2 = csa.attn_fp8kv(step.q.view(B, 1, H, D), *step.kv8, full_ref.view(B, 1, -1),
                                step.k_raw, step.v_raw, step.q_pos, wl.W, step.sink,
                                return_lse=True)
        o2, l2 = o2[:, 0], l2[:, 0]
        tol = lse_tol(oracle.bf16_decode(a["q"])[:, None], a["k_cmp"], list(a["n_cmp"]))[:, 0]
    else:
        o2, l2 = csa.sparse_attn_decode(step.q, step.k_cmp, step.v_cmp, full_ref, step.k_raw,
                                        step.v_raw, step.seq_len, wl.W, step.sink,
                                        return_lse=True)
        tol = None
    torch.cuda.synchronize()
    check_attention(o2[seqs], ro, l2[seqs], rl, name + " attention", tol)
    # the step's own output wherever its top-k set is the oracle's
    same = [i for i, b in enumerate(seqs)
            if set(gidx[i, 0].tolist()) == set(ref[i, 0].tolist())]
    assert len(same) >= len(seqs) - 1
    att = getattr(step, "attn_out", out)
    check_attention(att[[seqs[i] for i in same]], ro[same], what=name + " step")
    if wl.proj_groups:
        # the projection of the step's own attention output
        K = (wl.H // wl.proj_groups) * wl.D
        yr = oracle.grouped_out_proj(u16(att[seqs]), a["W_o"])
        mag = np.abs(oracle.grouped_out_proj(u16(att[seqs].abs()), u16(step.W_o.abs())))
        assert np.all(np.abs(f64(out[seqs]) - yr) <= bf16_bound(yr) + K * 2.0 ** -23 * mag)


def test_csa_decode_tiny(cuda_device):
    _check_decode("csa_decode_tiny", [0])


def test_csa_decode_128k(cuda_device):
    _check_decode("csa_decode_128k", [0, 13, 31])


def test_hca_decode_1m(cuda_device):
    _check_decode("hca_decode_1m", [0, 9, 15])


def test_csa_decode_1m_fp8_streaming(cuda_device):
    _check_decode("csa_decode_1m_fp8", [0, 7])


def test_csa_decode_128k_fp8kv(cuda_device):
    _check_decode("csa_decode_128k_fp8kv", [0, 13, 31])


def test_hca_decode_1m_fp8kv(cuda_device):
    _check_decode("hca_decode_1m_fp8kv", [0, 9, 15])


@pytest.mark.parametrize("name", ["csa_prefill_4k", "csa_prefill_4k_overlap"])
def test_csa_prefill_4k(cuda_device, name):
    # the overlap variant forms every new block from 2m raw tokens
    wl, inp, step, out = _run(name)
    toks = [0, 1, 2, 3, 4, 1023, 2048, 4093, 4094, 4095]
    a = oracle_inputs(wl, inp, 0, tokens=toks)
    y = fill_new_entries(wl, inp, a)
    n_old, n_new = wl.L // wl.m, wl.T // wl.m
    _check_bf16_entries(step.k_cmp[:, n_old:n_old + n_new], y["k"], "prefill K entries")
    _check_bf16_entries(step.v_cmp[:, n_old:n_old + n_new], y["v"], "prefill V entries")
    _check_bf16_entries(step.k_idx[:, n_old:n_old + n_new], y["idx"], "prefill index keys")
    sc, nv = oracle.indexer_scores(a["q_idx"], a["w"], a["k_idx"], a["q_pos"], a["n_cmp"], wl.m)
    ref = oracle.topk(sc, nv, wl.k)
    gidx = step.idx[:, toks].cpu().numpy()
    check_topk(gidx, ref, sc, nv, wl.k, "prefill top-k")
    ro, rl = oracle.csa_prefill(a["q"], a["k_cmp"], a["v_cmp"], ref, a["k_raw"], a["v_raw"],
                                a["q_pos"], wl.W, a["sink"], 1.0, a["raw_base"])
    same = [i for i in range(len(toks))
            if set(gidx[0, i].tolist()) == set(ref[0, i].tolist())]
    assert len(same) >= len(toks) - 2
    check_attention(out[:, [toks[i] for i in same]], ro[:, same], what="prefill step")


def test_csa_decode_128k_batch_invariant(cuda_device):
    # the same step with fixed 320-key attention splits
    _check_decode("csa_decode_128k_bi", [0, 13, 31])


def test_csa_decode_1m_fp4_streaming(cuda_device):
    _check_decode("csa_decode_1m_fp4", [0, 7])


def test_csa_decode_128k_with_grouped_out_proj(cuda_device):
    _check_decode("csa_decode_128k_proj", [0, 13, 31])


def test_decode_step_is_deterministic(cuda_device):
    wl, inp, step, out = _run("csa_decode_128k")
    idx = step.idx.clone()
    again = step()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    assert torch.equal(idx, step.idx)
