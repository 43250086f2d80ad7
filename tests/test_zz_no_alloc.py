"""csa_indexer_topk_static: the indexer top-k call for callers that cannot
allocate device memory during a call (its scratch is a fixed array inside the
library).  Checked three ways on the GPU, each on two calls in a row:
  * against csa_indexer_topk (caller workspace) on the same inputs -- both
    run the same kernels, so indices and scores agree exactly, and the second
    problem shows the shared scratch carries nothing from one call into the
    next;
  * against the oracle's exact top-k (check_topk's near-tie rule);
  * that the call allocates nothing: with every output preallocated, neither
    the device's free memory nor torch's allocated bytes move across it.
One case needs exactly the scratch's capacity (8 queries over 524288
entries).  The file sorts last so that it also runs after every other GPU
test in one process; it passes alone as well."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_28_b300 as csa
import synth
from _util import check_topk, u8, u16

DEV = "cuda:0"


def _case(B, T, N_cap, m, fp8, seed):
    if fp8:
        qi, qs = synth.randn_fp8_rows((B, T, 4, 64), seed, 1)
        ki, ks = synth.randn_fp8_rows((B, N_cap, 64), seed, 2)
    else:
        qi, qs = synth.randn((B, T, 4, 64), seed, 1), None
        ki, ks = synth.randn((B, N_cap, 64), seed, 2), None
    w = synth.randn((B, T, 4), seed, 3, dtype=torch.float32)
    g = torch.Generator().manual_seed(seed)
    n_cmp = torch.randint(N_cap // 2, N_cap + 1, (B,), generator=g, dtype=torch.int32)
    n_cmp[0] = N_cap
    q_pos = ((n_cmp * m - 1).view(B, 1) - torch.arange(T - 1, -1, -1, dtype=torch.int32) * 3)
    host = dict(q_idx=qi, w=w, k_idx=ki, q_pos=q_pos.to(torch.int32).contiguous(), n_cmp=n_cmp,
                q_scale=qs, k_scale=ks)
    mv = lambda t: None if t is None else t.to(DEV)
    dev = {n: mv(t) for n, t in host.items()}
    dev["m"] = m
    return host, dev


def _oracle_topk(host, m, k, fp8, seqs):
    conv = u8 if fp8 else u16
    pick = lambda t: None if t is None else t[seqs].numpy()
    s, nv = oracle.indexer_scores(conv(host["q_idx"][seqs]), pick(host["w"]),
                                  conv(host["k_idx"][seqs]), pick(host["q_pos"]),
                                  pick(host["n_cmp"]), m,
                                  oracle.FP8_E4M3 if fp8 else oracle.BF16, pick(host["q_scale"]),
                                  pick(host["k_scale"]))
    return oracle.topk(s, nv, k), s, nv


def _run_pair(dev, k):
    """Static entry (preallocated outputs) and the workspace entry."""
    B, T = dev["q_idx"].shape[:2]
    idx_s = torch.empty((B, T, k), dtype=torch.int32, device=DEV)
    sc_s = torch.empty((B, T, k), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa.indexer_topk_static(**dev, k=k, return_scores=True, out=idx_s, scores_out=sc_s,
                            err_word=err)
    idx_w, sc_w = csa.indexer_topk(**dev, k=k, return_scores=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(idx_s.cpu().numpy(), idx_w.cpu().numpy())
    np.testing.assert_array_equal(sc_s.cpu().numpy(), sc_w.cpu().numpy())
    return idx_s.cpu().numpy()


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_and_oracle_twice(cuda_device):
    cases = [
        (_case(32, 1, 32768, 4, False, 11), 1024, False, [0, 17, 31]),  # 32 queries x 32768
        (_case(4, 3, 20000, 4, True, 12), 512, True, [0, 1, 2, 3]),     # FP8, 3 tokens each
    ]
    for (host, dev), k, fp8, seqs in cases:
        B, T, N_cap = dev["q_idx"].shape[0], dev["q_idx"].shape[1], dev["k_idx"].shape[1]
        assert csa.indexer_topk_workspace(B, T, N_cap, k) <= csa.INDEXER_STATIC_SCRATCH_BYTES
        idx = _run_pair(dev, k)
        ref, s, nv = _oracle_topk(host, dev["m"], k, fp8, seqs)
        check_topk(idx[seqs], ref, s, nv, k, "static-scratch top-k")


@pytest.mark.gpu
def test_static_scratch_at_exact_capacity(cuda_device):
    # 8 queries over 524288 entries: exactly CSA_INDEXER_STATIC_SCRATCH_BYTES
    host, dev = _case(8, 1, 524288, 4, False, 14)
    assert csa.indexer_topk_workspace(8, 1, 524288, 2048) == csa.INDEXER_STATIC_SCRATCH_BYTES
    for _ in range(2):
        idx = _run_pair(dev, 2048)
    ref, s, nv = _oracle_topk(host, 4, 2048, False, [0, 5])
    check_topk(idx[[0, 5]], ref, s, nv, 2048, "static-scratch top-k at capacity")


@pytest.mark.gpu
def test_static_scratch_call_allocates_nothing(cuda_device):
    _, dev = _case(16, 1, 65536, 4, False, 15)
    k = 2048
    idx = torch.empty((16, 1, k), dtype=torch.int32, device=DEV)
    sc = torch.empty((16, 1, k), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def call():
        csa.indexer_topk_static(**dev, k=k, return_scores=True, out=idx, scores_out=sc,
                                err_word=err)

    call()  # first call: kernels loaded, the array's address looked up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.memory_reserved() == reserved0
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
    assert int(err.item()) == 0


@pytest.mark.gpu
def test_static_scratch_refuses_oversized_problem(cuda_device):
    # 64 tokens of one sequence over 131072 entries: 32 MiB of scores
    _, dev = _case(1, 64, 131072, 4, False, 13)
    assert csa.indexer_topk_workspace(1, 64, 131072, 64) > csa.INDEXER_STATIC_SCRATCH_BYTES
    with pytest.raises(csa.CsaError) as e:
        csa.indexer_topk_static(**dev, k=64)
    assert e.value.status == 3
