"""csa_indexer_topk_static (library-owned scratch, no device allocation in the
call) against csa_indexer_topk (caller workspace) on the same inputs.  Both
run the same kernels, so indices and scores must agree exactly; two different
problems in a row check that the shared scratch carries nothing from one call
into the next.  The file sorts last so that it also runs after every other
GPU test in one process; it passes alone as well."""
import numpy as np
import pytest
import torch

import sparse_attention_28_b300 as csa
import synth

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
    q_pos = (n_cmp * m - 1).view(B, 1) - torch.arange(T - 1, -1, -1, dtype=torch.int32) * 3
    mv = lambda t: None if t is None else t.to(DEV)
    return dict(q_idx=mv(qi), w=mv(w), k_idx=mv(ki), q_pos=mv(q_pos.to(torch.int32).contiguous()),
                n_cmp=mv(n_cmp), m=m, q_scale=mv(qs), k_scale=mv(ks))


@pytest.mark.gpu
def test_static_scratch_matches_workspace_entry_twice(cuda_device):
    cases = [
        (_case(32, 1, 32768, 4, False, 11), 1024),  # 32 queries over 32768 entries
        (_case(4, 3, 20000, 4, True, 12), 512),     # FP8 keys, several tokens per sequence
    ]
    for inp, k in cases:
        assert csa.indexer_topk_workspace(inp["q_idx"].shape[0], inp["q_idx"].shape[1],
                                          inp["k_idx"].shape[1], k) \
            <= csa.INDEXER_STATIC_SCRATCH_BYTES
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        idx_s, sc_s = csa.indexer_topk_static(**inp, k=k, return_scores=True, err_word=err)
        idx_w, sc_w = csa.indexer_topk(**inp, k=k, return_scores=True)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        np.testing.assert_array_equal(idx_s.cpu().numpy(), idx_w.cpu().numpy())
        np.testing.assert_array_equal(sc_s.cpu().numpy(), sc_w.cpu().numpy())
        # at least one index list is full and ascending
        first = idx_s[0, 0].cpu().numpy()
        assert np.all(first >= 0) and np.all(np.diff(first) > 0)


@pytest.mark.gpu
def test_static_scratch_refuses_oversized_problem(cuda_device):
    # 64 tokens of one sequence over 131072 entries: 32 MiB of scores
    inp = _case(1, 64, 131072, 4, False, 13)
    assert csa.indexer_topk_workspace(1, 64, 131072, 64) > csa.INDEXER_STATIC_SCRATCH_BYTES
    with pytest.raises(csa.CsaError):
        csa.indexer_topk_static(**inp, k=64)
