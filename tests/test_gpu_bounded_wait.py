"""The bounded-wait path of the pipelined kernels, made to run out on the GPU
without faulting or hanging it: csa_selftest_bounded_wait waits on an
mbarrier that nobody completes, with a short iteration limit, through the
same wait helper and error flag the kernels use.  The call must return, the
flag must be set, and the library must work normally afterwards in the same
process (an attention call checked against the oracle)."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_28_b300 as csa
import synth
from _util import check_attention, u16, window_arrays, place_window

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_bounded_wait_gives_up_and_flags(cuda_device):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa.selftest_bounded_wait(err, arrive=False, limit=200)
    torch.cuda.synchronize()
    assert int(err.item()) == csa.EW_TIMEOUT
    # the flag is ORed: other bits survive
    err.fill_(csa.EW_BAD_INDEX)
    csa.selftest_bounded_wait(err, arrive=False, limit=1)
    torch.cuda.synchronize()
    assert int(err.item()) == csa.EW_BAD_INDEX | csa.EW_TIMEOUT


def test_bounded_wait_that_completes_leaves_the_word(cuda_device):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa.selftest_bounded_wait(err, arrive=True, limit=200)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


def test_library_works_after_a_timed_out_wait(cuda_device):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa.selftest_bounded_wait(err, arrive=False, limit=100)
    # a sparse decode right behind it on the same stream
    B, H, N_cap, k, W = 2, 64, 600, 200, 128
    lens = [2400, 1700]
    q = synth.randn((B, H, 128), 41, 1, scale=128 ** -0.5)
    kc = synth.randn((B, N_cap, 128), 41, 2)
    vc = synth.randn((B, N_cap, 128), 41, 3)
    kw = synth.randn((B, W, 128), 41, 4)
    vw = synth.randn((B, W, 128), 41, 5)
    sink = synth.randn((H,), 41, 6, dtype=torch.float32)
    g = torch.Generator().manual_seed(41)
    idx = torch.stack([torch.sort(torch.randperm(min(N_cap, n // 4), generator=g)[:k])[0]
                       for n in lens]).to(torch.int32)
    L_cap = max(lens)
    err2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, lse = csa.sparse_attn_decode(q.to(DEV), kc.to(DEV), vc.to(DEV), idx.to(DEV),
                                      place_window(kw, lens, L_cap), place_window(vw, lens, L_cap),
                                      torch.tensor(lens, dtype=torch.int32, device=DEV), W,
                                      sink.to(DEV), return_lse=True, err_word=err2)
    torch.cuda.synchronize()
    assert int(err.item()) == csa.EW_TIMEOUT
    assert int(err2.item()) == 0
    kwa, base = window_arrays(kw, lens)
    vwa, _ = window_arrays(vw, lens)
    ro, rl = oracle.csa_decode(u16(q), u16(kc), u16(vc), idx.numpy(), kwa, vwa,
                               np.array(lens), W, sink.numpy(), 1.0, base)
    check_attention(out, ro, lse, rl, "decode after a timed-out wait")
