"""The feed probes behind `bench.py --probe` run and read what they are given:
over all-zero data the XOR of everything read is 0, so the sink (written only
for one fixed nonzero value) stays untouched; over a buffer whose XOR is that
value, it is written.  Small sizes, one launch each."""
import pytest
import torch

import sparse_attention_28_b300 as csa

DEV = "cuda:0"


@pytest.mark.gpu
def test_probe_stream_read_reads_every_vector(cuda_device):
    n = 148 * 2 * 512 * 16 * 4  # four vectors per thread
    src = torch.zeros(n, dtype=torch.uint8, device=DEV)
    sink = torch.zeros(1, dtype=torch.float32, device=DEV)
    csa.probe_stream_read(src, sink, ctas_per_sm=2, in_flight=4)
    torch.cuda.synchronize()
    assert sink.item() == 0.0
    # one 32-bit word of the last vector of the last CTA carries the constant
    src.view(torch.int32)[-1] = torch.tensor(0x9E3779B9 - (1 << 32), dtype=torch.int32)
    csa.probe_stream_read(src, sink, ctas_per_sm=2, in_flight=4)
    torch.cuda.synchronize()
    assert sink.item() == 1.0


@pytest.mark.gpu
@pytest.mark.parametrize("tma,wide,issuers", [(False, False, 0), (False, True, 0), (True, False, 1),
                                              (True, True, 4), (True, False, 8)])
@pytest.mark.parametrize("ring", [2, 4, 6])
def test_probe_row_gather_reads_the_indexed_rows(cuda_device, ring, tma, wide, issuers):
    n_rows, ctas, stages = 1000, 3, 5
    table = torch.zeros((n_rows, 512), dtype=torch.uint8, device=DEV)
    idx = torch.randint(0, n_rows - 1, (ctas * stages * 64,), dtype=torch.int32, device=DEV)
    sink = torch.zeros(1, dtype=torch.float32, device=DEV)
    csa.probe_row_gather(table, idx, ctas, stages, ring, sink, tma, wide, issuers)
    torch.cuda.synchronize()
    assert sink.item() == 0.0
    # row n_rows-1 is read once (by CTA 1's first stage); it holds the constant
    idx[64 * stages] = n_rows - 1
    table[n_rows - 1, :4] = torch.tensor([0xB9, 0x79, 0x37, 0x9E], dtype=torch.uint8)
    csa.probe_row_gather(table, idx, ctas, stages, ring, sink, tma, wide, issuers)
    torch.cuda.synchronize()
    assert sink.item() == 1.0
