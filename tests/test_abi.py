"""The C-ABI library on the host (no GPU needed): it loads, exports every
symbol include/csa.h declares, and rejects bad arguments before launching
anything."""
import ctypes
import os
import re

import pytest

import sparse_attention_28_b300 as csa

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "csa.h")
FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: validation fails first


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:csa|hca)_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 9
    L = csa.lib()
    for n in names:
        assert hasattr(L, n), f"libcsa.so does not export {n}"
    assert set(names) == set(csa.ABI_SYMBOLS)


def test_status_strings():
    L = csa.lib()
    for code in range(6):
        assert L.csa_status_str(code).startswith(b"CSA_")
    assert L.csa_status_str(99) == b"unknown status"
    assert L.csa_abi_version() == 1


def _decode(**over):
    args = dict(q=FAKE, k_cmp=FAKE, v_cmp=FAKE, cmp_bstride=1024 * 128, N_cap=1024,
                topk_idx=FAKE, k=64, k_raw=FAKE, v_raw=FAKE, raw_bstride=4096 * 128,
                raw_cap=4096, seq_len=FAKE, window=128, sink=None, scale=1.0, B=2, H=64, D=128,
                out=FAKE, lse=None, ws=FAKE, ws_bytes=1, err=None, stream=None)
    args.update(over)
    return csa.lib().csa_sparse_attn_decode(*args.values())


@pytest.mark.parametrize("over,status", [
    (dict(q=None), 1), (dict(out=None), 1), (dict(D=64), 2), (dict(H=48), 2), (dict(B=-1), 1),
    (dict(window=-1), 1), (dict(cmp_bstride=1000), 1), (dict(k_raw=None), 1),
    (dict(raw_bstride=100), 1), (dict(raw_cap=100), 1), (dict(q=ctypes.c_void_p(0x10002)), 1), (dict(k=-3), 1),
    (dict(topk_idx=None), 1), (dict(seq_len=None), 1),
])
def test_sparse_decode_rejects(over, status):
    assert _decode(**over) == status


def test_zero_batch_is_a_no_op():
    assert _decode(B=0, q=None, out=None) == 0


def test_indexer_rejects():
    L = csa.lib()

    def call(**over):
        a = dict(q=FAKE, qs=None, w=FAKE, kk=FAKE, kbs=4096 * 64, ks=None, ksbs=0, dt=0,
                 pos=FAKE, ncmp=FAKE, B=2, T=1, HI=4, dI=64, N=4096, m=4, k=256, idx=FAKE,
                 sc=None, ws=FAKE, wsb=1, err=None, st=None)
        a.update(over)
        return L.csa_indexer_topk(*a.values())

    assert call(HI=8) == 2 and call(dI=128) == 2 and call(dt=7) == 2
    assert call(k=5000) == 1 and call(k=0) == 1 and call(q=None) == 1
    assert call(dt=1) == 1  # FP8 without scales
    assert call(kbs=100) == 1
    assert call(N=1 << 20) == 2
    assert call() == 3  # workspace too small
    assert L.csa_indexer_topk_workspace(2, 1, 4096, 256) >= 2 * 4096 * 4  # one fp32 score per entry


def test_indexer_scores_rejects():
    L = csa.lib()

    def call(**over):
        a = dict(q=FAKE, qs=None, w=FAKE, kk=FAKE, kbs=4096 * 64, ks=None, ksbs=0, dt=0,
                 pos=FAKE, ncmp=FAKE, B=2, T=1, HI=4, dI=64, N=4096, m=4, sc=FAKE, ld=4096,
                 err=None, st=None)
        a.update(over)
        return L.csa_indexer_scores(*a.values())

    assert call(HI=8) == 2 and call(dt=7) == 2 and call(N=1 << 20) == 2
    assert call(sc=None) == 1 and call(ld=4095) == 1 and call(m=0) == 1
    assert call(dt=1) == 1  # FP8 without scales
    assert call(B=0, q=None, sc=None) == 0  # nothing to do


def test_compress_rejects():
    L = csa.lib()

    def call(**over):
        a = dict(raw=FAKE, rbs=64 * 128, rcap=64, B=2, d=128, m=4, b0=0, nb=16, W=FAKE, pb=FAKE,
                 out=FAKE, obs=16 * 128, dt=0, sc=None, sbs=0, err=None, st=None)
        a.update(over)
        return L.csa_compress_kv(*a.values())

    assert call(d=96) == 2 and call(m=300) == 2 and call(dt=5) == 2
    assert call(rcap=3) == 1  # a ring shorter than one block
    assert call(rcap=65) == 1  # ring rows beyond the sequence stride
    assert call(obs=15 * 128) == 1
    assert call(dt=1) == 1  # FP8 output needs a scale array
    assert call(W=None) == 1
    assert call(B=0) == 0 and call(nb=0) == 0


def test_compress_span_rejects():
    L = csa.lib()

    def call(**over):
        a = dict(raw=FAKE, rbs=64 * 128, rcap=64, B=2, d=128, m=4, span=8, b0=0, nb=16, W=FAKE,
                 pb=FAKE, out=FAKE, obs=16 * 128, dt=0, sc=None, sbs=0, err=None, st=None)
        a.update(over)
        return L.csa_compress_kv_span(*a.values())

    assert call(span=3) == 1          # shorter than the stride
    assert call(span=257) == 2        # more rows than the kernel stages
    assert call(rcap=7) == 1          # the ring must hold the whole span
    assert call(B=0, raw=None) == 0


def test_batch_invariant_rejects():
    L = csa.lib()

    def call(**over):
        a = dict(q=FAKE, kc=FAKE, vc=FAKE, cbs=1024 * 128, N=1024, idx=FAKE, k=512, kr=FAKE,
                 vr=FAKE, rbs=4096 * 128, rcap=4096, pos=FAKE, W=128, sink=None, scale=1.0, B=2,
                 T=2, H=64, D=128, out=FAKE, lse=None, kps=256, err=None, st=None)
        a.update(over)
        return L.csa_sparse_attn_batch_invariant(*a.values())

    assert call(kps=0) == 1
    assert call(kps=32, k=1024) == 1   # 1155 slots in ranges of 64: 19 splits (> 16)
    assert call(kps=64, k=1000) == 1   # 1131 slots: 18 splits
    assert call(pos=None) == 1
    assert call(B=0, q=None) == 0


def test_grouped_out_proj_rejects():
    L = csa.lib()

    def call(**over):
        a = dict(o=FAKE, W=FAKE, y=FAKE, n=32, H=64, D=128, G=8, d_g=512, err=None, st=None)
        a.update(over)
        return L.csa_grouped_out_proj(*a.values())

    assert call(G=7) == 1           # heads do not split into 7 groups
    assert call(d_g=100) == 2       # output channels per group: a multiple of 128
    assert call(D=40, G=64) == 2    # K = 40: not a multiple of 64
    assert call(y=None) == 1
    assert call(n=0, o=None) == 0


def test_attention_workspace_only_for_split_queries():
    # partial rows + lse (129 fp32 per head) for every split of every query
    # when a query can get several splits (fewer queries than SMs / 2); none
    # when each query gets one split
    L = csa.lib()

    def ws(n_query, ns, H):
        b = n_query * ns * H * 129 * 4
        return (b + 255) // 256 * 256

    assert L.csa_attn_workspace(32, 1, 64, 1152) == ws(32, 4, 64)     # 148 // 32 splits
    assert L.csa_attn_workspace(16, 1, 64, 8320) == ws(16, 9, 64)
    assert L.csa_attn_workspace(8, 1, 128, 2176) == ws(8, 18, 128)    # 18 tiles of keys
    assert L.csa_attn_workspace(1, 4096, 64, 2176) == 0                # one split per query
    assert L.csa_attn_workspace(100, 1, 64, 1152) == 0


def test_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(2, 64, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        csa.sparse_attn_decode(q, q, q, torch.zeros(2, 4, dtype=torch.int32), q, q,
                               torch.zeros(2, dtype=torch.int32), 128, None)


def test_static_indexer_refuses_beyond_its_scratch():
    # 256 queries over 2^19 entries need far more than the fixed scratch; the
    # refusal comes before any CUDA call, so it needs no GPU
    L = csa.lib()
    need = L.csa_indexer_topk_workspace(256, 1, 1 << 19, 64)
    assert need > csa.INDEXER_STATIC_SCRATCH_BYTES
    assert L.csa_indexer_topk_workspace(32, 1, 32768, 1024) <= csa.INDEXER_STATIC_SCRATCH_BYTES
    st = L.csa_indexer_topk_static(FAKE, None, FAKE, FAKE, (1 << 19) * 64, None, 0, 0, FAKE, FAKE,
                                   256, 1, 4, 64, 1 << 19, 4, 64, FAKE, None, None, None)
    assert st == 3


def _static(**over):
    a = dict(q=FAKE, qs=None, w=FAKE, kk=FAKE, kbs=16416 * 64, ks=None, ksbs=0, dt=0, pos=FAKE,
             ncmp=FAKE, B=256, T=1, HI=4, dI=64, N=16385, m=4, k=64, idx=FAKE, sc=None, err=None,
             st=None)
    a.update(over)
    return csa.lib().csa_indexer_topk_static(*a.values())


def test_static_indexer_capacity_boundary():
    # any number of queries over 16384 entries fits exactly (the scores are
    # taken 256 queries at a time); one entry more (rows rounded up to 32
    # entries) no longer does
    L = csa.lib()
    cap = csa.INDEXER_STATIC_SCRATCH_BYTES
    assert L.csa_indexer_topk_workspace(256, 1, 16384, 64) == cap
    assert L.csa_indexer_topk_workspace(8, 1, 1 << 19, 64) == cap
    assert L.csa_indexer_topk_workspace(256, 1, 16385, 64) > cap
    assert L.csa_indexer_topk_workspace(9, 1, 1 << 19, 64) > cap
    assert _static() == 3
    assert _static(B=9, N=1 << 19, kbs=(1 << 19) * 64) == 3


def test_static_indexer_gives_the_workspace_entrys_statuses():
    # a call that is both oversized and invalid reports what csa_indexer_topk
    # reports for the invalid argument, not the capacity
    assert _static(k=0) == 1
    assert _static(q=None) == 1
    assert _static(idx=None) == 1
    assert _static(HI=8) == 2
    assert _static(dt=7) == 2
    assert _static(N=(1 << 19) + 1, kbs=((1 << 19) + 32) * 64) == 2
    assert _static(B=0) == 0  # nothing to do, no CUDA call


def test_selftest_bounded_wait_rejects():
    L = csa.lib()
    assert L.csa_selftest_bounded_wait(0, 100, None, None) == 1
    assert L.csa_selftest_bounded_wait(0, 100, ctypes.c_void_p(0x10002), None) == 1
    assert L.csa_selftest_bounded_wait(0, 0, FAKE, None) == 1
    assert L.csa_selftest_bounded_wait(0, (1 << 20) + 1, FAKE, None) == 1


def test_probe_rejects():
    # invalid arguments are refused on the host, before any CUDA call
    L = csa.lib()
    odd = ctypes.c_void_p(0x10008)  # not 16-byte aligned
    assert L.csa_probe_stream_read(None, 1 << 20, 2, 4, FAKE, None) == 1
    assert L.csa_probe_stream_read(FAKE, 1 << 20, 2, 4, None, None) == 1
    assert L.csa_probe_stream_read(odd, 1 << 20, 2, 4, FAKE, None) == 1
    assert L.csa_probe_stream_read(FAKE, 0, 2, 4, FAKE, None) == 1
    assert L.csa_probe_stream_read(FAKE, 1 << 20, 0, 4, FAKE, None) == 1
    assert L.csa_probe_stream_read(FAKE, 1 << 20, 5, 4, FAKE, None) == 1
    assert L.csa_probe_stream_read(FAKE, 1 << 20, 2, 3, FAKE, None) == 1
    assert L.csa_probe_stream_read(FAKE, 16, 2, 4, FAKE, None) == 1  # under one vector per CTA
    assert L.csa_probe_row_gather(None, 100, FAKE, 1, 1, 2, 0, FAKE, None) == 1
    assert L.csa_probe_row_gather(FAKE, 100, None, 1, 1, 2, 0, FAKE, None) == 1
    assert L.csa_probe_row_gather(FAKE, 100, FAKE, 1, 1, 2, 0, None, None) == 1
    assert L.csa_probe_row_gather(odd, 100, FAKE, 1, 1, 2, 0, FAKE, None) == 1
    assert L.csa_probe_row_gather(FAKE, 0, FAKE, 1, 1, 2, 0, FAKE, None) == 1
    assert L.csa_probe_row_gather(FAKE, 100, FAKE, 0, 1, 2, 0, FAKE, None) == 1
    assert L.csa_probe_row_gather(FAKE, 100, FAKE, 1, 0, 2, 0, FAKE, None) == 1
    assert L.csa_probe_row_gather(FAKE, 100, FAKE, 1, 65, 2, 0, FAKE, None) == 1  # index list cap
    assert L.csa_probe_row_gather(FAKE, 100, FAKE, 1, 1, 3, 0, FAKE, None) == 1
    assert L.csa_probe_row_gather(FAKE, 100, FAKE, 1, 1, 2, 5, FAKE, None) == 1
    assert L.csa_probe_row_gather(FAKE, 100, FAKE, 1, 1, 2, -1, FAKE, None) == 1
    assert L.csa_probe_row_gather(FAKE, 1 << 31, FAKE, 1, 1, 2, 1, FAKE, None) == 1


def test_compress_mixed_rejects():
    L = csa.lib()

    def call(**over):
        a = dict(raw=FAKE, rbs=64 * 128, rcap=64, B=2, d=128, m=4, span=4, b0=0, nb=16, W=FAKE,
                 pb=FAKE, codes=FAKE, cbs=16 * 64, sc=FAKE, sbs=16, rope=FAKE, ropebs=16 * 64,
                 n_rope=64, err=None, st=None)
        a.update(over)
        return L.csa_compress_kv_mixed(*a.values())

    assert call(n_rope=0) == 1 and call(n_rope=128) == 1
    assert call(n_rope=60) == 1       # RoPE channels in whole 16-byte bf16 chunks
    assert call(n_rope=56) == 1       # E4M3 part in whole 16-byte chunks
    assert call(d=96) == 2
    assert call(cbs=15 * 64) == 1     # codes rows beyond the sequence stride
    assert call(ropebs=15 * 64) == 1
    assert call(sbs=15) == 1
    assert call(sc=None) == 1 and call(rope=None) == 1
    assert call(B=0, raw=None) == 0


def test_attn_fp8kv_rejects():
    L = csa.lib()

    def call(**over):
        a = dict(q=FAKE, kn=FAKE, ks=FAKE, kr=FAKE, v=FAKE, vs=FAKE, N=1024, idx=FAKE, k=512,
                 nc=None, mp=1, kraw=FAKE, vraw=FAKE, rbs=4096 * 128, rcap=4096, pos=FAKE, W=128,
                 sink=None, scale=1.0, B=2, T=1, H=64, D=128, out=FAKE, lse=None, ws=None,
                 wsb=0, err=None, st=None)
        a.update(over)
        return L.csa_attn_fp8kv(*a.values())

    assert call(H=128) == 2                # FP8 entries: at most 64 heads
    assert call(D=64) == 2
    assert call(pos=None) == 1
    assert call(ks=None) == 1 and call(vs=None) == 1 and call(kr=None) == 1
    assert call(idx=None) == 1             # HCA needs n_cmp
    assert call(idx=None, nc=FAKE, mp=0) == 1
    assert call(k=0) == 1
    assert call(B=0, q=None) == 0
