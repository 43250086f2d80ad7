"""One step of each hot-path workload on resident device buffers.

A step object takes the inputs of a workload (the dict that ``synth``
returns), lays them out on the GPU once -- compressed caches at full
capacity, raw caches as rings of only the rows a step can read (the window;
position p at row p mod R), every row a step must not read filled with NaN so
that a stray read cannot go unnoticed, workspaces and outputs preallocated --
and then runs one step per call:

* CSA decode:  [compress the newest block of K, V and indexer keys]
  -> indexer top-k -> sparse attention (split-K + merge)
* HCA decode:  dense attention (split-K + merge)
* CSA prefill: compress the new blocks -> indexer top-k for every new token
  -> sparse attention for every new token

Each call only launches library kernels on the current stream (no host
synchronisation, no allocation), so a step can be captured in a CUDA graph.
"""
from __future__ import annotations

import torch

from . import (attn_fp8kv, attn_workspace, compress_kv, grouped_out_proj, hca_dense_attn_decode,
               indexer_scores, indexer_topk, indexer_topk_workspace,
               sparse_attn_batch_invariant, sparse_attn_decode, sparse_attn_prefill)

KV8_KEYS = ("kc_nope", "kc_scale", "kc_rope", "vc8", "vc_scale")


def _ring_put(cache, b, positions, rows):
    """Store rows for absolute positions into a ring cache (row = p mod R)."""
    R = cache.shape[1]
    idx = torch.as_tensor(positions, device=cache.device) % R
    cache[b, idx] = rows


def _nan(shape, dtype, device):
    if dtype in (torch.uint8,):
        return torch.full(shape, 0x7F, dtype=dtype, device=device)  # E4M3 NaN code
    return torch.full(shape, float("nan"), dtype=dtype, device=device)


def _overlapped(step, side_fn, main_fns, join_fn):
    """side_fn on a side stream while main_fns run on the current stream;
    join_fn after both.  Stream-ordered, so it can be captured in a graph."""
    cur = torch.cuda.current_stream(step.out.device)
    side = getattr(step, "_side", None)
    if side is None:
        side = step._side = torch.cuda.Stream(device=step.out.device)
    side.wait_stream(cur)
    with torch.cuda.stream(side):
        side_fn()
    for fn in main_fns:
        fn()
    cur.wait_stream(side)
    join_fn()
    return step.out


class _Step:
    """Shared by the step classes: ``stages()`` lists (name, callable) in
    order and ``out`` is the output tensor.  ``inputs`` is one device buffer
    that holds every tensor the host provides anew each step (the queries,
    positions, lengths, indexer queries and weights), so that a serving loop
    uploads a step's inputs with a single copy."""

    INPUTS = ()  # attribute names of the per-step inputs

    def _pack_inputs(self):
        """Re-home the per-step input tensors as views of one device buffer
        (each at a 256-byte aligned offset)."""
        names = [n for n in self.INPUTS if getattr(self, n, None) is not None]
        offs, total = [], 0
        for n in names:
            t = getattr(self, n)
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(max(total, 256), dtype=torch.uint8, device=self.out.device)
        for n, o in zip(names, offs):
            t = getattr(self, n).contiguous()
            nb = t.numel() * t.element_size()
            view = buf[o:o + nb].view(t.dtype).view(t.shape)
            view.copy_(t)
            setattr(self, n, view)
        self.inputs = buf

    def __call__(self):
        for _, fn in self.stages():
            fn()
        return self.out

    def graphed(self, h2d=(), d2h=None):
        """Capture one whole step in a CUDA graph (after an eager warm-up
        call) and return a callable that replays it on the current stream and
        returns ``out``.  The graph reads the step's own device tensors when it
        replays, so new inputs are copied into them first: ``h2d`` lists
        (pinned host tensor, device tensor) pairs copied in at the start of
        the graph and ``d2h`` a pinned host tensor that ``out`` is copied to
        at its end, so that one replay is one submission for the whole
        host -> device -> host round trip."""
        dev = self.out.device
        self()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.graph(graph, stream=side):
            for h, d in h2d:
                d.copy_(h, non_blocking=True)
            self()
            if d2h is not None:
                d2h.copy_(self.out, non_blocking=True)
        torch.cuda.synchronize(dev)

        def replay():
            graph.replay()
            return self.out
        self._graph = graph  # keep the graph alive with the step
        return replay


class CsaDecodeStep(_Step):
    INPUTS = ("q", "q_idx", "w", "q_scale", "seq_len", "q_pos")

    def __init__(self, inp: dict, device="cuda"):
        wl = inp["workload"]
        self.wl = wl
        dev = torch.device(device)
        B, W, m, D = wl.B, wl.W, wl.m, wl.D
        lens = list(wl.lens)
        g = lambda k: None if inp.get(k) is None else inp[k].to(dev).clone()
        self.q, self.sink = g("q"), g("sink")
        self.seq_len, self.n_cmp = g("seq_len"), g("n_cmp")
        self.k_cmp, self.v_cmp = g("k_cmp"), g("v_cmp")
        self.kv8 = tuple(g(k) for k in KV8_KEYS) if wl.kv_fp8 else None
        self.q_idx, self.w, self.k_idx = g("q_idx"), g("w"), g("k_idx")
        self.q_scale, self.k_scale = g("q_scale"), g("k_scale")
        self.q_pos = (self.seq_len - 1).view(B, 1).contiguous()
        # raw caches: rings of W rows holding the window
        self.k_raw = _nan((B, W, D), torch.bfloat16, dev)
        self.v_raw = _nan((B, W, D), torch.bfloat16, dev)
        kw, vw = g("k_win"), g("v_win")
        for b, n in enumerate(lens):
            lo = max(0, n - W)
            _ring_put(self.k_raw, b, range(lo, n), kw[b, W - (n - lo):])
            _ring_put(self.v_raw, b, range(lo, n), vw[b, W - (n - lo):])
        self.compress = wl.stream_compress
        if self.compress:
            self.idx_raw = _nan((B, W, wl.d_I), torch.bfloat16, dev)
            rn = g("raw_new_idx")
            for b, n in enumerate(lens):
                _ring_put(self.idx_raw, b, range(n - m, n), rn[b])
            self.gates = {s: tuple(t.to(dev) for t in inp["gate_" + s]) for s in ("k", "v", "idx")}
            # the newest entry is produced by the step itself
            for b, n in enumerate(lens):
                j = n // m - 1
                self.k_cmp[b, j] = float("nan")
                self.v_cmp[b, j] = float("nan")
                if self.k_scale is not None and self.k_scale.dtype == torch.uint8:
                    self.k_idx[b, j] = 0x77      # FP4 codes 6.0 ...
                    self.k_scale[b, j] = 0x7F    # ... times an E4M3 NaN scale
                elif self.k_scale is not None:
                    self.k_idx[b, j] = 0x7F
                    self.k_scale[b, j] = float("nan")
                else:
                    self.k_idx[b, j] = float("nan")
            assert len(set(lens)) == 1, "streaming compression assumes equal lengths"
            self.new_block = lens[0] // m - 1
        self.idx = torch.empty((B, 1, wl.k), dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.q)
        if wl.proj_groups:
            # the attention output feeds the grouped output projection, whose
            # output is the step's
            self.W_o = g("W_o")
            self.attn_out = self.out
            self.out = torch.empty((B, wl.proj_groups * wl.proj_dim), dtype=torch.bfloat16,
                                   device=dev)
        self.ws_idx = torch.empty(max(1, indexer_topk_workspace(B, 1, wl.N_cap, wl.k)),
                                  dtype=torch.uint8, device=dev)
        self.ws_attn = torch.empty(max(1, attn_workspace(B, 1, wl.H, wl.k + W)),
                                   dtype=torch.uint8, device=dev)
        self._pack_inputs()

    def _compress_kv(self):
        wl, j = self.wl, self.new_block
        compress_kv(self.k_raw, *self.gates["k"], wl.m, j, 1, self.k_cmp)
        compress_kv(self.v_raw, *self.gates["v"], wl.m, j, 1, self.v_cmp)

    def _compress_idx(self):
        wl, j = self.wl, self.new_block
        compress_kv(self.idx_raw, *self.gates["idx"], wl.m, j, 1, self.k_idx, self.k_scale)

    def _compress(self):
        self._compress_kv()
        self._compress_idx()

    def __call__(self):
        if not self.compress:
            return super().__call__()
        # the K/V entries are first needed by the attention: compress them on
        # a side stream while the indexer runs
        return _overlapped(self, self._compress_kv, [self._compress_idx, self._index],
                           self._finish)

    def _finish(self):
        self._attend()
        if self.wl.proj_groups:
            self._project()

    def _index(self):
        wl = self.wl
        indexer_topk(self.q_idx, self.w, self.k_idx, self.q_pos, self.n_cmp, wl.m, wl.k,
                     q_scale=self.q_scale, k_scale=self.k_scale, out=self.idx, ws=self.ws_idx)

    def _attend(self):
        wl = self.wl
        if wl.kv_fp8:
            B, H, D = self.q.shape
            attn_fp8kv(self.q.view(B, 1, H, D), *self.kv8, self.idx, self.k_raw, self.v_raw,
                       self.q_pos, wl.W, self.sink,
                       out=getattr(self, "attn_out", self.out).view(B, 1, H, D), ws=self.ws_attn)
            return
        if wl.batch_invariant:
            # fixed key splits: each sequence's result is independent of the batch
            B, H, D = self.q.shape
            sparse_attn_batch_invariant(self.q.view(B, 1, H, D), self.k_cmp, self.v_cmp, self.idx,
                                        self.k_raw, self.v_raw, self.q_pos, wl.W, self.sink,
                                        keys_per_split=wl.batch_invariant,
                                        out=getattr(self, "attn_out", self.out).view(B, 1, H, D))
            return
        sparse_attn_decode(self.q, self.k_cmp, self.v_cmp, self.idx.view(wl.B, wl.k),
                           self.k_raw, self.v_raw, self.seq_len, wl.W, self.sink,
                           out=getattr(self, "attn_out", self.out), ws=self.ws_attn)

    def _project(self):
        grouped_out_proj(self.attn_out, self.W_o, out=self.out)

    def stages(self):
        """(name, callable) per stage, in order."""
        st = [("compress", self._compress)] if self.compress else []
        st += [("indexer_topk", self._index), ("attention", self._attend)]
        if self.wl.proj_groups:
            st.append(("out_proj", self._project))
        return st

    def kernel_probe(self):
        """The step's dominant kernel launched alone on the step's buffers:
        the indexer's scoring (a2), as (name, callable)."""
        wl = self.wl
        if not hasattr(self, "_scores"):
            self._scores = torch.empty((wl.B, 1, self.k_idx.shape[1]), dtype=torch.float32,
                                       device=self.out.device)

        def run():
            indexer_scores(self.q_idx, self.w, self.k_idx, self.q_pos, self.n_cmp, wl.m,
                           q_scale=self.q_scale, k_scale=self.k_scale, out=self._scores)
        return "indexer_score", run


class HcaDecodeStep(_Step):
    INPUTS = ("q", "seq_len", "q_pos")

    def __init__(self, inp: dict, device="cuda"):
        wl = inp["workload"]
        self.wl = wl
        dev = torch.device(device)
        B, W, D = wl.B, wl.W, wl.D
        lens = list(wl.lens)
        g = lambda k: None if inp.get(k) is None else inp[k].to(dev).clone()
        self.q, self.sink = g("q"), g("sink")
        self.seq_len, self.n_cmp = g("seq_len"), g("n_cmp")
        self.k_cmp, self.v_cmp = g("k_cmp"), g("v_cmp")
        self.kv8 = tuple(g(k) for k in KV8_KEYS) if wl.kv_fp8 else None
        self.q_pos = (self.seq_len - 1).view(B, 1).contiguous() if wl.kv_fp8 else None
        self.k_raw = _nan((B, W, D), torch.bfloat16, dev)
        self.v_raw = _nan((B, W, D), torch.bfloat16, dev)
        kw, vw = g("k_win"), g("v_win")
        for b, n in enumerate(lens):
            lo = max(0, n - W)
            _ring_put(self.k_raw, b, range(lo, n), kw[b, W - (n - lo):])
            _ring_put(self.v_raw, b, range(lo, n), vw[b, W - (n - lo):])
        self.out = torch.empty_like(self.q)
        self.ws_attn = torch.empty(max(1, attn_workspace(B, 1, wl.H, wl.N_cap + W)),
                                   dtype=torch.uint8, device=dev)
        self._pack_inputs()

    def _attend(self):
        wl = self.wl
        if wl.kv_fp8:
            B, H, D = self.q.shape
            attn_fp8kv(self.q.view(B, 1, H, D), *self.kv8, None, self.k_raw, self.v_raw,
                       self.q_pos, wl.W, self.sink, n_cmp=self.n_cmp, m_prime=wl.m,
                       out=self.out.view(B, 1, H, D), ws=self.ws_attn)
            return
        hca_dense_attn_decode(self.q, self.k_cmp, self.v_cmp, self.n_cmp, wl.m, self.k_raw,
                              self.v_raw, self.seq_len, wl.W, self.sink, out=self.out,
                              ws=self.ws_attn)

    def stages(self):
        return [("attention", self._attend)]

    def kernel_probe(self):
        """The step's one kernel: the dense attention, as (name, callable)."""
        return "attention", self._attend


class CsaPrefillStep(_Step):
    INPUTS = ("q", "q_idx", "w", "q_pos")

    def __init__(self, inp: dict, device="cuda"):
        wl = inp["workload"]
        self.wl = wl
        dev = torch.device(device)
        B, T, L, W, m, D = wl.B, wl.T, wl.L, wl.W, wl.m, wl.D
        R = W - 1 + T  # ring rows: positions L-W+1 .. L+T-1
        g = lambda k: None if inp.get(k) is None else inp[k].to(dev).clone()
        self.q, self.sink = g("q"), g("sink")
        self.q_pos, self.n_cmp = g("q_pos"), g("n_cmp")
        self.q_idx, self.w = g("q_idx"), g("w")
        self.k_cmp, self.v_cmp, self.k_idx = g("k_cmp"), g("v_cmp"), g("k_idx")
        n_old = L // m
        # new entries are produced by the step
        self.k_cmp[:, n_old:] = float("nan")
        self.v_cmp[:, n_old:] = float("nan")
        self.k_idx[:, n_old:] = float("nan")
        self.k_raw = _nan((B, R, D), torch.bfloat16, dev)
        self.v_raw = _nan((B, R, D), torch.bfloat16, dev)
        self.idx_raw = _nan((B, R, wl.d_I), torch.bfloat16, dev)
        base = L - (W - 1)
        rk, rv, ri = g("raw_k"), g("raw_v"), g("raw_idx")
        pre = wl.cspan - m  # rows before the first new block that its span reads
        assert pre <= W - 1, "the ring holds the window, so at most W-1 older rows"
        for b in range(B):
            _ring_put(self.k_raw, b, range(base, L + T), rk[b])
            _ring_put(self.v_raw, b, range(base, L + T), rv[b])
            _ring_put(self.idx_raw, b, range(L - pre, L + T), ri[b])
        self.gates = {s: tuple(t.to(dev) for t in inp["gate_" + s]) for s in ("k", "v", "idx")}
        self.block0, self.n_new = n_old, T // m
        self.idx = torch.empty((B, T, wl.k), dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.q)
        self.ws_idx = torch.empty(max(1, indexer_topk_workspace(B, T, wl.N_cap, wl.k)),
                                  dtype=torch.uint8, device=dev)
        self.ws_attn = torch.empty(max(1, attn_workspace(B, T, wl.H, wl.k + W)),
                                   dtype=torch.uint8, device=dev)
        self._pack_inputs()

    def _compress_kv(self):
        wl = self.wl
        for raw, dst, gate in ((self.k_raw, self.k_cmp, self.gates["k"]),
                               (self.v_raw, self.v_cmp, self.gates["v"])):
            compress_kv(raw, *gate, wl.m, self.block0, self.n_new, dst)

    def _compress_idx(self):
        wl = self.wl
        compress_kv(self.idx_raw, *self.gates["idx"], wl.m, self.block0, self.n_new, self.k_idx)

    def _compress(self):
        self._compress_kv()
        self._compress_idx()

    def __call__(self):
        return _overlapped(self, self._compress_kv, [self._compress_idx, self._index],
                           self._attend)

    def _index(self):
        wl = self.wl
        indexer_topk(self.q_idx, self.w, self.k_idx, self.q_pos, self.n_cmp, wl.m, wl.k,
                     out=self.idx, ws=self.ws_idx)

    def _attend(self):
        wl = self.wl
        sparse_attn_prefill(self.q, self.k_cmp, self.v_cmp, self.idx, self.k_raw, self.v_raw,
                            self.q_pos, wl.W, self.sink, out=self.out, ws=self.ws_attn)

    def stages(self):
        return [("compress", self._compress), ("indexer_topk", self._index),
                ("attention", self._attend)]

    def kernel_probe(self):
        """The step's longest single kernel: the sparse attention of every new
        token (one launch), as (name, callable)."""
        return "attention", self._attend


def make_step(inp: dict, device="cuda"):
    kind = inp["workload"].kind
    return {"csa_decode": CsaDecodeStep, "hca_decode": HcaDecodeStep,
            "csa_prefill": CsaPrefillStep}[kind](inp, device)
