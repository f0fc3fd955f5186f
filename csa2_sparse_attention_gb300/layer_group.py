"""One CSA2 layer group on one GPU: device state and the decode step's calls.

[T1] "DeepSeek V4.1-Flash 为什么这么强？CED 与 CSA2 架构全拆解", §二: the decoder's
20 layers run as [Full + 3 Reuse] + 4 x [Reindex + 3 Reuse]; Full layers write
the main KV and indexer K and run the full index, Reindex layers share them
and pick their own top-k inside the pool, Reuse layers reuse the indices
(the same top-k buffer is passed again).  Every layer keeps its own attention
query and sliding-window KV.

This module only allocates device memory (torch) and issues C-ABI calls in
that order; all arithmetic runs in libcsa2.so.
"""
from __future__ import annotations

import math
from typing import NamedTuple

import numpy as np
import torch

from . import abi
from . import workloads as W


def _round8(n):
    return (int(n) + 7) // 8 * 8


class _Flat:
    """Typed tensors carved in order out of one flat byte buffer, each
    starting 256-byte aligned, so that a run of them moves in one copy."""

    def __init__(self):
        self.items = []
        self.size = 0

    def add(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.items.append((self.size, n, tuple(shape), dtype))
        self.size = (self.size + n + 255) // 256 * 256
        return len(self.items) - 1

    def offset(self, i):
        return self.items[i][0] if i < len(self.items) else self.size

    def views(self, buf):
        return [buf[o:o + n].view(dt).view(sh) for o, n, sh, dt in self.items]


class HostIO(NamedTuple):
    """Pinned host buffers of one step's inputs and outputs: per-tensor views
    (app inputs, per-layer inputs, per-layer [out, lse]) of two flat buffers."""
    app: list
    layers: list
    outs: list
    flat_in: torch.Tensor
    flat_out: torch.Tensor


class LayerGroup:
    """Caches, per-layer inputs/outputs and workspaces of one workload."""

    def __init__(self, wl: W.Workload, device="cuda", sm_scale=1.0 / math.sqrt(512.0),
                 rope_theta=10000.0, out_dtype=torch.float32, ik_layout=abi.LAYOUT_BLOCK8R, fused_q=True):
        self.wl = wl
        # fused_q: the index calls take the bf16 indexer query and quantize it
        # themselves (csa2_index_*_bf16); else a separate FP4 append per layer
        # fills iq_codes / iq_scales first
        self.fused_q = fused_q
        self.dev = torch.device(device)
        self.B = wl.batch
        self.layers = wl.layers
        self.P, self.K, self.Wn = wl.pool_blocks, wl.topk, wl.window
        self.sm_scale = sm_scale
        self.contexts = np.array(wl.contexts, dtype=np.int64)
        if wl.shared_cache:
            self.n_rows = _round8(wl.cache_entries)
            starts = np.zeros(self.B, dtype=np.int64)
            self.row_base = [0]
        else:
            caps = np.array([_round8(n) for n in wl.contexts], dtype=np.int64)
            starts = np.concatenate([[0], np.cumsum(caps)[:-1]]).astype(np.int64)
            self.n_rows = int(caps.sum())
            self.row_base = list(starts)
        self.kv_start_h = starts
        d = self.dev
        self.kv_start = torch.from_numpy(starts).to(d)
        self.n_visible = torch.from_numpy(self.contexts.astype(np.int32)).to(d)
        self.max_visible = int(self.contexts.max())
        u8 = torch.uint8
        self.kv_codes = torch.zeros((self.n_rows, 256), dtype=u8, device=d)
        self.kv_scales = torch.zeros((self.n_rows, 32), dtype=u8, device=d)
        # indexer K: 576-byte records of 8 rows (codes then scales), or BLOCK8
        # codes with a separate scale plane
        self.ik_layout = ik_layout
        if ik_layout == abi.LAYOUT_BLOCK8R:
            self.ik_codes = torch.zeros((self.n_rows // 8 * 576,), dtype=u8, device=d)
            self.ik_scales = None
        else:
            self.ik_codes = torch.zeros((self.n_rows * 64,), dtype=u8, device=d)
            self.ik_scales = torch.zeros((self.n_rows, 8), dtype=u8, device=d)
        max_pos = int(max(self.n_rows, self.contexts.max() * wl.m + wl.m))
        self.rope_max_pos = max_pos
        self.rope = torch.empty(abi.csa2_rope_table_bytes(512, max_pos), dtype=u8, device=d)
        abi.csa2_rope_table_init(rope_theta, 512, max_pos, self.rope, torch.cuda.current_stream(d))
        L = len(self.layers)
        # window latents per layer: a ring per query (decode), or one E4M3 row
        # per position of the shared sequence (prefill over a shared cache)
        if wl.shared_window:
            self.swa = [torch.zeros((self.n_rows, 512), dtype=u8, device=d) for _ in range(L)]
        else:
            self.swa = [torch.zeros((self.B, self.Wn, 512), dtype=u8, device=d) for _ in range(L)]
        self.out_dtype = out_dtype
        self.out_code = abi.OUT_F32 if out_dtype == torch.float32 else abi.OUT_BF16
        self.index_layers = [i for i, m in enumerate(self.layers) if m in (W.FULL, W.REINDEX)]
        # the step's inputs and outputs live in two flat buffers, in the
        # order the step uses them: [current-token latents] + per layer
        # [(indexer q, w), attention q, window latent], and per layer [out, lse]
        bf = torch.bfloat16
        fin, fout = _Flat(), _Flat()
        i_tok = (fin.add((self.B, 512), bf), fin.add((self.B, 128), bf))
        self._in_layer = []  # per layer: first item of its index part, of its attention part
        vid = {}
        for li in range(L):
            first = len(fin.items)
            if li in self.index_layers:
                vid[li, "iq"] = fin.add((self.B * 32, 128), bf)
                vid[li, "iw"] = fin.add((self.B, 32), torch.float32)
            first_attn = len(fin.items)
            vid[li, "q"] = fin.add((self.B, 64, 512), bf)
            vid[li, "swa"] = fin.add((self.B, 512), bf)
            self._in_layer.append((first, first_attn))
        self._out_layer = [(fout.add((self.B, 64, 512), out_dtype), fout.add((self.B, 64), torch.float32))
                           for _ in range(L)]
        self._fin, self._fout = fin, fout
        self.io_in = torch.zeros(fin.size, dtype=u8, device=d)
        self.io_out = torch.zeros(fout.size, dtype=u8, device=d)
        vin, vout = fin.views(self.io_in), fout.views(self.io_out)
        self.attn_q = [vin[vid[li, "q"]] for li in range(L)]
        self.out = [vout[o] for o, _ in self._out_layer]
        self.lse = [vout[l_] for _, l_ in self._out_layer]
        self.iq_bf16 = {i: vin[vid[i, "iq"]] for i in self.index_layers}
        self.iq_codes = {i: torch.zeros((self.B * 32 * 64,), dtype=u8, device=d) for i in self.index_layers}
        self.iq_scales = {i: torch.zeros((self.B * 32, 8), dtype=u8, device=d) for i in self.index_layers}
        self.iw = {i: vin[vid[i, "iw"]] for i in self.index_layers}
        self.topk = {i: torch.full((self.B, self.K), -1, dtype=torch.int32, device=d) for i in self.index_layers}
        # one pool per Full layer (its group's Reindex layers read it); .pool
        # is the first group's
        self.full_layers = [i for i, m in enumerate(self.layers) if m == W.FULL]
        self.pools = {i: torch.full((self.B, self.P), -1, dtype=torch.int32, device=d) for i in self.full_layers}
        self.pool = self.pools[self.full_layers[0]]
        # per layer, the top-k tensor its attention call was given (Reuse
        # layers get their index source's buffer itself, not a copy)
        self.attn_index = {}
        # current-token inputs of a decode step
        self.tok_latent, self.tok_ik = vin[i_tok[0]], vin[i_tok[1]]
        self.tok_swa = [vin[vid[li, "swa"]] for li in range(L)]
        last = self.contexts - 1
        self.tok_pos = torch.from_numpy(last * wl.m + (wl.m - 1)).to(d)
        self.tok_row = torch.from_numpy(starts + last).to(d)
        # workspaces
        B, mv = self.B, self.max_visible
        self.ws_app = torch.zeros(abi.csa2_workspace_bytes(abi.OP_APPEND, B, mv, self.P, self.K), dtype=u8, device=d)
        self.ws_full = torch.zeros(abi.csa2_workspace_bytes(abi.OP_INDEX_FULL, B, mv, self.P, self.K), dtype=u8, device=d)
        self.ws_re = torch.zeros(abi.csa2_workspace_bytes(abi.OP_INDEX_REINDEX, B, mv, self.P, self.K), dtype=u8, device=d)
        self.ws_attn = torch.zeros(abi.csa2_workspace_bytes(abi.OP_SPARSE_ATTN, B, mv, self.P, self.K), dtype=u8, device=d)
        self.graph = None

    # ------------------------------------------------------------ inputs
    def fill(self, stream=None, requests=None):
        """Draw the workload's synthetic inputs and write the caches through
        the library's own append kernels (bulk), plus per-layer inputs."""
        wl, d = self.wl, self.dev
        s = stream or torch.cuda.current_stream(d)
        reqs = [0] if wl.shared_cache else range(self.B)
        for r in (requests if requests is not None else reqs):
            base = self.row_base[r]
            rows = W.cache_rows(wl, r)
            k = torch.from_numpy(W.indexer_k(wl, r)).to(torch.bfloat16).to(d)
            dst = torch.arange(base, base + rows, dtype=torch.int64, device=d)
            abi.csa2_quantize_append(k, rows, 128, abi.FMT_FP4, self.ik_layout, None, None, 0, dst,
                                     self.n_rows, self.ik_codes, self.ik_scales, self.ws_app,
                                     self.ws_app.numel(), s)
            del k
            lat = torch.from_numpy(W.main_latent(wl, r)).to(torch.bfloat16).to(d)
            pos = torch.from_numpy(W.latent_positions(wl, r)).to(d)
            abi.csa2_quantize_append(lat, rows, 512, abi.FMT_FP4, abi.LAYOUT_ROWS, pos, self.rope,
                                     self.rope_max_pos, dst, self.n_rows, self.kv_codes, self.kv_scales,
                                     self.ws_app, self.ws_app.numel(), s)
            s.synchronize()
            del lat, pos, dst
        self.fill_layer_inputs(stream=s)

    def fill_layer_inputs(self, stream=None):
        wl, d = self.wl, self.dev
        s = stream or torch.cuda.current_stream(d)
        bf = torch.bfloat16
        for li in range(len(self.layers)):
            if wl.shared_window:  # the layer's window latents over the whole shared sequence
                step = 65536
                for r0 in range(0, wl.cache_entries, step):
                    r1 = min(wl.cache_entries, r0 + step)
                    rows_t = torch.from_numpy(W.swa_seq_rows(wl, li, r0, r1)).to(bf).to(d)
                    dst = torch.arange(r0, r1, dtype=torch.int64, device=d)
                    abi.csa2_quantize_append(rows_t, r1 - r0, 512, abi.FMT_FP8, abi.LAYOUT_ROWS, None, None, 0,
                                             dst, self.n_rows, self.swa[li], None, self.ws_app,
                                             self.ws_app.numel(), s)
                    s.synchronize()
            else:
                rings = np.stack([W.swa_ring(wl, q, li) for q in range(self.B)])
                ring_t = torch.from_numpy(rings.reshape(-1, 512)).to(bf).to(d)
                abi.csa2_quantize_append(ring_t, ring_t.shape[0], 512, abi.FMT_FP8, abi.LAYOUT_ROWS, None, None,
                                         0, None, self.B * self.Wn, self.swa[li], None, self.ws_app,
                                         self.ws_app.numel(), s)
                last = self.contexts - 1
                self.tok_swa[li].copy_(torch.from_numpy(rings[np.arange(self.B), last % self.Wn]).to(bf))
            self.attn_q[li].copy_(torch.from_numpy(np.stack([W.attn_q(wl, q, li) for q in range(self.B)])).to(bf))
            if li in self.index_layers:
                self.iq_bf16[li].copy_(torch.from_numpy(
                    np.stack([W.indexer_q(wl, q, li) for q in range(self.B)]).reshape(-1, 128)).to(bf))
                self.iw[li].copy_(torch.from_numpy(np.stack([W.indexer_w(wl, q, li) for q in range(self.B)])))
        if not wl.shared_cache:
            lat_tok, ik_tok = [], []
            for q in range(self.B):
                n = int(self.contexts[q])
                lat_tok.append(W.main_latent_rows(wl, q, n - 1, n)[0])
                ik_tok.append(W.indexer_k_rows(wl, q, n - 1, n)[0])
            self.tok_latent.copy_(torch.from_numpy(np.stack(lat_tok)).to(bf))
            self.tok_ik.copy_(torch.from_numpy(np.stack(ik_tok)).to(bf))
        s.synchronize()

    # ------------------------------------------------------------ the step
    def append_token(self, s):
        """Append the current token (position n-1) of every request."""
        abi.csa2_quantize_append(self.tok_ik, self.B, 128, abi.FMT_FP4, self.ik_layout, None, None, 0,
                                 self.tok_row, self.n_rows, self.ik_codes, self.ik_scales, self.ws_app,
                                 self.ws_app.numel(), s)
        abi.csa2_quantize_append(self.tok_latent, self.B, 512, abi.FMT_FP4, abi.LAYOUT_ROWS, self.tok_pos,
                                 self.rope, self.rope_max_pos, self.tok_row, self.n_rows, self.kv_codes,
                                 self.kv_scales, self.ws_app, self.ws_app.numel(), s)

    def layer(self, li, s, swa_append=True):
        """One layer: index (Full / Reindex; Reuse makes no call), then
        attention with this layer's window append fused in (swa_append)."""
        self.layer_index(li, s)
        self.layer_attn(li, s, swa_append)

    def layer_index(self, li, s):
        """The index part of a layer (Full / Reindex; Reuse makes no call)."""
        mode = self.layers[li]
        B = self.B
        if self.fused_q:
            if mode == W.FULL:
                abi.csa2_index_full_bf16(self.iq_bf16[li], self.iw[li], B, self.ik_codes, self.ik_scales, self.n_rows,
                                         self.kv_start, self.n_visible, self.max_visible, self.P, self.K,
                                         self.pools[li], self.topk[li], self.ws_full, self.ws_full.numel(), s)
            elif mode == W.REINDEX:
                abi.csa2_index_reindex_bf16(self.iq_bf16[li], self.iw[li], B, self.ik_codes, self.ik_scales,
                                            self.n_rows, self.kv_start, self.n_visible, self.max_visible,
                                            self.pools[self.group_full(li)], self.P, self.K, self.topk[li],
                                            self.ws_re, self.ws_re.numel(), s)
            return
        if mode in (W.FULL, W.REINDEX):
            abi.csa2_quantize_append(self.iq_bf16[li], B * 32, 128, abi.FMT_FP4, abi.LAYOUT_BLOCK8, None, None,
                                     0, None, B * 32, self.iq_codes[li], self.iq_scales[li], self.ws_app,
                                     self.ws_app.numel(), s)
        if mode == W.FULL:
            abi.csa2_index_full(self.iq_codes[li], self.iq_scales[li], self.iw[li], B, self.ik_codes,
                                self.ik_scales, self.n_rows, self.kv_start, self.n_visible, self.max_visible,
                                self.P, self.K, self.pools[li], self.topk[li], self.ws_full, self.ws_full.numel(), s)
        elif mode == W.REINDEX:
            abi.csa2_index_reindex(self.iq_codes[li], self.iq_scales[li], self.iw[li], B, self.ik_codes,
                                   self.ik_scales, self.n_rows, self.kv_start, self.n_visible,
                                   self.max_visible, self.pools[self.group_full(li)], self.P, self.K,
                                   self.topk[li], self.ws_re, self.ws_re.numel(), s)

    def group_full(self, li):
        """The Full layer whose pool layer li's group uses."""
        return max(i for i in self.full_layers if i <= li)

    def layer_attn(self, li, s, swa_append=True):
        """The attention of a layer over its index source's top-k."""
        B = self.B
        idx = self.topk[W.index_source(self.wl, li)]
        self.attn_index[li] = idx
        if self.wl.shared_window:  # prefill: each query's causal window over the shared sequence
            abi.csa2_sparse_attn_prefill(self.attn_q[li], B, self.kv_codes, self.kv_scales, self.n_rows,
                                         self.kv_start, self.n_visible, idx, self.K, self.swa[li], self.Wn,
                                         self.sm_scale, self.out[li], self.out_code, self.lse[li], self.ws_attn,
                                         self.ws_attn.numel(), s)
            return
        abi.csa2_sparse_attn(self.attn_q[li], B, self.kv_codes, self.kv_scales, self.n_rows, self.kv_start,
                             self.n_visible, idx, self.K, self.swa[li],
                             self.tok_swa[li] if swa_append else None, self.Wn, self.sm_scale,
                             self.out[li], self.out_code, self.lse[li], self.ws_attn, self.ws_attn.numel(), s)

    def step(self, stream=None, append=True):
        """One pass of the whole group: append, then every layer in order."""
        s = stream or torch.cuda.current_stream(self.dev)
        if append and not self.wl.shared_cache:
            self.append_token(s)
        for li in range(len(self.layers)):
            self.layer(li, s, swa_append=append and not self.wl.shared_cache)

    def io_tensors(self):
        """The per-step inputs (append, then per layer) and outputs (per layer)
        that travel between host and device in step_io()."""
        ins_app = [self.tok_latent, self.tok_ik] if not self.wl.shared_cache else []
        ins_layer = []
        for li in range(len(self.layers)):
            t = [self.attn_q[li]]
            if not self.wl.shared_cache:
                t.append(self.tok_swa[li])
            if li in self.index_layers:
                t += [self.iq_bf16[li], self.iw[li]]
            ins_layer.append(t)
        outs_layer = [[self.out[li], self.lse[li]] for li in range(len(self.layers))]
        return ins_app, ins_layer, outs_layer

    def host_buffers(self):
        """Pinned host copies of the step's flat input and output buffers
        (holding the current inputs), with per-tensor views, for step_io()."""
        flat_in = self.io_in.cpu().pin_memory()
        flat_out = self.io_out.cpu().pin_memory()
        vin, vout = self._fin.views(flat_in), self._fout.views(flat_out)
        app = vin[:2] if not self.wl.shared_cache else []
        layers = []
        for li, (first, first_attn) in enumerate(self._in_layer):
            t = [vin[first_attn]] + ([vin[first_attn + 1]] if not self.wl.shared_cache else [])
            layers.append(t + vin[first:first_attn])
        outs = [[vout[o], vout[l_]] for o, l_ in self._out_layer]
        return HostIO(app, layers, outs, flat_in, flat_out)

    # where the compute stream waits for the inputs copied so far, as (layer,
    # part) with part 0 the index calls and 1 the attention: a wait breaks
    # the chain of programmatic launches and costs a few microseconds, so the
    # inputs come in a few growing groups, the first one small
    IO_WAIT_AT = ((0, 0), (0, 1), (3, 0), (8, 0), (15, 0))

    def step_io(self, stream, copy_streams, host):
        """step() with its host I/O pipelined on two more streams: the first
        brings the inputs in from pinned host memory in a few growing groups
        (one copy each, ahead of their use), the second returns each layer's
        [out, lse] in one copy as soon as that layer is done, while `stream`
        computes the later layers.  `host` comes from host_buffers()."""
        h2d, d2h = copy_streams
        L = len(self.layers)
        waits = [w for w in self.IO_WAIT_AT if w[0] < L]
        first_item = lambda w: self._in_layer[w[0]][w[1]]
        starts = [0] + [self._fin.offset(first_item(w)) for w in waits[1:]]
        ends = starts[1:] + [self._fin.size]
        start = torch.cuda.Event()
        start.record(stream)
        h2d.wait_event(start)
        d2h.wait_event(start)
        ev = {}
        with torch.cuda.stream(h2d):
            for w, lo, hi in zip(waits, starts, ends):
                self.io_in[lo:hi].copy_(host.flat_in[lo:hi], non_blocking=True)
                e = torch.cuda.Event()
                e.record(h2d)
                ev[w] = e
        stream.wait_event(ev[waits[0]])
        if not self.wl.shared_cache:
            self.append_token(stream)
        for li in range(L):
            for part in (0, 1):
                if (li, part) in ev and (li, part) != waits[0]:
                    stream.wait_event(ev[li, part])
                if part == 0:
                    self.layer_index(li, stream)
                else:
                    self.layer_attn(li, stream, swa_append=not self.wl.shared_cache)
            done = torch.cuda.Event()
            done.record(stream)
            d2h.wait_event(done)
            o_, l_ = self._out_layer[li]
            lo, hi = self._fout.offset(o_), self._fout.offset(l_ + 1)
            with torch.cuda.stream(d2h):
                host.flat_out[lo:hi].copy_(self.io_out[lo:hi], non_blocking=True)
        for cs in (h2d, d2h):
            end = torch.cuda.Event()
            end.record(cs)
            stream.wait_event(end)

    def capture_io(self, stream, copy_streams, host):
        """Capture step_io() into a CUDA graph (replayed by replay_io())."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.step_io(stream, copy_streams, host)
        self.graph_io = g
        return g

    def replay_io(self):
        self.graph_io.replay()

    def capture(self, stream):
        """Capture step() into a CUDA graph on `stream` (replayed by replay())."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.step(stream=stream)
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()

    def status(self):
        """Status words of every workspace (first device-detected problem)."""
        return {name: abi.csa2_status_fetch(ws) for name, ws in
                (("append", self.ws_app), ("full", self.ws_full), ("reindex", self.ws_re), ("attn", self.ws_attn))}
