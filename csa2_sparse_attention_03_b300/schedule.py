"""Device state for one CSA2 decode step over a static layer-mode schedule.

Allocates the packed caches (through torch), fills them through
``csa2_quantize_kv`` from seeded synthetic values, and assembles the
``csa2_layer_desc`` array that ``csa2_decode_layers`` consumes.  All
arithmetic of the path runs in the CUDA library; this module only moves
memory and builds descriptors.

Mode semantics follow the Helmcode "DeepSeek V4.1 Flash" explainer,
"03 · CSA2" (Full / Reindex / Reuse / SWA-only; Reuse layers keep their own
query and SWA state) and Louis Bouchard's KV-cache report, "Share the cache
and the search work" (pool-restricted Reindex).
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import (FMT_FP4_IDX, FMT_FP4_KV, FMT_FP8_SWA, MODE_FULL, MODE_REINDEX, MODE_REUSE, MODE_SWA_ONLY,
               Cache, csa2_cache, csa2_decode_layer, csa2_decode_layer_workspace, csa2_decode_layers,
               csa2_decode_layers_workspace, csa2_index_topk, csa2_layer_desc, csa2_quantize_kv, csa2_sparse_attn,
               layer_array, load, new_workspace, synth)

_MODE = {synth.FULL: MODE_FULL, synth.REINDEX: MODE_REINDEX, synth.REUSE: MODE_REUSE,
         synth.SWA_ONLY: MODE_SWA_ONLY}
BUILD_CHUNK = 65536


def _round_up(x, m):
    return (x + m - 1) // m * m


class DecodeStep:
    """Caches, per-layer inputs/outputs and descriptors of one workload.

    fill="host": values come from synth's numpy streams (bit-identical to what
    the oracle sees); fill="device": from seeded torch CUDA generators (bench
    sizes); fill="sampled": the caches of the sequences in ``host_seqs`` from
    the host streams, the others' caches from the device generators, every
    per-layer input (queries, weights, window rows) from the host streams -- a
    full-size step whose sampled sequences the oracle can follow.  The token at
    position L_b - 1 is left out of the build and passed as the step's append
    input, so every step re-writes it (idempotent).
    """

    def __init__(self, w: synth.Workload, device="cuda", fill="host", append=True, host_seqs=()):
        self.w = w
        self.device = device
        self.fill = fill
        self.host_seqs = set(int(b) for b in host_seqs)
        B, Lmax = w.batch, w.max_len
        self.B, self.Lmax = B, Lmax
        self.seq_lens = torch.tensor(w.seq_lens, dtype=torch.int32, device=device)
        self.window = w.window
        self.topk = w.topk
        self.pool_len = w.pool_len
        self.caches = {}      # full layer -> (kv Cache, idx Cache)
        self.swa = {}         # layer -> Cache
        self.new_rows = {}    # (kind, layer) -> [B, C] fp32 device
        self.page_tables = {}
        L_list = [int(x) for x in w.seq_lens]
        for f, ly in enumerate(w.layers):
            if ly.mode != synth.FULL:
                continue
            if w.paged:
                pages_per = [(_round_up(L, 64)) // 64 for L in L_list]
                n_pages = sum(pages_per)
                perm = synth.page_permutation(w, n_pages, f)
                maxp = max(pages_per)
                table = np.full((B, maxp), -1, np.int32)
                k = 0
                for b in range(B):
                    table[b, :pages_per[b]] = perm[k:k + pages_per[b]]
                    k += pages_per[b]
                t = torch.from_numpy(table).to(device)
                self.page_tables[f] = t
                kv = Cache.paged(FMT_FP4_KV, n_pages, 64, t, device)
                ik = Cache.paged(FMT_FP4_IDX, n_pages, 64, t, device)
            else:
                stride = _round_up(Lmax, 64)
                kv = Cache.contiguous(FMT_FP4_KV, B, stride, device)
                ik = Cache.contiguous(FMT_FP4_IDX, B, stride, device)
            self.caches[f] = (kv, ik)
            self._build_full(f, kv, ik, append)
        for l, ly in enumerate(w.layers):
            ring = Cache.contiguous(FMT_FP8_SWA, B, _round_up(max(w.window, 4), 4), device)
            self.swa[l] = ring
            self._build_swa(l, ring, append)
        self._alloc_layers()
        self._pack_arenas()
        self.descs = self._descs()
        self.arr = layer_array(self.descs)
        self.ws_bytes = csa2_decode_layers_workspace(self.descs, B, Lmax, self.topk, self.pool_len, self.window)
        if self.ws_bytes == 0:
            from . import csa2_last_error
            raise RuntimeError("workspace query failed: " + csa2_last_error())
        self.workspace = new_workspace(self.ws_bytes, device)

    # ---- value sources ----
    def _host(self, kind, b):
        if self.fill == "host":
            return True
        if self.fill == "sampled":
            return kind == "swa" or b in self.host_seqs
        return False

    def _rows(self, kind, layer, b, row0, n, width, scale=1.0):
        if self._host(kind, b):
            name = {"kv": "kv", "idxk": "idxk", "swa": "swa"}[kind]
            if kind == "swa":
                v = synth.swa_values(self.w, layer, b)[row0:row0 + n]
            else:
                v = synth.normal_rows(self.w.seed, name, (layer, b), row0, n, width)
            return torch.from_numpy(np.ascontiguousarray(v)).to(self.device)
        t = torch.empty((n, width), dtype=torch.float32, device=self.device)
        return synth.device_normal_(t, self.w.seed, kind, layer, b, row0, scale=scale)

    def _build_full(self, f, kv, ik, append):
        B = self.B
        new_kv = torch.zeros((B, 512), dtype=torch.float32, device=self.device)
        new_ik = torch.zeros((B, 64), dtype=torch.float32, device=self.device)
        start = torch.zeros(1, dtype=torch.int32, device=self.device)
        for b, L in enumerate(self.w.seq_lens):
            L = int(L)
            n_build = L - 1 if append else L
            kv_b, ik_b = kv.seq_view(b), ik.seq_view(b)
            for r0 in range(0, n_build, BUILD_CHUNK):
                n = min(BUILD_CHUNK, n_build - r0)
                start.fill_(r0)
                csa2_quantize_kv(self._rows("kv", f, b, r0, n, 512)[None], kv_b, start_pos=start)
                csa2_quantize_kv(self._rows("idxk", f, b, r0, n, 64)[None], ik_b, start_pos=start)
            if L >= 1:
                new_kv[b] = self._rows("kv", f, b, L - 1, 1, 512)[0]
                new_ik[b] = self._rows("idxk", f, b, L - 1, 1, 64)[0]
        torch.cuda.synchronize()
        if append:
            self.new_rows[("kv", f)] = new_kv
            self.new_rows[("idxk", f)] = new_ik

    def _build_swa(self, l, ring, append):
        """Window rows: synth row i of sequence b is position L_b - W + i (kept when >= 0)."""
        B, W = self.B, self.window
        src = torch.zeros((B, W, 512), dtype=torch.float32, device=self.device)
        new = torch.zeros((B, 512), dtype=torch.float32, device=self.device)
        start = torch.zeros((B,), dtype=torch.int32, device=self.device)
        lens = torch.zeros((B,), dtype=torch.int32, device=self.device)
        for b, L in enumerate(self.w.seq_lens):
            L = int(L)
            n = min(W, L)
            rows = self._rows("swa", l, b, W - n, n, 512)
            n_build = n - 1 if append else n
            src[b, :n_build] = rows[:n_build]
            start[b] = L - n
            lens[b] = L - n + n_build
            if n >= 1:
                new[b] = rows[n - 1]
        csa2_quantize_kv(src, ring, start_pos=start, seq_lens=lens)
        torch.cuda.synchronize()
        if append:
            self.new_rows[("swa", l)] = new

    def _alloc_layers(self):
        B, dev = self.B, self.device
        self.q, self.q_idx, self.wts, self.out, self.lse, self.idx, self.pool = {}, {}, {}, {}, {}, {}, {}
        host_inputs = self.fill in ("host", "sampled")
        for l, ly in enumerate(self.w.layers):
            if host_inputs:
                self.q[l] = torch.from_numpy(synth.query(self.w, l)).to(dev)
            else:
                self.q[l] = synth.device_normal_(torch.empty((B, 16, 512), device=dev), self.w.seed, "q", l,
                                                 scale=synth.query_scale(self.w))
            self.out[l] = torch.zeros((B, 16, 512), dtype=torch.float32, device=dev)
            self.lse[l] = torch.zeros((B, 16), dtype=torch.float32, device=dev)
            if ly.mode in (synth.FULL, synth.REINDEX):
                if host_inputs:
                    self.q_idx[l] = torch.from_numpy(synth.index_query(self.w, l)).to(dev)
                    self.wts[l] = torch.from_numpy(synth.index_weights(self.w, l)).to(dev)
                else:
                    self.q_idx[l] = synth.device_normal_(torch.empty((B, 4, 64), device=dev), self.w.seed,
                                                         "qidx", l, scale=1.0 / 8.0)
                    self.wts[l] = synth.device_uniform_(torch.empty((B, 4), device=dev), self.w.seed, "widx", l)
                self.idx[l] = torch.full((B, self.topk), -7, dtype=torch.int32, device=dev)
                if ly.mode == synth.FULL and self.pool_len:
                    self.pool[l] = torch.full((B, self.pool_len), -7, dtype=torch.int32, device=dev)

    def _pack_arenas(self):
        """Place the per-step inputs (queries, indexer queries and weights, the
        appended rows) in one contiguous device buffer and the per-step outputs
        (out, lse, indices, pools) in another, so a caller moves each direction
        with a single copy.  Both are laid out layer by layer (every input of
        layer l before any of layer l + 1), so that a prefix of layers is a
        prefix of bytes: ``in_ranges[l]`` / ``out_ranges[l]`` are layer l's
        byte ranges."""
        import torch

        def pack(per_layer):
            offs, total, ranges = [], 0, []
            for ts in per_layer:
                start = total
                for t in ts:
                    offs.append(total)
                    total += (t.numel() * t.element_size() + 255) // 256 * 256
                ranges.append((start, total))
            arena = torch.zeros(max(total, 256), dtype=torch.uint8, device=self.device)
            views, k = [], 0
            for ts in per_layer:
                vs = []
                for t in ts:
                    n = t.numel() * t.element_size()
                    view = arena[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
                    view.copy_(t)
                    vs.append(view)
                    k += 1
                views.append(vs)
            return arena, views, ranges

        L = len(self.w.layers)
        in_groups = [self.q, self.q_idx, self.wts]
        in_keys = [[(g, l) for g in range(3) if l in in_groups[g]] +
                   [("row", key) for key in self.new_rows if key[1] == l] for l in range(L)]

        def fetch(ref):
            return in_groups[ref[0]][ref[1]] if ref[0] != "row" else self.new_rows[ref[1]]

        self.arena_in, views, self.in_ranges = pack([[fetch(r) for r in keys] for keys in in_keys])
        for keys, vs in zip(in_keys, views):
            for r, v in zip(keys, vs):
                if r[0] == "row":
                    self.new_rows[r[1]] = v
                else:
                    in_groups[r[0]][r[1]] = v
        out_groups = [self.out, self.lse, self.idx, self.pool]
        out_keys = [[(g, l) for g in range(4) if l in out_groups[g]] for l in range(L)]
        self.arena_out, views, self.out_ranges = pack([[out_groups[g][l] for g, l in keys] for keys in out_keys])
        for keys, vs in zip(out_keys, views):
            for (g, l), v in zip(keys, vs):
                out_groups[g][l] = v
        torch.cuda.synchronize(self.device)

    def _descs(self):
        descs = []
        P = lambda t: t.data_ptr() if t is not None else None
        for l, ly in enumerate(self.w.layers):
            d = csa2_layer_desc()
            d.mode = _MODE[ly.mode]
            d.kv_src = ly.kv_src
            d.idx_src = ly.idx_src
            d.use_pool = 1 if ly.use_pool else 0
            if ly.mode == synth.FULL:
                kv, ik = self.caches[l]
                d.kv = ctypes.pointer(kv.desc)
                d.idx_keys = ctypes.pointer(ik.desc)
                d.new_kv = P(self.new_rows.get(("kv", l)))
                d.new_idx_key = P(self.new_rows.get(("idxk", l)))
            d.swa = ctypes.pointer(self.swa[l].desc)
            d.new_swa = P(self.new_rows.get(("swa", l)))
            d.q = P(self.q[l])
            d.q_idx = P(self.q_idx.get(l))
            d.w = P(self.wts.get(l))
            d.out = P(self.out[l])
            d.lse = P(self.lse[l])
            d.idx_out = P(self.idx.get(l))
            d.pool_out = P(self.pool.get(l))
            descs.append(d)
        return descs

    def run(self, stream=None):
        csa2_decode_layers(self.descs, self.B, self.seq_lens, self.Lmax, self.topk, self.pool_len, self.window,
                           self.workspace, stream=stream, arr=self.arr)

    def capture(self, stream, host_in=None, host_out=None):
        """Capture one decode step in a CUDA graph on `stream` and return it.

        With pinned host buffers `host_in` (the size of ``step_inputs()[0]``)
        and `host_out` (the size of ``step_outputs()[0]``), the graph also
        copies the step's inputs in from the host first and its outputs back
        after, so one replay is a whole serving step.  The step's kernels are
        captured as launched by ``csa2_decode_layers``."""
        import torch

        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            if host_in is not None:
                self.arena_in.copy_(host_in, non_blocking=True)
            self.run(stream=stream)
            if host_out is not None:
                host_out.copy_(self.arena_out, non_blocking=True)
        return g

    def capture_sequential(self, stream, host_in, host_out, in_groups=None, out_groups=None):
        """Capture one serving step in the layer-sequential order in a CUDA
        graph on `stream`: the step's inputs copied in from the pinned host
        buffer `host_in`, every layer's ``csa2_decode_layer`` call, its
        outputs copied back to the pinned `host_out`.  The copies overlap the
        kernels: groups of layers' inputs are copied on a second stream, in
        layer order, and a layer waits only for its own group; each group of
        layers' outputs goes back on a third stream as soon as its last layer
        is done.  `in_groups` / `out_groups` are the first layers of each
        group (default: growing groups in, shrinking groups out, so that the
        first layer waits for little and the last copy is short)."""
        import torch

        L = len(self.w.layers)
        in_groups = sorted(set(in_groups if in_groups is not None else [0, 1, 4, 12])) or [0]
        out_groups = sorted(set(out_groups if out_groups is not None else [0, L - 8, L - 3, L - 1]))
        in_groups = [l for l in in_groups if 0 <= l < L]
        out_groups = [l for l in out_groups if 0 <= l < L]
        if not in_groups or in_groups[0] != 0:
            in_groups = [0] + in_groups
        if not out_groups or out_groups[0] != 0:
            out_groups = [0] + out_groups
        if not hasattr(self, "_seq_ws"):
            need = csa2_decode_layer_workspace(self.descs, self.B, self.Lmax, self.topk, self.pool_len, self.window)
            self._seq_ws = new_workspace(need, self.device)
        dev = self.device
        s_in = torch.cuda.Stream(device=dev)
        s_out = torch.cuda.Stream(device=dev)

        def span(ranges, l0, l1):
            return ranges[l0][0], ranges[l1 - 1][1]

        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            start = torch.cuda.Event()
            start.record(stream)
            s_in.wait_event(start)
            bounds = in_groups + [L]
            ready = []
            with torch.cuda.stream(s_in):
                for k in range(len(in_groups)):
                    a, b = span(self.in_ranges, bounds[k], bounds[k + 1])
                    if b > a:
                        self.arena_in[a:b].copy_(host_in[a:b], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(s_in)
                    ready.append(e)
            obounds = out_groups + [L]
            ends = set(b - 1 for b in obounds[1:])
            k_in = 0
            for l in range(L):
                if k_in < len(in_groups) and l == in_groups[k_in]:
                    stream.wait_event(ready[k_in])
                    k_in += 1
                csa2_decode_layer(self.descs, l, self.B, self.seq_lens, self.Lmax, self.topk, self.pool_len,
                                  self.window, self._seq_ws, stream=stream, arr=self.arr)
                if l in ends:
                    k = obounds.index(l + 1) - 1
                    done = torch.cuda.Event()
                    done.record(stream)
                    s_out.wait_event(done)
                    a, b = span(self.out_ranges, obounds[k], l + 1)
                    if b > a:
                        with torch.cuda.stream(s_out):
                            host_out[a:b].copy_(self.arena_out[a:b], non_blocking=True)
            joined = torch.cuda.Event()
            joined.record(s_out)
            stream.wait_event(joined)
        return g

    def run_sequential(self, stream=None):
        """The same step in the layer-sequential order a model runs it in: one
        ``csa2_decode_layer`` call per layer, in schedule order (each layer's
        appends, its indexing when it is a Full or Reindex layer, its
        attention).  Writes the same outputs as ``run``.  Graph-capturable."""
        if not hasattr(self, "_seq_ws"):
            need = csa2_decode_layer_workspace(self.descs, self.B, self.Lmax, self.topk, self.pool_len, self.window)
            if need == 0:
                from . import csa2_last_error
                raise RuntimeError("layer workspace query failed: " + csa2_last_error())
            self._seq_ws = new_workspace(need, self.device)
        for l in range(len(self.descs)):
            csa2_decode_layer(self.descs, l, self.B, self.seq_lens, self.Lmax, self.topk, self.pool_len,
                              self.window, self._seq_ws, stream=stream, arr=self.arr)

    def run_sequential_calls(self, stream=None):
        """The layer-sequential order through the step-1..3 entry points
        (csa2_quantize_kv, csa2_index_topk, csa2_sparse_attn), one call each."""
        if not hasattr(self, "_calls_ws"):
            lib = load()
            need = max(int(lib.csa2_index_topk_workspace(self.B, self.Lmax, self.pool_len, self.topk,
                                                           self.pool_len)), 1)
            self._calls_ws = new_workspace(need, self.device)
            self._seq_last = (self.seq_lens - 1).clamp(min=0)
        ws, last = self._calls_ws, self._seq_last
        for l, ly in enumerate(self.w.layers):
            if ly.mode == synth.FULL and ("kv", l) in self.new_rows:
                kv, ik = self.caches[l]
                csa2_quantize_kv(self.new_rows[("kv", l)][:, None], kv, start_pos=last, seq_lens=self.seq_lens,
                                 stream=stream)
                csa2_quantize_kv(self.new_rows[("idxk", l)][:, None], ik, start_pos=last, seq_lens=self.seq_lens,
                                 stream=stream)
            if ("swa", l) in self.new_rows and self.window > 0:
                csa2_quantize_kv(self.new_rows[("swa", l)][:, None], self.swa[l], start_pos=last,
                                 seq_lens=self.seq_lens, stream=stream)
            if ly.mode == synth.FULL:
                csa2_index_topk(MODE_FULL, self.caches[l][1], self.q_idx[l], self.wts[l], self.seq_lens, self.Lmax,
                                self.topk, out_idx=self.idx[l], out_pool=self.pool.get(l), workspace=ws,
                                stream=stream)
            elif ly.mode == synth.REINDEX:
                pool = self.pool.get(ly.kv_src) if ly.use_pool else None
                csa2_index_topk(MODE_REINDEX, self.caches[ly.kv_src][1], self.q_idx[l], self.wts[l], self.seq_lens,
                                self.Lmax, self.topk, pool=pool, out_idx=self.idx[l], workspace=ws, stream=stream)
            if ly.mode == synth.SWA_ONLY:
                kv, idx, topk = None, None, 0
            else:
                kv = self.caches[ly.kv_src][0]
                idx = self.idx[l] if ly.mode in (synth.FULL, synth.REINDEX) else self.idx[ly.idx_src]
                topk = self.topk
            csa2_sparse_attn(kv, self.swa[l], self.q[l], self.seq_lens, self.Lmax, idx, topk, self.window,
                             out=self.out[l], lse=self.lse[l], stream=stream)

    def attention_only(self, l, stream=None):
        """Layer l's attention alone (csa2_sparse_attn over its selection and
        window, no append), for timing the attention kernel."""
        ly = self.w.layers[l]
        if ly.mode == synth.SWA_ONLY:
            kv, idx, topk = None, None, 0
        else:
            kv = self.caches[ly.kv_src][0]
            idx = self.idx[l] if ly.mode in (synth.FULL, synth.REINDEX) else self.idx[ly.idx_src]
            topk = self.topk
        csa2_sparse_attn(kv, self.swa[l], self.q[l], self.seq_lens, self.Lmax, idx, topk, self.window,
                         out=self.out[l], lse=self.lse[l], stream=stream)

    def index_only(self, l, stream=None):
        """Indexing layer l's scoring and Top-K alone (csa2_index_topk, no
        append), for timing the indexing kernel."""
        if not hasattr(self, "_calls_ws"):
            need = max(int(load().csa2_index_topk_workspace(self.B, self.Lmax, self.pool_len, self.topk,
                                                            self.pool_len)), 1)
            self._calls_ws = new_workspace(need, self.device)
            self._seq_last = (self.seq_lens - 1).clamp(min=0)
        ly = self.w.layers[l]
        if ly.mode == synth.FULL:
            csa2_index_topk(MODE_FULL, self.caches[l][1], self.q_idx[l], self.wts[l], self.seq_lens, self.Lmax,
                            self.topk, out_idx=self.idx[l], out_pool=self.pool.get(l), workspace=self._calls_ws,
                            stream=stream)
        elif ly.mode == synth.REINDEX:
            pool = self.pool.get(ly.kv_src) if ly.use_pool else None
            csa2_index_topk(MODE_REINDEX, self.caches[ly.kv_src][1], self.q_idx[l], self.wts[l], self.seq_lens,
                            self.Lmax, self.topk, pool=pool, out_idx=self.idx[l], workspace=self._calls_ws,
                            stream=stream)

    # ---- inputs/outputs moved per step in the end-to-end measurement ----
    def step_inputs(self):
        """What a caller supplies per decode step (queries, indexer queries,
        weights and the appended token rows), as one contiguous buffer."""
        return [self.arena_in]

    def step_outputs(self):
        """What a step returns (out, lse, indices, pools), as one contiguous buffer."""
        return [self.arena_out]
