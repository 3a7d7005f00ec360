"""DecodeRunner: the decode step over a layer range, as a user calls it.

Holds the cache, the per-step device buffers and the workspace, and issues the
calls of one decode step (index + select, ensure, remap, attention) on the
current stream.  Two launch modes:
  * layer-batched (default): each call covers all layers of the range in one
    launch -- valid whenever every layer's query is known before the step;
  * per-layer: the four calls per layer, layer after layer, as a model whose
    next layer's query depends on this layer's output must run them.
No call synchronises the host, so a whole step can be captured in a CUDA graph.

With ``overlap_groups`` = G > 1 (layer-batched steps, host tier), the ensure
is split into its state update (ssa_ensure_remap_bind, all layers) and the
host-link copy (ssa_fetch_misses), issued per range of layers; the attention
over a range runs on a second stream as soon as that range's copy is done, so
it overlaps the next range's copy.  The residency state, lists and pool bytes
are those of the plain step; the attention splits each range's units over its
CTAs by the range's size, so its outputs can differ from the all-layer launch
by the rounding of a different merge order.

With ``preload_width`` > 0 (layer-batched steps), every step also issues the
top-k preload (ssa_prefetch_pages) on a second stream once its remap is done:
the next step's likely pages are fetched while this step's attention and the
next step's indexer run, and the next step's ensure waits for it.  The
step's scores alternate between two buffers so that the preload reads one
while the next indexer writes the other.
"""
from __future__ import annotations

import math

import torch

from . import (KVCache, Layout, ssa_ensure_remap, ssa_ensure_remap_bind,
               ssa_ensure_remap_deferred, ssa_ensure_remap_shared, ssa_ensure_resident,
               ssa_fetch_misses, ssa_index_topk, ssa_lru_init, ssa_prefetch_pages,
               ssa_remap_block_table, ssa_sparse_paged_decode, ssa_sparse_paged_decode_fetch,
               ssa_store_kv_mirror, ssa_workspace_size)


def split_layers(n_layers: int, groups: int):
    """`groups` contiguous ranges of near-equal size covering [0, n_layers),
    the larger ones first, as (layer0, n); groups is clamped to [1, n_layers]."""
    G = max(1, min(int(groups), n_layers))
    sizes = [n_layers // G + (1 if i < n_layers % G else 0) for i in range(G)]
    starts = [sum(sizes[:i]) for i in range(G)]
    return list(zip(starts, sizes))


class DecodeRunner:
    def __init__(self, layout: Layout, host_tier: bool, identity: bool, block_table, seq_lens,
                 device="cuda", preload_width: int = 0, shared_residency: bool = False,
                 fetch_in_attention: bool = False, graphs: bool = False,
                 overlap_groups: int = 0):
        self.layout = layout
        self.cache = KVCache(layout, host_tier, device)
        L, B, W = layout.n_layers, layout.batch, layout.max_sel
        i32 = torch.int32
        self.block_table = torch.as_tensor(block_table, dtype=i32).to(device).contiguous()
        self.seq_lens = torch.as_tensor(seq_lens, dtype=i32).to(device).contiguous()
        self.sel = torch.full((L, B, W), -1, dtype=i32, device=device)
        self.n_sel = torch.zeros((L, B), dtype=i32, device=device)
        self.phys = torch.full((L, B, W), -1, dtype=i32, device=device)
        self.scores = torch.zeros((L, B, layout.max_pages), dtype=i32, device=device)
        self.miss_page = torch.full((L, B * W), -1, dtype=i32, device=device)
        self.miss_slot = torch.full((L, B * W), -1, dtype=i32, device=device)
        self.n_miss = torch.zeros((L,), dtype=i32, device=device)
        self.out = torch.zeros((L, B, layout.n_q_heads, layout.head_dim), dtype=torch.bfloat16,
                               device=device)
        self.status = torch.zeros((1,), dtype=i32, device=device)
        # zeroed once: the attention keeps split tickets in it and leaves them zero
        self.ws = torch.zeros((max(ssa_workspace_size(layout), 256),), dtype=torch.uint8,
                              device=device)
        self.sm_scale = 1.0 / math.sqrt(layout.head_dim)
        ssa_lru_init(self.cache, identity)
        # one LRU state for all layers (the first layer's), each miss copied
        # for every layer; layer-batched steps only
        self.shared_residency = bool(shared_residency)
        # misses fetched inside the attention (ssa_ensure_remap_deferred +
        # ssa_sparse_paged_decode_fetch) instead of by a copy before it
        self.fetch_in_attention = bool(fetch_in_attention) and host_tier
        self.preload_width = 0
        if preload_width:
            self.enable_preload(preload_width)
        # layer-batched steps as CUDA graph replays, one per q buffer (see step)
        self.graphs = bool(graphs)
        self._graphs = {}
        self.host_tier = bool(host_tier)
        self.overlap_groups = int(overlap_groups)

    def enable_preload(self, width: int):
        """Issue the top-k preload of `width` pages per request with every
        later layer-batched step (0 turns it off)."""
        self.preload_width = int(width)
        if not self.preload_width or hasattr(self, "side"):
            return
        L, B, W = self.layout.n_layers, self.layout.batch, self.layout.max_sel
        dev, i32 = self.scores.device, torch.int32
        self.scores_alt = torch.zeros_like(self.scores)
        self.fetch_page = torch.full((L, B * W), -1, dtype=i32, device=dev)
        self.fetch_slot = torch.full((L, B * W), -1, dtype=i32, device=dev)
        self.n_fetch = torch.zeros((L,), dtype=i32, device=dev)
        self.side = torch.cuda.Stream(device=dev)
        self.ev_remap = torch.cuda.Event()
        self.ev_preload = torch.cuda.Event()
        self.n_steps = 0

    # write path ---------------------------------------------------------------
    def store(self, layer0: int, n_layers: int, k, v, pos):
        """k, v: bf16 [n_layers][T][Hkv][D] on the device; pos: int64 [T]."""
        ssa_store_kv_mirror(self.cache, layer0, n_layers, k, v, pos, self.status)

    # one decode step ------------------------------------------------------------
    def _calls(self, q, layer0: int, n_layers: int, keep_scores: bool, fused: bool):
        sl = slice(layer0, layer0 + n_layers)
        c = self.cache
        ssa_index_topk(c, layer0, n_layers, q, self.block_table, self.seq_lens, self.sel[sl],
                       self.n_sel[sl], self.scores[sl] if keep_scores else None, self.status,
                       self.ws)
        if fused and self.shared_residency:
            ssa_ensure_remap_shared(c, layer0, n_layers, self.sel[sl], self.block_table,
                                    self.phys[sl], self.miss_page[sl], self.miss_slot[sl],
                                    self.n_miss[sl], self.status, self.ws)
        elif fused and self.fetch_in_attention:
            ssa_ensure_remap_deferred(c, layer0, n_layers, self.sel[sl], self.block_table,
                                      self.phys[sl], self.miss_page[sl], self.miss_slot[sl],
                                      self.n_miss[sl], self.status, self.ws)
            ssa_sparse_paged_decode_fetch(c, layer0, n_layers, q, self.sel[sl], self.phys[sl],
                                          self.block_table, self.seq_lens, self.sm_scale,
                                          self.out[sl], self.status, self.ws)
            return
        elif fused:
            ssa_ensure_remap(c, layer0, n_layers, self.sel[sl], self.block_table, self.phys[sl],
                             self.miss_page[sl], self.miss_slot[sl], self.n_miss[sl],
                             self.status, self.ws)
        else:
            ssa_ensure_resident(c, layer0, n_layers, self.sel[sl], self.block_table,
                                self.miss_page[sl], self.miss_slot[sl], self.n_miss[sl],
                                self.status, self.ws)
            ssa_remap_block_table(c, layer0, n_layers, self.sel[sl], self.block_table,
                                  self.phys[sl], self.status)
        ssa_sparse_paged_decode(c, layer0, n_layers, q, self.sel[sl], self.phys[sl],
                                self.seq_lens, self.sm_scale, self.out[sl], self.status, self.ws)

    def layer_groups(self):
        """The contiguous layer ranges of an overlapped step, as (layer0, n)."""
        return split_layers(self.layout.n_layers, self.overlap_groups)

    def _overlap_calls(self, q, keep_scores: bool):
        L, c = self.layout.n_layers, self.cache
        if not hasattr(self, "att_stream"):
            self.att_stream = torch.cuda.Stream(device=self.sel.device)
            self.ev_fetched = [torch.cuda.Event() for _ in range(L)]
            self.ev_attended = torch.cuda.Event()
        main, att = torch.cuda.current_stream(), self.att_stream
        ssa_index_topk(c, 0, L, q, self.block_table, self.seq_lens, self.sel, self.n_sel,
                       self.scores if keep_scores else None, self.status, self.ws)
        ssa_ensure_remap_bind(c, 0, L, self.sel, self.block_table, self.phys, self.miss_page,
                              self.miss_slot, self.n_miss, self.status)
        for g, (l0, n) in enumerate(self.layer_groups()):
            sl = slice(l0, l0 + n)
            ssa_fetch_misses(c, l0, n, self.miss_page[sl], self.miss_slot[sl], self.n_miss[sl],
                             self.status)
            self.ev_fetched[g].record(main)
            att.wait_event(self.ev_fetched[g])
            # the attentions run one after another on att: one workspace
            ssa_sparse_paged_decode(c, l0, n, q[sl], self.sel[sl], self.phys[sl], self.seq_lens,
                                    self.sm_scale, self.out[sl], self.status, self.ws,
                                    stream=att)
        self.ev_attended.record(att)
        main.wait_event(self.ev_attended)

    def _batched_calls(self, q, keep_scores: bool):
        overlap = (self.overlap_groups > 1 and self.host_tier and not self.shared_residency
                   and not self.fetch_in_attention)
        if overlap:
            self._overlap_calls(q, keep_scores)
        else:
            self._calls(q, 0, self.layout.n_layers, keep_scores, fused=True)

    def _preload_step(self, q):
        L, c = self.layout.n_layers, self.cache
        scores = self.scores if self.n_steps % 2 == 0 else self.scores_alt
        main = torch.cuda.current_stream()
        ssa_index_topk(c, 0, L, q, self.block_table, self.seq_lens, self.sel, self.n_sel, scores,
                       self.status, self.ws)
        main.wait_event(self.ev_preload)          # the previous step's preload is done
        ssa_ensure_remap(c, 0, L, self.sel, self.block_table, self.phys, self.miss_page,
                         self.miss_slot, self.n_miss, self.status, self.ws)
        self.ev_remap.record(main)
        ssa_sparse_paged_decode(c, 0, L, q, self.sel, self.phys, self.seq_lens, self.sm_scale,
                                self.out, self.status, self.ws)
        self.side.wait_event(self.ev_remap)
        ssa_prefetch_pages(c, 0, L, scores, self.block_table, self.seq_lens, self.preload_width,
                           self.fetch_page, self.fetch_slot, self.n_fetch, self.status, self.ws,
                           stream=self.side)
        self.ev_preload.record(self.side)
        self.last_scores = scores
        self.n_steps += 1

    def step(self, q, per_layer: bool = False, keep_scores: bool = False):
        """q: bf16 [n_layers][B][Hq][D] on the device, all layers of the cache.
        Layer-batched steps take the ensure and the remap in one call
        (ssa_ensure_remap), or, with `overlap_groups` > 1 on a host tier, in
        a state call and one copy call per layer range with the attention of
        each range overlapping the next range's copy; per-layer steps make
        the four separate calls.
        With `graphs` set, a layer-batched step (without the preload) is one
        CUDA graph replay, captured on the first call with that q buffer: a
        serving loop that reuses its query buffer pays the launch path once."""
        L = self.layout.n_layers
        if self.preload_width and not per_layer:
            self._preload_step(q)
        elif per_layer:
            for l in range(L):
                self._calls(q[l:l + 1], l, 1, keep_scores, fused=False)
        elif self.graphs:
            key = (q.data_ptr(), tuple(q.shape), keep_scores)
            g = self._graphs.get(key)
            if g is None:
                # this call's step runs eagerly (and sets the kernels'
                # attributes); the capture only records the same launches
                self._batched_calls(q, keep_scores)
                torch.cuda.current_stream().synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    self._batched_calls(q, keep_scores)
                self._graphs[key] = g
            else:
                g.replay()
        else:
            self._batched_calls(q, keep_scores)
        return self.out
