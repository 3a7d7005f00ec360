"""DecodeRunner: the decode step over a layer range, as a user calls it.

Holds the cache, the per-step device buffers and the workspace, and issues the
four calls of one decode step (index + select, ensure, remap, attention) on
the current stream.  Two launch modes:
  * layer-batched (default): each call covers all layers of the range in one
    launch -- valid whenever every layer's query is known before the step;
  * per-layer: the four calls per layer, layer after layer, as a model whose
    next layer's query depends on this layer's output must run them.
No call synchronises the host, so a whole step can be captured in a CUDA graph.
"""
from __future__ import annotations

import math

import torch

from . import (KVCache, Layout, ssa_ensure_resident, ssa_index_topk, ssa_lru_init,
               ssa_remap_block_table, ssa_sparse_paged_decode, ssa_store_kv_mirror,
               ssa_workspace_size)


class DecodeRunner:
    def __init__(self, layout: Layout, host_tier: bool, identity: bool, block_table, seq_lens,
                 device="cuda"):
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

    # write path ---------------------------------------------------------------
    def store(self, layer0: int, n_layers: int, k, v, pos):
        """k, v: bf16 [n_layers][T][Hkv][D] on the device; pos: int64 [T]."""
        ssa_store_kv_mirror(self.cache, layer0, n_layers, k, v, pos, self.status)

    # one decode step ------------------------------------------------------------
    def _calls(self, q, layer0: int, n_layers: int, keep_scores: bool):
        sl = slice(layer0, layer0 + n_layers)
        c = self.cache
        ssa_index_topk(c, layer0, n_layers, q, self.block_table, self.seq_lens, self.sel[sl],
                       self.n_sel[sl], self.scores[sl] if keep_scores else None, self.status,
                       self.ws)
        ssa_ensure_resident(c, layer0, n_layers, self.sel[sl], self.block_table,
                            self.miss_page[sl], self.miss_slot[sl], self.n_miss[sl], self.status,
                            self.ws)
        ssa_remap_block_table(c, layer0, n_layers, self.sel[sl], self.block_table, self.phys[sl],
                              self.status)
        ssa_sparse_paged_decode(c, layer0, n_layers, q, self.sel[sl], self.phys[sl],
                                self.seq_lens, self.sm_scale, self.out[sl], self.status, self.ws)

    def step(self, q, per_layer: bool = False, keep_scores: bool = False):
        """q: bf16 [n_layers][B][Hq][D] on the device, all layers of the cache."""
        L = self.layout.n_layers
        if per_layer:
            for l in range(L):
                self._calls(q[l:l + 1], l, 1, keep_scores)
        else:
            self._calls(q, 0, L, keep_scores)
        return self.out
