"""GB300 (sm_103a) sparse-attention decode step: Python binding of libssa_gb300.so.

The five calls of the decode step keep their C names and only marshal
arguments (torch tensors -> raw pointers, the current CUDA stream); every step
of the path runs in the library's CUDA kernels.  PyTorch provides device
memory, pinned host memory and streams.  There is no CPU fallback: if the
library is missing or no GPU is present the calls raise.

    ssa_store_kv_mirror      write path: quantise/store K,V, mirror, slab
    ssa_index_topk           int8 indexer + top-k page selection
    ssa_ensure_resident      device LRU + miss fetch from the host mirror
    ssa_remap_block_table    logical -> physical block table
    ssa_sparse_paged_decode  attention over the selected pages
    ssa_prefetch_pages       top-k preload of the next step's likely pages
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libssa_gb300.so")

SSA_KV_BF16 = 0
SSA_KV_FP8_E4M3 = 1

ST_DROP, ST_BAD_ID, ST_MISS_NO_MIRROR, ST_UNRESOLVED, ST_BAD_POS, ST_TIMEOUT = 1, 2, 4, 8, 16, 32
ST_INTERNAL = 64

EXPORTS = ("ssa_workspace_size", "ssa_lru_init", "ssa_store_kv_mirror", "ssa_index_topk",
           "ssa_ensure_resident", "ssa_remap_block_table", "ssa_sparse_paged_decode",
           "ssa_status_str", "ssa_last_cuda_error", "ssa_launch_count",
           "ssa_index_topk_static_scratch", "ssa_selftest_bounded_wait", "ssa_host_read_probe",
           "ssa_prefetch_pages", "ssa_ensure_remap", "ssa_sparse_paged_decode_host_tail",
           "ssa_ensure_remap_shared", "ssa_ensure_remap_deferred",
           "ssa_sparse_paged_decode_fetch", "ssa_ensure_remap_bind", "ssa_fetch_misses")


class SsaError(RuntimeError):
    def __init__(self, code: int, msg: str, cuda: int = 0):
        super().__init__(f"{msg} (code {code}" + (f", cudaError {cuda})" if cuda else ")"))
        self.code = code


class SsaLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "page_size", "n_q_heads", "n_kv_heads", "head_dim", "kv_dtype", "n_layers",
        "logical_pages", "pool_slots", "batch", "max_pages", "block_topk", "max_sel")]


class SsaCache(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "k_pool", "v_pool", "k_scale", "v_scale", "k_mirror", "v_mirror", "k_scale_mirror",
        "v_scale_mirror", "slab", "slab_scale", "slab_sum", "slab_cnt", "slot_of", "page_of",
        "last_use", "clock")]


_lib = None


def lib():
    """The loaded C-ABI library (built by build.py); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run sparse_attention_decode_indexer_gb300/build.py")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, P = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER
        L.ssa_workspace_size.restype = ctypes.c_size_t
        L.ssa_workspace_size.argtypes = [P(SsaLayout)]
        L.ssa_lru_init.restype = i32
        L.ssa_lru_init.argtypes = [P(SsaLayout), P(SsaCache), i32, vp]
        L.ssa_store_kv_mirror.restype = i32
        L.ssa_store_kv_mirror.argtypes = [P(SsaLayout), P(SsaCache), i32, i32, vp, vp, vp, i32,
                                          vp, vp]
        L.ssa_index_topk.restype = i32
        L.ssa_index_topk.argtypes = [P(SsaLayout), P(SsaCache), i32, i32] + [vp] * 9
        L.ssa_ensure_resident.restype = i32
        L.ssa_ensure_resident.argtypes = [P(SsaLayout), P(SsaCache), i32, i32] + [vp] * 8
        L.ssa_remap_block_table.restype = i32
        L.ssa_remap_block_table.argtypes = [P(SsaLayout), P(SsaCache), i32, i32] + [vp] * 5
        L.ssa_sparse_paged_decode.restype = i32
        L.ssa_sparse_paged_decode.argtypes = ([P(SsaLayout), P(SsaCache), i32, i32, vp, vp, vp, vp,
                                               ctypes.c_float, vp, vp, vp, vp])
        L.ssa_status_str.restype = ctypes.c_char_p
        L.ssa_status_str.argtypes = [i32]
        L.ssa_last_cuda_error.restype = i32
        L.ssa_last_cuda_error.argtypes = []
        L.ssa_launch_count.restype = ctypes.c_longlong
        L.ssa_launch_count.argtypes = []
        L.ssa_selftest_bounded_wait.restype = i32
        L.ssa_selftest_bounded_wait.argtypes = [vp, vp]
        L.ssa_sparse_paged_decode_host_tail.restype = i32
        L.ssa_sparse_paged_decode_host_tail.argtypes = ([P(SsaLayout), P(SsaCache), i32, i32, vp,
                                                         vp, vp, vp, ctypes.c_float, vp, vp, vp,
                                                         vp])
        L.ssa_ensure_remap_deferred.restype = i32
        L.ssa_ensure_remap_deferred.argtypes = [P(SsaLayout), P(SsaCache), i32, i32] + [vp] * 9
        L.ssa_sparse_paged_decode_fetch.restype = i32
        L.ssa_sparse_paged_decode_fetch.argtypes = ([P(SsaLayout), P(SsaCache), i32, i32, vp, vp,
                                                     vp, vp, vp, ctypes.c_float, vp, vp, vp, vp])
        L.ssa_ensure_remap_bind.restype = i32
        L.ssa_ensure_remap_bind.argtypes = [P(SsaLayout), P(SsaCache), i32, i32] + [vp] * 8
        L.ssa_fetch_misses.restype = i32
        L.ssa_fetch_misses.argtypes = [P(SsaLayout), P(SsaCache), i32, i32] + [vp] * 5
        L.ssa_ensure_remap_shared.restype = i32
        L.ssa_ensure_remap_shared.argtypes = [P(SsaLayout), P(SsaCache), i32, i32] + [vp] * 9
        L.ssa_ensure_remap.restype = i32
        L.ssa_ensure_remap.argtypes = [P(SsaLayout), P(SsaCache), i32, i32] + [vp] * 9
        L.ssa_prefetch_pages.restype = i32
        L.ssa_prefetch_pages.argtypes = ([P(SsaLayout), P(SsaCache), i32, i32, vp, vp, vp, i32]
                                         + [vp] * 6)
        L.ssa_host_read_probe.restype = i32
        L.ssa_host_read_probe.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        _lib = L
    return _lib


def status_str(code: int) -> str:
    return lib().ssa_status_str(int(code)).decode()


def _check(code: int):
    if code != 0:
        raise SsaError(code, status_str(code), lib().ssa_last_cuda_error())


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def max_sel_pages(block_topk: int) -> int:
    """Selection width and per-request pool reservation: 2*block_topk + 8."""
    return 2 * block_topk + 8


# ---------------------------------------------------------------------------
# layout and cache (device memory through torch; mirror in pinned host memory)
# ---------------------------------------------------------------------------

@dataclass
class Layout:
    page_size: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    fp8: bool
    n_layers: int
    logical_pages: int
    pool_slots: int
    batch: int
    max_pages: int
    block_topk: int

    @property
    def max_sel(self) -> int:
        return max_sel_pages(self.block_topk)

    def c(self) -> SsaLayout:
        return SsaLayout(self.page_size, self.n_q_heads, self.n_kv_heads, self.head_dim,
                         SSA_KV_FP8_E4M3 if self.fp8 else SSA_KV_BF16, self.n_layers,
                         self.logical_pages, self.pool_slots, self.batch, self.max_pages,
                         self.block_topk, self.max_sel)


def ssa_workspace_size(layout: Layout) -> int:
    lay = layout.c()
    return int(lib().ssa_workspace_size(ctypes.byref(lay)))


class KVCache:
    """Owns the tensors behind one ssa_cache: the paged pool and its scales,
    the optional pinned host mirror, the indexer slab and the LRU state.
    Pool and mirror start zeroed so that rows never written (the tail of a
    request's last page) hold defined bytes; the kernels do not rely on it."""

    def __init__(self, layout: Layout, host_tier: bool, device="cuda"):
        self.layout = layout
        L, Lp, S = layout.n_layers, layout.logical_pages, layout.pool_slots
        H, P, D = layout.n_kv_heads, layout.page_size, layout.head_dim
        esz = 1 if layout.fp8 else 2
        pb = H * P * D * esz
        u8 = torch.uint8
        self.k_pool = torch.zeros((L, S, pb), dtype=u8, device=device)
        self.v_pool = torch.zeros((L, S, pb), dtype=u8, device=device)
        if layout.fp8:
            self.k_scale = torch.zeros((L, S, P), dtype=torch.float32, device=device)
            self.v_scale = torch.zeros((L, S, P), dtype=torch.float32, device=device)
        else:
            self.k_scale = self.v_scale = None
        if host_tier:
            self.k_mirror = torch.zeros((L, Lp, pb), dtype=u8, pin_memory=True)
            self.v_mirror = torch.zeros((L, Lp, pb), dtype=u8, pin_memory=True)
            if layout.fp8:
                self.k_scale_mirror = torch.zeros((L, Lp, P), dtype=torch.float32, pin_memory=True)
                self.v_scale_mirror = torch.zeros((L, Lp, P), dtype=torch.float32, pin_memory=True)
            else:
                self.k_scale_mirror = self.v_scale_mirror = None
        else:
            self.k_mirror = self.v_mirror = self.k_scale_mirror = self.v_scale_mirror = None
        self.slab = torch.empty((L, Lp, H * D), dtype=torch.int8, device=device)
        self.slab_scale = torch.empty((L, Lp), dtype=torch.float32, device=device)
        self.slab_sum = torch.empty((L, Lp, H * D), dtype=torch.float32, device=device)
        self.slab_cnt = torch.empty((L, Lp), dtype=torch.int32, device=device)
        self.slot_of = torch.empty((L, Lp), dtype=torch.int32, device=device)
        self.page_of = torch.empty((L, S), dtype=torch.int32, device=device)
        self.last_use = torch.empty((L, S), dtype=torch.int32, device=device)
        self.clock = torch.empty((L,), dtype=torch.int32, device=device)
        self._c = SsaCache(*[ctypes.c_void_p(t.data_ptr()) if t is not None else None for t in (
            self.k_pool, self.v_pool, self.k_scale, self.v_scale, self.k_mirror, self.v_mirror,
            self.k_scale_mirror, self.v_scale_mirror, self.slab, self.slab_scale, self.slab_sum,
            self.slab_cnt, self.slot_of, self.page_of, self.last_use, self.clock)])
        self._lay = layout.c()

    @property
    def c(self) -> SsaCache:
        return self._c


# ---------------------------------------------------------------------------
# the calls
# ---------------------------------------------------------------------------

def ssa_lru_init(cache: KVCache, identity: bool, stream=None):
    _check(lib().ssa_lru_init(ctypes.byref(cache._lay), ctypes.byref(cache.c), int(identity),
                              _stream(stream)))


def ssa_store_kv_mirror(cache: KVCache, layer0: int, n_layers: int, k, v, pos, status,
                        stream=None):
    """k, v: bf16 [n_layers][T][Hkv][D]; pos: int64 [T] logical token ids."""
    T = int(pos.shape[0])
    _check(lib().ssa_store_kv_mirror(ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0,
                                     n_layers, _ptr(k), _ptr(v), _ptr(pos), T, _ptr(status),
                                     _stream(stream)))


def ssa_index_topk(cache: KVCache, layer0: int, n_layers: int, q, block_table, seq_lens, sel,
                   n_sel, scores, status, ws, stream=None):
    _check(lib().ssa_index_topk(ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0,
                                n_layers, _ptr(q), _ptr(block_table), _ptr(seq_lens), _ptr(sel),
                                _ptr(n_sel), _ptr(scores), _ptr(status), _ptr(ws),
                                _stream(stream)))


def ssa_ensure_resident(cache: KVCache, layer0: int, n_layers: int, sel, block_table, miss_page,
                        miss_slot, n_miss, status, ws, stream=None):
    _check(lib().ssa_ensure_resident(ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0,
                                     n_layers, _ptr(sel), _ptr(block_table), _ptr(miss_page),
                                     _ptr(miss_slot), _ptr(n_miss), _ptr(status), _ptr(ws),
                                     _stream(stream)))


def ssa_ensure_remap(cache: KVCache, layer0: int, n_layers: int, sel, block_table, phys,
                     miss_page, miss_slot, n_miss, status, ws, stream=None):
    """ssa_ensure_resident that also writes the remapped table (one launch fewer)."""
    _check(lib().ssa_ensure_remap(ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0,
                                  n_layers, _ptr(sel), _ptr(block_table), _ptr(phys),
                                  _ptr(miss_page), _ptr(miss_slot), _ptr(n_miss), _ptr(status),
                                  _ptr(ws), _stream(stream)))


def ssa_ensure_remap_bind(cache: KVCache, layer0: int, n_layers: int, sel, block_table, phys,
                          miss_page, miss_slot, n_miss, status, stream=None):
    """ssa_ensure_remap without the copy: state, phys and the miss lists are
    final; ssa_fetch_misses copies the misses, per layer range, afterwards."""
    _check(lib().ssa_ensure_remap_bind(ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0,
                                       n_layers, _ptr(sel), _ptr(block_table), _ptr(phys),
                                       _ptr(miss_page), _ptr(miss_slot), _ptr(n_miss),
                                       _ptr(status), _stream(stream)))


def ssa_fetch_misses(cache: KVCache, layer0: int, n_layers: int, miss_page, miss_slot, n_miss,
                     status, stream=None):
    """Copy the listed misses of layers [layer0, layer0 + n_layers) mirror ->
    slot; the lists are those ssa_ensure_remap_bind wrote for these layers."""
    _check(lib().ssa_fetch_misses(ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0,
                                  n_layers, _ptr(miss_page), _ptr(miss_slot), _ptr(n_miss),
                                  _ptr(status), _stream(stream)))


def ssa_ensure_remap_deferred(cache: KVCache, layer0: int, n_layers: int, sel, block_table, phys,
                              miss_page, miss_slot, n_miss, status, ws, stream=None):
    """The ensure's state update and remap without the copy: misses marked
    -2 - slot in phys, for ssa_sparse_paged_decode_fetch to fetch."""
    _check(lib().ssa_ensure_remap_deferred(ctypes.byref(cache._lay), ctypes.byref(cache.c),
                                           layer0, n_layers, _ptr(sel), _ptr(block_table),
                                           _ptr(phys), _ptr(miss_page), _ptr(miss_slot),
                                           _ptr(n_miss), _ptr(status), _ptr(ws), _stream(stream)))


def ssa_sparse_paged_decode_fetch(cache: KVCache, layer0: int, n_layers: int, q, sel, phys,
                                  block_table, seq_lens, sm_scale: float, out, status, ws,
                                  stream=None):
    """Attention that fetches the pages ssa_ensure_remap_deferred marked from
    the host mirror and writes them into their slots as it goes."""
    _check(lib().ssa_sparse_paged_decode_fetch(
        ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0, n_layers, _ptr(q), _ptr(sel),
        _ptr(phys), _ptr(block_table), _ptr(seq_lens), float(sm_scale), _ptr(out), _ptr(status),
        _ptr(ws), _stream(stream)))


def ssa_ensure_remap_shared(cache: KVCache, layer0: int, n_layers: int, sel, block_table, phys,
                            miss_page, miss_slot, n_miss, status, ws, stream=None):
    """One residency for the layer range (layer0's state): the union of the
    layers' selections ensured, each miss copied for every layer, phys for
    every layer."""
    _check(lib().ssa_ensure_remap_shared(ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0,
                                         n_layers, _ptr(sel), _ptr(block_table), _ptr(phys),
                                         _ptr(miss_page), _ptr(miss_slot), _ptr(n_miss),
                                         _ptr(status), _ptr(ws), _stream(stream)))


def ssa_prefetch_pages(cache: KVCache, layer0: int, n_layers: int, scores, block_table,
                       seq_lens, width: int, fetch_page, fetch_slot, n_fetch, status, ws,
                       stream=None):
    """Top-k preload after a step's ensure: fetch the top (width-1) pages plus
    the last page of each request by that step's scores ahead of the next."""
    _check(lib().ssa_prefetch_pages(ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0,
                                    n_layers, _ptr(scores), _ptr(block_table), _ptr(seq_lens),
                                    int(width), _ptr(fetch_page), _ptr(fetch_slot),
                                    _ptr(n_fetch), _ptr(status), _ptr(ws), _stream(stream)))


def ssa_remap_block_table(cache: KVCache, layer0: int, n_layers: int, sel, block_table, phys,
                          status, stream=None):
    _check(lib().ssa_remap_block_table(ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0,
                                       n_layers, _ptr(sel), _ptr(block_table), _ptr(phys),
                                       _ptr(status), _stream(stream)))


def ssa_sparse_paged_decode(cache: KVCache, layer0: int, n_layers: int, q, sel, phys, seq_lens,
                            sm_scale: float, out, status, ws, stream=None):
    _check(lib().ssa_sparse_paged_decode(ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0,
                                         n_layers, _ptr(q), _ptr(sel), _ptr(phys),
                                         _ptr(seq_lens), float(sm_scale), _ptr(out),
                                         _ptr(status), _ptr(ws), _stream(stream)))


def ssa_sparse_paged_decode_host_tail(cache: KVCache, layer0: int, n_layers: int, q, sel,
                                      block_table, seq_lens, sm_scale: float, out, status, ws,
                                      stream=None):
    """Attention over the selected pages, non-resident ones read straight from
    the pinned host mirror (no ensure, no copy)."""
    _check(lib().ssa_sparse_paged_decode_host_tail(
        ctypes.byref(cache._lay), ctypes.byref(cache.c), layer0, n_layers, _ptr(q), _ptr(sel),
        _ptr(block_table), _ptr(seq_lens), float(sm_scale), _ptr(out), _ptr(status), _ptr(ws),
        _stream(stream)))


def ssa_selftest_bounded_wait(status, stream=None):
    """One CTA waits on an mbarrier nothing arrives on; the bounded wait gives
    up after about a second and sets ST_TIMEOUT in ``status``."""
    _check(lib().ssa_selftest_bounded_wait(_ptr(status), _stream(stream)))


def ssa_host_read_probe(src, dst, offsets, chunk_bytes: int, loads_per_thread: int = 8,
                        stream=None):
    """Copy chunks of ``src`` (pinned host or device) at the int64 byte
    ``offsets`` (a device tensor) into ``dst`` with SM loads: the host link's
    rate for the access pattern of the miss fetch."""
    _check(lib().ssa_host_read_probe(_ptr(src), _ptr(dst), _ptr(offsets), int(offsets.numel()),
                                     int(chunk_bytes), int(loads_per_thread), _stream(stream)))


def launch_count() -> int:
    return int(lib().ssa_launch_count())
