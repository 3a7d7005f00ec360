"""Plain CPU oracle for the sparse-attention decode step (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never does, and this package
never imports the library: the two share no code.  The arithmetic lives in
``ssa_oracle.c`` (plain C, fp64 attention, built with ``-O2
-ffp-contract=off``; independent loops spread over the cores by OpenMP,
with results independent of the thread count); this module only builds it, holds the oracle's own
copy of the KV state in numpy arrays and marshals arguments.

State layout per layer (the oracle's own, plain [P][D] for both K and V):
    pool K/V codes   [S][Hkv][P][D]  (bf16 as uint16 bits, or e4m3 bytes)
    pool scales      [S][P] fp32 (fp8 only)
    mirror           [Lp][Hkv][P][D], mirror scales [Lp][P]
    slab             [Lp][Hkv][D] int8, slab scale [Lp] fp32
    slab sum/count   [Lp][Hkv][D] fp32, [Lp] int32
    slot_of [Lp], page_of [S], last_use [S], clock
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssa_oracle.c")
_HDR = os.path.join(_HERE, "ssa_oracle.h")
_LIB = os.path.join(_HERE, "libssa_oracle.so")
_lib = None

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (host architecture) if it is missing or stale.
    With OpenMP where the compiler has it (independent loops on every core;
    the results are the same at any thread count), else single-threaded."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR, __file__))
    if force or stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        r = subprocess.run(["gcc", *CFLAGS, "-fopenmp", _SRC, "-o", tmp, "-lm"],
                           capture_output=True, text=True)
        if r.returncode != 0:
            subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("P", "Hq", "Hkv", "D", "fp8", "Lp", "S", "B", "n_max", "k", "W")]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp = ctypes.c_void_p
        i32 = ctypes.c_int
        lib.or_e4m3_encode.restype = ctypes.c_uint8
        lib.or_e4m3_encode.argtypes = [ctypes.c_float]
        lib.or_e4m3_decode.restype = ctypes.c_double
        lib.or_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.or_store.restype = i32
        lib.or_store.argtypes = [vp] * 17 + [i32]
        lib.or_index_scores.restype = i32
        lib.or_index_scores.argtypes = [vp] * 6
        lib.or_select.restype = i32
        lib.or_select.argtypes = [vp] * 5
        lib.or_ensure.restype = i32
        lib.or_ensure.argtypes = [vp] * 18
        lib.or_remap.restype = i32
        lib.or_remap.argtypes = [vp] * 5
        lib.or_decode.restype = None
        lib.or_decode.argtypes = [vp] * 9 + [ctypes.c_double, vp]
        lib.or_ensure_shared.restype = i32
        lib.or_ensure_shared.argtypes = [vp, i32] + [vp] * 17
        lib.or_prefetch.restype = i32
        lib.or_prefetch.argtypes = [vp, i32] + [vp] * 18
        lib.or_set_threads.restype = None
        lib.or_set_threads.argtypes = [i32]
        lib.or_threads.restype = i32
        lib.or_threads.argtypes = []
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def set_threads(n: int) -> None:
    """Threads for the oracle's independent loops (n <= 0: every core).  The
    results are the same at any count."""
    _load().or_set_threads(int(n))


def threads() -> int:
    return int(_load().or_threads())


def e4m3_encode(x: float) -> int:
    return int(_load().or_e4m3_encode(float(x)))


def e4m3_decode(c: int) -> float:
    return float(_load().or_e4m3_decode(int(c)))


def max_sel_pages(block_topk: int) -> int:
    """Fixed selection width: 2*block_topk + 8 (FreeToken PR #499, "Design",
    anti-silent-corruption bullet)."""
    return 2 * block_topk + 8


@dataclass
class OracleLayout:
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
    max_sel_override: int | None = None   # tests of the LRU alone use a narrow width

    @property
    def max_sel(self) -> int:
        if self.max_sel_override is not None:
            return self.max_sel_override
        return max_sel_pages(self.block_topk)

    def c(self) -> _Layout:
        return _Layout(self.page_size, self.n_q_heads, self.n_kv_heads, self.head_dim,
                       int(self.fp8), self.logical_pages, self.pool_slots, self.batch,
                       self.max_pages, self.block_topk, self.max_sel)


class OracleKV:
    """The oracle's own KV state for all layers, plus the five steps."""

    def __init__(self, lay: OracleLayout, host_tier: bool, identity: bool):
        self.lay = lay
        L, Lp, S = lay.n_layers, lay.logical_pages, lay.pool_slots
        H, P, D = lay.n_kv_heads, lay.page_size, lay.head_dim
        self.esz = 1 if lay.fp8 else 2
        pe = H * P * D * self.esz
        self.k_pool = np.zeros((L, S, pe), np.uint8)
        self.v_pool = np.zeros((L, S, pe), np.uint8)
        self.k_scale = np.zeros((L, S, P), np.float32)
        self.v_scale = np.zeros((L, S, P), np.float32)
        if host_tier:
            self.k_mirror = np.zeros((L, Lp, pe), np.uint8)
            self.v_mirror = np.zeros((L, Lp, pe), np.uint8)
            self.k_scale_m = np.zeros((L, Lp, P), np.float32)
            self.v_scale_m = np.zeros((L, Lp, P), np.float32)
        else:
            self.k_mirror = self.v_mirror = self.k_scale_m = self.v_scale_m = None
        self.slab = np.zeros((L, Lp, H * D), np.int8)
        self.slab_scale = np.zeros((L, Lp), np.float32)
        self.slab_sum = np.zeros((L, Lp, H * D), np.float32)
        self.slab_cnt = np.zeros((L, Lp), np.int32)
        self.slot_of = np.full((L, Lp), -1, np.int32)
        self.page_of = np.full((L, S), -1, np.int32)
        self.last_use = np.full((L, S), -1, np.int32)
        self.clock = np.zeros((L,), np.int32)
        if identity:
            n = min(Lp, S)
            self.slot_of[:, :n] = np.arange(n, dtype=np.int32)
            self.page_of[:, :n] = np.arange(n, dtype=np.int32)

    # -- helpers -------------------------------------------------------------
    def _mir(self, a, l):
        return None if a is None else a[l]

    # -- a0 ------------------------------------------------------------------
    def store(self, layer: int, k_bits: np.ndarray, v_bits: np.ndarray, pos: np.ndarray) -> int:
        lib, lay = _load(), self.lay.c()
        k = np.ascontiguousarray(k_bits, np.uint16)
        v = np.ascontiguousarray(v_bits, np.uint16)
        pos = np.ascontiguousarray(pos, np.int64)
        l = layer
        return lib.or_store(
            ctypes.byref(lay), _p(self.k_pool[l]), _p(self.v_pool[l]), _p(self.k_scale[l]),
            _p(self.v_scale[l]), _p(self._mir(self.k_mirror, l)), _p(self._mir(self.v_mirror, l)),
            _p(self._mir(self.k_scale_m, l)), _p(self._mir(self.v_scale_m, l)),
            _p(self.slab[l]), _p(self.slab_scale[l]), _p(self.slab_sum[l]), _p(self.slab_cnt[l]),
            _p(self.slot_of[l]), _p(k), _p(v), _p(pos), int(pos.shape[0]))

    # -- a1 + a2 -------------------------------------------------------------
    def index_topk(self, layer: int, q_bits: np.ndarray, bt: np.ndarray, seq_lens: np.ndarray):
        lib, lay = _load(), self.lay.c()
        B, nmax, W = self.lay.batch, self.lay.max_pages, self.lay.max_sel
        q = np.ascontiguousarray(q_bits, np.uint16)
        bt = np.ascontiguousarray(bt, np.int32)
        sl = np.ascontiguousarray(seq_lens, np.int32)
        scores = np.empty((B, nmax), np.int32)
        bad = lib.or_index_scores(ctypes.byref(lay), _p(self.slab[layer]), _p(q), _p(bt), _p(sl),
                                  _p(scores))
        sel = np.empty((B, W), np.int32)
        n_sel = np.empty((B,), np.int32)
        drops = lib.or_select(ctypes.byref(lay), _p(scores), _p(sl), _p(sel), _p(n_sel))
        return sel, n_sel, scores, drops, bad

    # -- a3 + a4 -------------------------------------------------------------
    def ensure(self, layer: int, sel: np.ndarray, bt: np.ndarray):
        lib, lay = _load(), self.lay.c()
        BW = self.lay.batch * self.lay.max_sel
        l = layer
        sel = np.ascontiguousarray(sel, np.int32)
        bt = np.ascontiguousarray(bt, np.int32)
        mp = np.empty((BW,), np.int32)
        ms = np.empty((BW,), np.int32)
        nm = np.zeros((1,), np.int32)
        clk = self.clock[l:l + 1]
        flags = lib.or_ensure(
            ctypes.byref(lay), _p(self.slot_of[l]), _p(self.page_of[l]), _p(self.last_use[l]),
            _p(clk), _p(sel), _p(bt), _p(self._mir(self.k_mirror, l)),
            _p(self._mir(self.v_mirror, l)), _p(self._mir(self.k_scale_m, l)),
            _p(self._mir(self.v_scale_m, l)), _p(self.k_pool[l]), _p(self.v_pool[l]),
            _p(self.k_scale[l]), _p(self.v_scale[l]), _p(mp), _p(ms), _p(nm))
        return mp, ms, int(nm[0]), flags

    # -- NEXT-2: one residency for a layer range ----------------------------
    def ensure_shared(self, layer0: int, n_layers: int, sel: np.ndarray, bt: np.ndarray):
        """Ensure the union of the layers' selections (sel [n][B][W]) on the
        first layer's LRU state; every miss copied for every layer of the
        range (or_ensure_shared)."""
        lib, lay = _load(), self.lay.c()
        n = n_layers
        l0, l1 = layer0, layer0 + n
        BW = self.lay.batch * self.lay.max_sel
        mp = np.empty((n * BW,), np.int32)
        ms = np.empty((n * BW,), np.int32)
        nm = np.zeros((1,), np.int32)
        mir = self.k_mirror is not None
        flags = lib.or_ensure_shared(
            ctypes.byref(lay), n, _p(self.slot_of[l0]), _p(self.page_of[l0]),
            _p(self.last_use[l0]), _p(self.clock[l0:l0 + 1]), _p(np.ascontiguousarray(sel, np.int32)),
            _p(np.ascontiguousarray(bt, np.int32)),
            _p(self.k_mirror[l0:l1] if mir else None), _p(self.v_mirror[l0:l1] if mir else None),
            _p(self.k_scale_m[l0:l1] if mir else None), _p(self.v_scale_m[l0:l1] if mir else None),
            _p(self.k_pool[l0:l1]), _p(self.v_pool[l0:l1]), _p(self.k_scale[l0:l1]),
            _p(self.v_scale[l0:l1]), _p(mp), _p(ms), _p(nm))
        return mp, ms, int(nm[0]), flags

    def remap_shared(self, layer0: int, layer: int, sel: np.ndarray, bt: np.ndarray):
        """Remap of one layer's selection through the shared state (the first
        layer's slot_of)."""
        lib, lay = _load(), self.lay.c()
        phys = np.empty((self.lay.batch, self.lay.max_sel), np.int32)
        unresolved = lib.or_remap(ctypes.byref(lay), _p(self.slot_of[layer0]),
                                  _p(np.ascontiguousarray(sel, np.int32)),
                                  _p(np.ascontiguousarray(bt, np.int32)), _p(phys))
        return phys, unresolved

    # -- NEXT-1: top-k preload ----------------------------------------------
    def prefetch(self, layer: int, width: int, scores: np.ndarray, seq_lens: np.ndarray,
                 bt: np.ndarray):
        """Fetch ahead the top (width-1) pages + last page of each request by a
        step's scores, after that step's ensure (or_prefetch)."""
        lib, lay = _load(), self.lay.c()
        BW = self.lay.batch * self.lay.max_sel
        l = layer
        mp = np.empty((BW,), np.int32)
        ms = np.empty((BW,), np.int32)
        nm = np.zeros((1,), np.int32)
        flags = lib.or_prefetch(
            ctypes.byref(lay), int(width), _p(self.slot_of[l]), _p(self.page_of[l]),
            _p(self.last_use[l]), _p(self.clock[l:l + 1]),
            _p(np.ascontiguousarray(scores, np.int32)),
            _p(np.ascontiguousarray(seq_lens, np.int32)), _p(np.ascontiguousarray(bt, np.int32)),
            _p(self._mir(self.k_mirror, l)), _p(self._mir(self.v_mirror, l)),
            _p(self._mir(self.k_scale_m, l)), _p(self._mir(self.v_scale_m, l)),
            _p(self.k_pool[l]), _p(self.v_pool[l]), _p(self.k_scale[l]), _p(self.v_scale[l]),
            _p(mp), _p(ms), _p(nm))
        return mp, ms, int(nm[0]), flags

    # -- a5 ------------------------------------------------------------------
    def remap(self, layer: int, sel: np.ndarray, bt: np.ndarray):
        lib, lay = _load(), self.lay.c()
        phys = np.empty((self.lay.batch, self.lay.max_sel), np.int32)
        unresolved = lib.or_remap(ctypes.byref(lay), _p(self.slot_of[layer]),
                                  _p(np.ascontiguousarray(sel, np.int32)),
                                  _p(np.ascontiguousarray(bt, np.int32)), _p(phys))
        return phys, unresolved

    # -- a6 + a7 -------------------------------------------------------------
    def decode(self, layer: int, q_bits: np.ndarray, sel: np.ndarray, phys: np.ndarray,
               seq_lens: np.ndarray, sm_scale: float | None = None) -> np.ndarray:
        lib, lay = _load(), self.lay.c()
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.lay.head_dim)
        out = np.empty((self.lay.batch, self.lay.n_q_heads, self.lay.head_dim), np.float64)
        l = layer
        lib.or_decode(ctypes.byref(lay), _p(self.k_pool[l]), _p(self.v_pool[l]),
                      _p(self.k_scale[l]), _p(self.v_scale[l]),
                      _p(np.ascontiguousarray(q_bits, np.uint16)),
                      _p(np.ascontiguousarray(sel, np.int32)),
                      _p(np.ascontiguousarray(phys, np.int32)),
                      _p(np.ascontiguousarray(seq_lens, np.int32)), float(sm_scale), _p(out))
        return out

    def decode_from_mirror(self, layer: int, q_bits: np.ndarray, sel: np.ndarray,
                           bt: np.ndarray, seq_lens: np.ndarray, sm_scale: float | None = None):
        """The attention over the selected pages read from the host mirror
        (which holds the pool's bytes for every page): or_decode with the
        mirror as the page store and the logical ids as its slots."""
        lib, lay = _load(), self.lay.c()
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.lay.head_dim)
        sel = np.ascontiguousarray(sel, np.int32)
        ids = np.full_like(sel, -1)
        for b in range(sel.shape[0]):
            v = sel[b] >= 0
            ids[b][v] = np.asarray(bt, np.int32)[b][sel[b][v]]
        out = np.empty((self.lay.batch, self.lay.n_q_heads, self.lay.head_dim), np.float64)
        l = layer
        lib.or_decode(ctypes.byref(lay), _p(self.k_mirror[l]), _p(self.v_mirror[l]),
                      _p(self.k_scale_m[l]), _p(self.v_scale_m[l]),
                      _p(np.ascontiguousarray(q_bits, np.uint16)), _p(sel), _p(ids),
                      _p(np.ascontiguousarray(seq_lens, np.int32)), float(sm_scale), _p(out))
        return out

    # -- one whole decode step for one layer --------------------------------
    def step(self, layer: int, q_bits, bt, seq_lens, sm_scale=None) -> dict:
        sel, n_sel, scores, drops, bad = self.index_topk(layer, q_bits, bt, seq_lens)
        mp, ms, nm, flags = self.ensure(layer, sel, bt)
        phys, unresolved = self.remap(layer, sel, bt)
        out = self.decode(layer, q_bits, sel, phys, seq_lens, sm_scale)
        return dict(sel=sel, n_sel=n_sel, scores=scores, drops=drops, bad=bad, miss_page=mp,
                    miss_slot=ms, n_miss=nm, flags=flags, phys=phys, unresolved=unresolved,
                    out=out)
