"""Seeded synthetic inputs for the sparse-attention decode step.

This module is the ONLY code that the oracle tests and the CUDA path share.  It
holds no step of the method: it draws random numbers, rounds them to bf16 (the
stored input format), plants needle pages, walks the decode queries and builds
block tables.  Quantisation, indexing, selection, residency and attention live
on each side separately.

Recipe (all draws: numpy PCG64 ``default_rng``, float32 N(0, 1), rounded to
bf16 with round-to-nearest-even):
  * K, V of request b in layer l:  rng([seed, l, 1, b]); K drawn first, then
    V, shape [seq_len[b]][Hkv][D].  Requests have streams of their own, so
    they are drawn in parallel threads with the same result.
  * queries for layer l: rng([seed, l, 2]); q_0 ~ N(0, 1) [B][Hq][D];
    q_t = rho * q_{t-1} + c * eps_t, kept in fp32 and rounded to bf16 per step.
  * needles: rng([seed, 3]) draws, per request, ``needles`` distinct pages from
    [0, n-1); every token of those pages gets K[h] += 0.5 * unit(sum of the
    query heads of KV head h at step 0), before rounding.
  * block table: request b, page p -> logical id b * n + p.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_layers: int
    ctx: int                 # tokens per request (before any ragged override)
    page_size: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    fp8: bool
    block_topk: int
    pool_slots: int | None   # None: fully resident, pool = logical pages, no host tier
    steps: int = 1
    rho: float | None = None # query random-walk coefficient (None: one fixed q)
    walk_c: float | None = None
    needles: int = 0
    seed: int = 0
    seq_lens: tuple | None = None  # per-request token counts (ragged); default ctx

    # ---- derived shapes --------------------------------------------------
    @property
    def lens(self) -> np.ndarray:
        if self.seq_lens is not None:
            return np.asarray(self.seq_lens, np.int32)
        return np.full((self.batch,), self.ctx, np.int32)

    @property
    def pages_per_request(self) -> int:
        return int(math.ceil(int(self.lens.max()) / self.page_size))

    @property
    def logical_pages(self) -> int:
        return self.batch * self.pages_per_request

    @property
    def host_tier(self) -> bool:
        return self.pool_slots is not None

    @property
    def slots(self) -> int:
        return self.logical_pages if self.pool_slots is None else self.pool_slots

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _c(rho: float) -> float:
    return math.sqrt(1.0 - rho * rho)


# The five synthetic workloads, by what they are.
WORKLOADS = {
    # 1 request, 1 layer, 4,096 tokens in 16-token pages, GQA 8:1, bf16,
    # top-16 pages plus the last page, everything resident.
    "decode_4k_bf16_resident": Workload(
        "decode_4k_bf16_resident", batch=1, n_layers=1, ctx=4096, page_size=16,
        n_q_heads=8, n_kv_heads=1, head_dim=128, fp8=False, block_topk=16,
        pool_slots=None, seed=0),
    # 4 requests x 12 layers, 32,768 tokens in 64-token pages, 16/2 heads,
    # bf16, 4 planted needle pages per request, top-32, everything resident.
    "batched_32k_bf16_needles": Workload(
        "batched_32k_bf16_needles", batch=4, n_layers=12, ctx=32768, page_size=64,
        n_q_heads=16, n_kv_heads=2, head_dim=128, fp8=False, block_topk=32,
        pool_slots=None, needles=4, seed=1),
    # 1 request x 12 layers, 196,608 tokens (3,072 pages), 1,635 GPU slots per
    # layer over a pinned host mirror, fp8, 64 decode steps, rho = 0.95.
    "host_tier_196k_fp8": Workload(
        "host_tier_196k_fp8", batch=1, n_layers=12, ctx=196608, page_size=64,
        n_q_heads=16, n_kv_heads=2, head_dim=128, fp8=True, block_topk=32,
        pool_slots=1635, steps=64, rho=0.95, walk_c=0.31, seed=2),
    # 4 requests x 12 layers, 65,536 tokens each (1,024 pages), 320 GPU slots
    # per layer, fp8, 32 decode steps, rho = 0.8 (frequent misses).
    "lru_pressure_64k_fp8": Workload(
        "lru_pressure_64k_fp8", batch=4, n_layers=12, ctx=65536, page_size=64,
        n_q_heads=16, n_kv_heads=2, head_dim=128, fp8=True, block_topk=32,
        pool_slots=320, steps=32, rho=0.8, walk_c=_c(0.8), seed=3),
}


def sweep_workload(batch: int, fp8: bool, resident_fraction: float, steps: int = 16) -> Workload:
    """Throughput sweep: 12 layers, 131,072 tokens per request in 64-token
    pages, 32/4 heads, top-32, rho = 0.9; fully resident (fraction 1.0) or a
    pool of ceil(fraction * logical pages) slots over the host mirror."""
    n = 131072 // 64
    lp = batch * n
    slots = None if resident_fraction >= 1.0 else int(math.ceil(resident_fraction * lp))
    tag = "resident" if slots is None else f"{int(round(resident_fraction * 100))}pct"
    return Workload(
        f"sweep_128k_{'fp8' if fp8 else 'bf16'}_{tag}_b{batch}", batch=batch, n_layers=12,
        ctx=131072, page_size=64, n_q_heads=32, n_kv_heads=4, head_dim=128, fp8=fp8,
        block_topk=32, pool_slots=slots, steps=steps, rho=0.9, walk_c=_c(0.9), seed=4)


# ---------------------------------------------------------------------------
# bf16 helpers (input format only)
# ---------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------

def block_table(w: Workload) -> np.ndarray:
    n = w.pages_per_request
    return (np.arange(w.batch, dtype=np.int32)[:, None] * n
            + np.arange(n, dtype=np.int32)[None, :]).astype(np.int32)


def query_walk_f32(w: Workload, layer: int) -> np.ndarray:
    """[steps][B][Hq][D] fp32 queries of the seeded random walk."""
    rng = np.random.default_rng([w.seed, layer, 2])
    shape = (w.batch, w.n_q_heads, w.head_dim)
    out = np.empty((w.steps,) + shape, np.float32)
    q = rng.standard_normal(shape, dtype=np.float32)
    out[0] = q
    if w.steps > 1:
        rho = np.float32(w.rho)
        c = np.float32(w.walk_c)
        for t in range(1, w.steps):
            q = rho * q + c * rng.standard_normal(shape, dtype=np.float32)
            out[t] = q
    return out


def queries(w: Workload, layer: int) -> np.ndarray:
    """[steps][B][Hq][D] bf16 bits."""
    return to_bf16_bits(query_walk_f32(w, layer))


def needle_pages(w: Workload) -> np.ndarray:
    """[B][needles] page indices (within each request), or an empty array."""
    if w.needles == 0:
        return np.zeros((w.batch, 0), np.int32)
    rng = np.random.default_rng([w.seed, 3])
    out = np.empty((w.batch, w.needles), np.int32)
    for b in range(w.batch):
        n = int(math.ceil(int(w.lens[b]) / w.page_size))
        out[b] = np.sort(rng.choice(n - 1, size=w.needles, replace=False))
    return out


def _needle_dirs(w: Workload, layer: int) -> np.ndarray | None:
    """[B][Hkv][D] unit directions of the needles (sum of each KV head's query
    heads at step 0), or None without needles."""
    if not w.needles:
        return None
    q0 = query_walk_f32(w.with_(steps=1), layer)[0]          # [B][Hq][D]
    qh = q0.reshape(w.batch, w.n_kv_heads, w.group, w.head_dim).sum(axis=2)
    return qh / np.linalg.norm(qh, axis=-1, keepdims=True)


def kv_request_f32(w: Workload, layer: int, b: int, qh=None):
    """K, V fp32 [seq_len[b]][Hkv][D] of request b (needles planted in K)."""
    rng = np.random.default_rng([w.seed, layer, 1, b])
    shape = (int(w.lens[b]), w.n_kv_heads, w.head_dim)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    if w.needles:
        if qh is None:
            qh = _needle_dirs(w, layer)
        P = w.page_size
        for p in needle_pages(w)[b]:
            k[p * P:(p + 1) * P] += np.float32(0.5) * qh[b][None, :, :]
    return k, v


def store_batch(w: Workload, layer: int):
    """Everything one prefill stores for one layer, flattened over requests:
    k_bits, v_bits [T][Hkv][D] (uint16) and logical token ids pos [T] (int64),
    request-major, strictly increasing."""
    import concurrent.futures as cf
    import os
    bt = block_table(w)
    P = w.page_size
    qh = _needle_dirs(w, layer)
    lens = [int(x) for x in w.lens]
    T = sum(lens)
    HD = (w.n_kv_heads, w.head_dim)
    kb = np.empty((T,) + HD, np.uint16)
    vb = np.empty((T,) + HD, np.uint16)
    pos = np.empty((T,), np.int64)
    start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)

    def one(b):
        k, v = kv_request_f32(w, layer, b, qh)
        t0, t1 = start[b], start[b + 1]
        kb[t0:t1] = to_bf16_bits(k)
        vb[t0:t1] = to_bf16_bits(v)
        t = np.arange(lens[b], dtype=np.int64)
        pos[t0:t1] = bt[b][t // P].astype(np.int64) * P + t % P

    workers = max(1, min(w.batch, os.cpu_count() or 1))
    if workers == 1:
        for b in range(w.batch):
            one(b)
    else:
        with cf.ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(one, range(w.batch)))
    return kb, vb, pos
