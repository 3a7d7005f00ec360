"""GPU parity: the CUDA library against the oracle, element by element.

Small cases run every layer through the oracle and span several tiles with a
ragged tail; full-size cases (the five synthetic workloads) run the library
on every layer in the benchmark's launch configuration (layer-batched) and
check sampled layers against the oracle.  Bit-exact: scores, selection,
remap, miss lists, LRU state, slab, pool and mirror bytes.  Outputs: max-abs
error within 1e-2 (bf16) / 3e-2 (fp8) of the fp64 oracle.
"""
import math

import numpy as np
import pytest

import workloads as wl
from tests.parity import run_parity

pytestmark = pytest.mark.gpu


def _w(name, **kw):
    base = dict(batch=2, n_layers=2, ctx=64 * 40, page_size=64, n_q_heads=16, n_kv_heads=2,
                head_dim=128, fp8=False, block_topk=8, pool_slots=None, steps=1, seed=100)
    base.update(kw)
    return wl.Workload(name, **base)


SMALL = [
    # resident bf16, GQA 8:1, 16-token pages, a real top-16 over 256 pages
    wl.WORKLOADS["decode_4k_bf16_resident"],
    # needles + ragged requests, 64-token pages
    _w("needles_ragged_bf16", batch=3, ctx=64 * 150 + 37, seq_lens=(64 * 150 + 37, 6000, 4160),
       block_topk=32, needles=4, seed=101),
    # host tier, fp8, LRU pressure over several steps
    _w("lru_fp8", batch=3, ctx=64 * 120 + 11, seq_lens=(64 * 120 + 11, 64 * 90, 64 * 100 + 63),
       fp8=True, block_topk=6, pool_slots=3 * 20 + 7, steps=6, rho=0.8, walk_c=0.6, seed=102),
    _w("host_tier_fp8_rho95", batch=1, ctx=64 * 600, fp8=True, block_topk=32, pool_slots=150,
       steps=5, rho=0.95, walk_c=0.31, seed=103),
    _w("host_tier_bf16", batch=2, ctx=64 * 90 + 5, fp8=False, block_topk=10, pool_slots=2 * 28 + 1,
       steps=4, rho=0.8, walk_c=0.6, seed=104),
    # 32/4 heads (the sweep's shape), resident and 20%-resident
    _w("wide_heads_bf16", batch=2, ctx=64 * 400, n_q_heads=32, n_kv_heads=4, block_topk=32,
       steps=2, rho=0.9, walk_c=math.sqrt(1 - 0.81), seed=105),
    _w("wide_heads_fp8_20pct", batch=2, ctx=64 * 400, n_q_heads=32, n_kv_heads=4, fp8=True,
       block_topk=32, pool_slots=160, steps=3, rho=0.9, walk_c=math.sqrt(1 - 0.81), seed=106),
    # other page sizes and groups
    _w("p32_fp8_g4", batch=2, ctx=32 * 77 + 9, page_size=32, n_q_heads=8, n_kv_heads=2, fp8=True,
       block_topk=12, pool_slots=2 * 32 + 3, steps=3, rho=0.8, walk_c=0.6, seed=107),
    _w("p128_bf16_g1", batch=2, ctx=128 * 50 + 100, page_size=128, n_q_heads=4, n_kv_heads=4,
       block_topk=5, seed=108),
    _w("p16_fp8_g2_h8", batch=1, ctx=16 * 300 + 3, page_size=16, n_q_heads=16, n_kv_heads=8,
       fp8=True, block_topk=20, seed=109),
    # every page selected (dense attention), tiny requests
    _w("dense_short", batch=3, ctx=64 * 5, seq_lens=(64 * 5, 1, 64 + 1), block_topk=32, seed=110),
    # many (layer, request, KV head) units per attention CTA: 512 units of 9
    # pages over one wave, so CTAs hold whole units and pieces of two others
    # (the mid-range merges); then ragged lengths, 1 token to full
    _w("many_units_fp8", batch=64, ctx=64 * 40, n_q_heads=32, n_kv_heads=4, fp8=True,
       block_topk=8, steps=2, rho=0.9, walk_c=math.sqrt(1 - 0.81), seed=111),
    _w("many_units_bf16_ragged", batch=48, ctx=64 * 40,
       seq_lens=tuple(64 * 40 if i % 3 == 0 else (i * 379) % (64 * 40) + 1 for i in range(48)),
       block_topk=8, steps=2, rho=0.9, walk_c=math.sqrt(1 - 0.81), seed=112),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_parity_small_layer_batched(w):
    rep = {}
    run_parity(w, report=rep)
    print(w.name, rep)


@pytest.mark.parametrize("w", SMALL[:3], ids=[w.name for w in SMALL[:3]])
def test_parity_small_per_layer_launches(w):
    run_parity(w, per_layer=True)


def test_needles_are_selected_on_both_sides():
    w = SMALL[1]
    run, orc = run_parity(w)
    pages = wl.needle_pages(w)
    for l in range(w.n_layers):
        sel = run.sel[l].cpu().numpy()
        for b in range(w.batch):
            assert set(pages[b].tolist()) <= set(sel[b].tolist())


HOST_TIER = [w for w in SMALL if w.host_tier]


@pytest.mark.parametrize("w", HOST_TIER, ids=[w.name for w in HOST_TIER])
def test_parity_misses_fetched_inside_the_attention(w):
    # ssa_ensure_remap_deferred + ssa_sparse_paged_decode_fetch: the same
    # state, miss lists, pool bytes (every step) and outputs as ensure + copy
    rep = {}
    run_parity(w, fetch_in_attention=True, report=rep)
    assert rep["misses"] > 0
    print(w.name, rep)


@pytest.mark.parametrize("w", HOST_TIER, ids=[w.name for w in HOST_TIER])
def test_parity_copy_overlapped_with_attention(w):
    # ssa_ensure_remap_bind for all layers, then per layer range
    # ssa_fetch_misses with that range's attention on a second stream: the
    # same state, lists, pool bytes (every step) and outputs as the oracle
    rep = {}
    run_parity(w, overlap_groups=w.n_layers, report=rep)
    assert rep["misses"] > 0
    print(w.name, rep)
