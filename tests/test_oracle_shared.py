"""Pins for the oracle's shared residency (or_ensure_shared).

The reading (FreeToken PR #499, "Design": one launch copies a page's K and V
for all the layers): the layers of a call share one LRU state, the first
layer's; the union of their selections is ensured by the per-layer rules;
each miss is copied into the same slot of every layer's pool.

Pinned by a hand-worked two-layer trace, by the case where every layer
selects the same pages (the shared state must then equal the state a single
layer's own LRU reaches), and by random traces with the pool's invariants.
"""
import numpy as np
import pytest

import oracle
from workloads import Workload, block_table, store_batch


def _kv(n_layers, B, n, S, k, fp8=False, P=16):
    w = Workload("shared", batch=B, n_layers=n_layers, ctx=n * P, page_size=P, n_q_heads=2,
                 n_kv_heads=1, head_dim=32, fp8=fp8, block_topk=k, pool_slots=S, seed=61)
    lay = oracle.OracleLayout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8,
                              n_layers, w.logical_pages, w.slots, w.batch, w.pages_per_request,
                              w.block_topk)
    kv = oracle.OracleKV(lay, host_tier=True, identity=False)
    for l in range(n_layers):
        kk, vv, pos = store_batch(w, l)
        kv.store(l, kk, vv, pos)
    return w, kv


def _sel(W, layers):
    """layers: per layer, per request, the selected pages."""
    out = np.full((len(layers), len(layers[0]), W), -1, np.int32)
    for l, reqs in enumerate(layers):
        for b, pages in enumerate(reqs):
            out[l, b, :len(pages)] = sorted(pages)
    return out


def _pools_match_mirror(kv, n_layers, l0=0):
    po = kv.page_of[l0]
    for l in range(l0, l0 + n_layers):
        for s in np.nonzero(po >= 0)[0]:
            assert np.array_equal(kv.k_pool[l, s], kv.k_mirror[l, po[s]])
            assert np.array_equal(kv.v_pool[l, s], kv.v_mirror[l, po[s]])
            assert np.array_equal(kv.k_scale[l, s], kv.k_scale_m[l, po[s]])


def test_hand_trace_two_layers():
    w, kv = _kv(n_layers=2, B=1, n=8, S=4, k=1, fp8=True)
    W, bt = 10, block_table(w)
    # step 0: layer 0 {2, 7}, layer 1 {4, 7}: the union {2, 4, 7} takes the
    # free slots 0, 1, 2 in ascending id order
    mp, ms, nm, fl = kv.ensure_shared(0, 2, _sel(W, [[[2, 7]], [[4, 7]]]), bt)
    assert fl == 0 and nm == 3 and list(mp[:3]) == [2, 4, 7] and list(ms[:3]) == [0, 1, 2]
    assert list(kv.page_of[0]) == [2, 4, 7, -1] and list(kv.last_use[0]) == [0, 0, 0, -1]
    assert kv.clock[0] == 1
    _pools_match_mirror(kv, 2)
    # step 1: {4, 7} and {5, 7}: hits 4, 7 touched at 1; miss 5 -> slot 3
    mp, ms, nm, _ = kv.ensure_shared(0, 2, _sel(W, [[[4, 7]], [[5, 7]]]), bt)
    assert nm == 1 and mp[0] == 5 and ms[0] == 3
    assert list(kv.last_use[0]) == [0, 1, 1, 1] and kv.clock[0] == 2
    # step 2: {0, 7} and {6, 7}: hit 7 (slot 2) touched at 2; misses 0, 6
    # take slot 0 (last_use 0), then slot 1 (last_use 1, before slot 3)
    mp, ms, nm, _ = kv.ensure_shared(0, 2, _sel(W, [[[0, 7]], [[6, 7]]]), bt)
    assert nm == 2 and list(mp[:2]) == [0, 6] and list(ms[:2]) == [0, 1]
    assert list(kv.page_of[0]) == [0, 6, 7, 5] and list(kv.last_use[0]) == [2, 2, 2, 1]
    assert kv.clock[0] == 3
    _pools_match_mirror(kv, 2)
    # the second layer's own LRU arrays are untouched
    assert (kv.page_of[1] == -1).all() and kv.clock[1] == 0


def test_identical_selections_reach_the_single_layer_state():
    rng = np.random.default_rng(5)
    B, n, k = 2, 40, 3
    W = 2 * k + 8
    w, shared = _kv(n_layers=3, B=B, n=n, S=B * W + 2, k=k)
    _, single = _kv(n_layers=3, B=B, n=n, S=B * W + 2, k=k)
    bt = block_table(w)
    for step in range(30):
        pages = [sorted(rng.choice(n, size=k + 1, replace=False).tolist()) for _ in range(B)]
        sel1 = _sel(W, [pages])[0]
        single.ensure(0, sel1, bt)
        mp, ms, nm, _ = shared.ensure_shared(0, 3, np.stack([sel1] * 3), bt)
        for name in ("slot_of", "page_of", "last_use", "clock"):
            assert np.array_equal(getattr(shared, name)[0], getattr(single, name)[0]), name
    _pools_match_mirror(shared, 3)


@pytest.mark.parametrize("fp8", [False, True])
def test_random_traces_keep_every_layer_resident(fp8):
    rng = np.random.default_rng(9 + fp8)
    L, B, n, k = 3, 2, 50, 4
    W = 2 * k + 8
    S = L * B * W
    w, kv = _kv(n_layers=L, B=B, n=n, S=S, k=k, fp8=fp8)
    bt = block_table(w)
    for step in range(40):
        layers = [[sorted(rng.choice(n, size=k + 1, replace=False).tolist()) for _ in range(B)]
                  for _ in range(L)]
        sel = _sel(W, layers)
        before = set(np.nonzero(kv.slot_of[0] >= 0)[0].tolist())
        mp, ms, nm, fl = kv.ensure_shared(0, L, sel, bt)
        assert fl == 0
        union = {int(bt[b][p]) for reqs in layers for b, ps in enumerate(reqs) for p in ps}
        assert all(kv.slot_of[0][i] >= 0 for i in union)
        assert sorted(mp[:nm].tolist()) == mp[:nm].tolist()
        assert set(mp[:nm].tolist()) == union - before
        po, so = kv.page_of[0], kv.slot_of[0]
        bound = np.nonzero(po >= 0)[0]
        assert len(set(po[bound].tolist())) == len(bound) and (so[po[bound]] == bound).all()
        for l in range(L):
            phys, unresolved = kv.remap_shared(0, l, sel[l], bt)
            assert unresolved == 0
    _pools_match_mirror(kv, L)
