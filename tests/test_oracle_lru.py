"""Pins for the oracle's LRU ensure, miss copy, remap and store mirror.

Invariants checked after every ensure on long random traces (shared pages
across requests included):
  * every selected page is resident afterwards; remap resolves every entry;
  * slot_of / page_of are mutual inverses on bound pairs (no slot bound twice);
  * misses are exactly the selected pages that were not resident, ascending;
  * free slots are used before any eviction; every evicted page was least
    recently used among the untouched bound slots (an independent model of
    the LRU order);
  * pool bytes equal mirror bytes for every bound slot (write-through mirror,
    drop-clean slots), codes and scales.
"""
import numpy as np
import pytest

import oracle
from workloads import Workload, block_table, queries, store_batch


def _state(w, identity=None):
    lay = oracle.OracleLayout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8,
                              w.n_layers, w.logical_pages, w.slots, w.batch,
                              w.pages_per_request, w.block_topk)
    ident = (not w.host_tier) if identity is None else identity
    return oracle.OracleKV(lay, host_tier=w.host_tier, identity=ident)


def _check_bijection(kv, l):
    so, po = kv.slot_of[l], kv.page_of[l]
    bound = np.nonzero(po >= 0)[0]
    assert len(set(po[bound].tolist())) == len(bound)
    assert (so[po[bound]] == bound).all()
    res = np.nonzero(so >= 0)[0]
    assert (po[so[res]] == res).all()


def _check_mirror(kv, l):
    po = kv.page_of[l]
    for s in np.nonzero(po >= 0)[0]:
        p = po[s]
        assert np.array_equal(kv.k_pool[l, s], kv.k_mirror[l, p])
        assert np.array_equal(kv.v_pool[l, s], kv.v_mirror[l, p])
        assert np.array_equal(kv.k_scale[l, s], kv.k_scale_m[l, p])
        assert np.array_equal(kv.v_scale[l, s], kv.v_scale_m[l, p])


@pytest.mark.parametrize("fp8", [False, True])
def test_random_trace_invariants(fp8):
    rng = np.random.default_rng(5 + fp8)
    B, n, P, k = 3, 40, 16, 3
    W = 2 * k + 8
    w = Workload("lru", batch=B, n_layers=1, ctx=n * P, page_size=P, n_q_heads=2, n_kv_heads=1,
                 head_dim=32, fp8=fp8, block_topk=k, pool_slots=B * W + 3, seed=31)
    kv = _state(w)
    kk, vv, pos = store_batch(w, 0)
    kv.store(0, kk, vv, pos)
    bt = block_table(w)
    bt[1, :10] = bt[0, :10]                  # requests 0 and 1 share 10 logical pages
    for step in range(60):
        before_slot = kv.slot_of[0].copy()
        before_lu = kv.last_use[0].copy()
        before_po = kv.page_of[0].copy()
        clock = int(kv.clock[0])
        sel = np.full((B, W), -1, np.int32)
        for b in range(B):
            m = rng.integers(1, W + 1)
            sel[b, :m] = np.sort(rng.choice(n, size=m, replace=False))
        mp, ms, nm, flags = kv.ensure(0, sel, bt)
        assert flags == 0
        ids = sorted({int(bt[b, p]) for b in range(B) for p in sel[b] if p >= 0})
        want_miss = [i for i in ids if before_slot[i] < 0]
        assert mp[:nm].tolist() == want_miss
        assert (mp[nm:] == -1).all() and (ms[nm:] == -1).all()
        # victim order model: free by slot, then untouched bound by (last_use, slot)
        touched = {int(before_slot[i]) for i in ids if before_slot[i] >= 0}
        free = [s for s in range(w.slots) if before_po[s] < 0]
        bound = sorted((int(before_lu[s]), s) for s in range(w.slots)
                       if before_po[s] >= 0 and s not in touched)
        order = free + [s for _, s in bound]
        assert ms[:nm].tolist() == order[:nm]
        # state
        for i in ids:
            assert kv.slot_of[0, i] >= 0
            assert kv.last_use[0, kv.slot_of[0, i]] == clock
        assert int(kv.clock[0]) == clock + 1
        _check_bijection(kv, 0)
        _check_mirror(kv, 0)
        phys, unresolved = kv.remap(0, sel, bt)
        assert unresolved == 0
        assert ((phys >= 0) == (sel >= 0)).all()


def test_identity_pool_has_no_misses_and_touches_hits():
    w = Workload("ident", batch=2, n_layers=1, ctx=20 * 16, page_size=16, n_q_heads=2,
                 n_kv_heads=1, head_dim=16, fp8=False, block_topk=4, pool_slots=None, seed=3)
    kv = _state(w)
    sel = np.full((2, 16), -1, np.int32)
    sel[0, :3] = [0, 5, 19]
    sel[1, :2] = [2, 19]
    mp, ms, nm, flags = kv.ensure(0, sel, block_table(w))
    assert nm == 0 and flags == 0
    assert sorted(np.nonzero(kv.last_use[0] == 0)[0].tolist()) == [0, 5, 19, 22, 39]


def test_miss_without_mirror_is_flagged():
    w = Workload("nomirror", batch=1, n_layers=1, ctx=8 * 16, page_size=16, n_q_heads=1,
                 n_kv_heads=1, head_dim=16, fp8=False, block_topk=2, pool_slots=None, seed=3)
    lay = oracle.OracleLayout(16, 1, 1, 16, False, 1, 8, 12, 1, 8, 2)
    kv = oracle.OracleKV(lay, host_tier=False, identity=False)   # empty pool, no mirror
    sel = np.full((1, 12), -1, np.int32)
    sel[0, :2] = [1, 7]
    mp, ms, nm, flags = kv.ensure(0, sel, block_table(w))
    assert nm == 2 and (flags & 4)


def test_store_writes_pool_only_for_resident_pages_and_mirror_always():
    w = Workload("store", batch=1, n_layers=1, ctx=10 * 16, page_size=16, n_q_heads=2,
                 n_kv_heads=2, head_dim=32, fp8=True, block_topk=2, pool_slots=12, seed=9)
    kv = _state(w)
    # bind pages 3 and 7 before the store
    sel = np.full((1, 12), -1, np.int32)
    sel[0, :2] = [3, 7]
    kv.ensure(0, sel, block_table(w))
    kv.k_pool[:] = 0
    k, v, pos = store_batch(w, 0)
    kv.store(0, k, v, pos)
    _check_mirror(kv, 0)
    bound = set(kv.page_of[0][kv.page_of[0] >= 0].tolist())
    assert bound == {3, 7}
    assert (kv.k_pool[0, 2:] == 0).all()     # unbound slots untouched


def test_fp8_store_scale_rule_and_codes_match_torch():
    import torch
    from workloads import bf16_bits_to_f32
    w = Workload("fp8", batch=1, n_layers=1, ctx=4 * 16, page_size=16, n_q_heads=2,
                 n_kv_heads=2, head_dim=64, fp8=True, block_topk=2, pool_slots=None, seed=4)
    kv = _state(w)
    k, v, pos = store_batch(w, 0)
    k[5] = 0                                    # an all-zero token: scale 1, codes 0
    kv.store(0, k, v, pos)
    x = bf16_bits_to_f32(k).reshape(len(pos), -1)
    amax = np.abs(x).max(axis=1)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    codes = torch.from_numpy((x / s[:, None]).astype(np.float32)).to(torch.float8_e4m3fn)
    codes = codes.view(torch.uint8).numpy()
    P, H, D = 16, 2, 64
    for t in range(len(pos)):
        page, j = divmod(int(pos[t]), P)
        slot = kv.slot_of[0, page]                # identity pool, no host tier
        assert kv.k_scale[0, slot, j] == s[t]
        got = kv.k_pool[0, slot].reshape(H, P, D)[:, j, :].reshape(-1)
        assert np.array_equal(got, codes[t])
    assert kv.k_scale[0, 0, 5] == 1.0
    assert (kv.k_pool[0, 0].reshape(H, P, D)[:, 5, :] == 0).all()
