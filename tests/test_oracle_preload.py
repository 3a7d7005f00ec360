"""Pins for the oracle's top-k preload (or_prefetch).

The reading (vLLM RFC #33980, "Topk KV preload"): after a step's ensure, the
top (width - 1) pages plus the last page of each request by that step's
scores are made resident ahead of the next step: resident ones are touched
with the step's epoch, missing ones take free slots, then bound slots older
than the epoch, by (last_use, slot); the clock does not move.

Pinned by a hand-worked trace (every slot, page and last_use value written
out below), by the no-op case (width = k + 1 right after the step's own
ensure), and by random traces checked against an independent model of the
rule written here in numpy, with the pool's invariants after every call.
"""
import numpy as np
import pytest

import oracle
from workloads import Workload, block_table, store_batch


def _kv(B, n, S, k, fp8=False, P=16):
    w = Workload("pre", batch=B, n_layers=1, ctx=n * P, page_size=P, n_q_heads=2, n_kv_heads=1,
                 head_dim=32, fp8=fp8, block_topk=k, pool_slots=S, seed=41)
    lay = oracle.OracleLayout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8, 1,
                              w.logical_pages, w.slots, w.batch, w.pages_per_request,
                              w.block_topk)
    kv = oracle.OracleKV(lay, host_tier=True, identity=False)
    kk, vv, pos = store_batch(w, 0)
    kv.store(0, kk, vv, pos)
    return w, kv


def _sel(W, pages_per_request):
    out = np.full((len(pages_per_request), W), -1, np.int32)
    for b, pages in enumerate(pages_per_request):
        out[b, :len(pages)] = sorted(pages)
    return out


def test_hand_trace():
    # S = 4 slots, one request of 8 pages (logical ids = page indices), k = 1
    w, kv = _kv(B=1, n=8, S=4, k=1)
    W, bt, lens = 2 * 1 + 8, block_table(w), w.lens
    # step 0: ensure {2, 7} on the empty pool -> slots 0, 1; clock 1 (epoch 0)
    kv.ensure(0, _sel(W, [[2, 7]]), bt)
    assert list(kv.page_of[0]) == [2, 7, -1, -1] and kv.clock[0] == 1
    # preload width 4 by scores: top 3 of pages 0..6 = 2 (90), 4 (70), 6 (60),
    # plus page 7; missing 4 and 6 take the free slots 2 and 3 with last_use 0
    scores = np.array([[5, 50, 90, 40, 70, 10, 60, -999]], np.int32)
    mp, ms, nm, fl = kv.prefetch(0, 4, scores, lens, bt)
    assert fl == 0 and nm == 2 and list(mp[:2]) == [4, 6] and list(ms[:2]) == [2, 3]
    assert list(kv.page_of[0]) == [2, 7, 4, 6]
    assert list(kv.last_use[0]) == [0, 0, 0, 0] and kv.clock[0] == 1
    # step 1: ensure {4, 7}: both hits (the preload's page 4), touched at 1
    mp, ms, nm, _ = kv.ensure(0, _sel(W, [[4, 7]]), bt)
    assert nm == 0 and list(kv.last_use[0]) == [0, 1, 1, 0] and kv.clock[0] == 2
    # preload (epoch 1): top 3 = 4 (95), 1 (80), 3 (75), plus 7; missing 1, 3
    # take the slots older than epoch 1 by (last_use, slot): slot 0 (page 2),
    # then slot 3 (page 6); the hits 4 and 7 keep last_use 1
    scores = np.array([[0, 80, 10, 75, 95, 20, 30, 0]], np.int32)
    mp, ms, nm, _ = kv.prefetch(0, 4, scores, lens, bt)
    assert nm == 2 and list(mp[:2]) == [1, 3] and list(ms[:2]) == [0, 3]
    assert list(kv.page_of[0]) == [1, 7, 4, 3] and list(kv.last_use[0]) == [1, 1, 1, 1]
    assert kv.slot_of[0][2] == -1 and kv.slot_of[0][6] == -1
    # step 2: ensure {3, 7}: hits, touched at 2 -> last_use (1, 2, 1, 2)
    kv.ensure(0, _sel(W, [[3, 7]]), bt)
    assert list(kv.last_use[0]) == [1, 2, 1, 2] and kv.clock[0] == 3
    # preload (epoch 2): top 3 = 0 (9), 5 (8), 6 (7) + 7: three missing, two
    # victims older than epoch 2 (slot 0, then slot 2): ids 0 and 5 bound,
    # id 6 left out
    scores = np.array([[9, 1, 1, 1, 1, 8, 7, 0]], np.int32)
    mp, ms, nm, _ = kv.prefetch(0, 4, scores, lens, bt)
    assert nm == 2 and list(mp[:3]) == [0, 5, -1] and list(ms[:3]) == [0, 2, -1]
    assert list(kv.page_of[0]) == [0, 7, 5, 3] and kv.slot_of[0][6] == -1
    assert list(kv.last_use[0]) == [2, 2, 2, 2] and kv.clock[0] == 3
    # step 3: ensure {5, 7} -> last_use (2, 3, 3, 2); preload (epoch 3):
    # top 3 = 0 (9), 3 (8), 4 (7) + 7: the resident candidates 0 and 3 are
    # touched to 3, so the one miss (4) finds no victim older than epoch 3
    kv.ensure(0, _sel(W, [[5, 7]]), bt)
    assert list(kv.last_use[0]) == [2, 3, 3, 2]
    scores = np.array([[9, 1, 1, 8, 7, 1, 1, 0]], np.int32)
    mp, ms, nm, _ = kv.prefetch(0, 4, scores, lens, bt)
    assert nm == 0 and list(kv.page_of[0]) == [0, 7, 5, 3]
    assert list(kv.last_use[0]) == [3, 3, 3, 3]
    # the preloaded pages' bytes are the mirror's
    for s, p in ((0, 0), (2, 5)):
        assert np.array_equal(kv.k_pool[0, s], kv.k_mirror[0, p])
        assert np.array_equal(kv.v_pool[0, s], kv.v_mirror[0, p])


def test_width_of_the_selection_right_after_its_ensure_is_a_no_op():
    w, kv = _kv(B=2, n=30, S=2 * 20, k=5)
    bt, lens = block_table(w), w.lens
    rng = np.random.default_rng(3)
    scores = rng.integers(-1000, 1000, size=(2, w.pages_per_request)).astype(np.int32)
    lay = kv.lay
    sel = np.empty((2, lay.max_sel), np.int32)
    # the step's own selection from the same scores (or_select, k = 5)
    import ctypes
    n_sel = np.empty((2,), np.int32)
    oracle._load().or_select(ctypes.byref(lay.c()), oracle._p(scores), oracle._p(lens),
                             oracle._p(sel), oracle._p(n_sel))
    kv.ensure(0, sel, bt)
    before = (kv.slot_of.copy(), kv.page_of.copy(), kv.last_use.copy(), kv.clock.copy())
    mp, ms, nm, _ = kv.prefetch(0, w.block_topk + 1, scores, lens, bt)
    assert nm == 0 and (mp == -1).all()
    for a, b in zip(before, (kv.slot_of, kv.page_of, kv.last_use, kv.clock)):
        assert np.array_equal(a, b)


def _model_prefetch(slot_of, page_of, last_use, clock, cand_ids):
    """The rule restated independently: numpy sorts, no C."""
    e = clock - 1
    slot_of, page_of, last_use = slot_of.copy(), page_of.copy(), last_use.copy()
    ids = np.unique(np.asarray(cand_ids, np.int64))
    missing = [int(i) for i in ids if slot_of[i] < 0]
    for i in ids:
        if slot_of[i] >= 0:
            last_use[slot_of[i]] = e
    slots = np.arange(len(page_of))
    ok = ~((page_of >= 0) & (last_use >= e))
    key = np.where(page_of < 0, -2, last_use)
    vic = slots[ok][np.lexsort((slots[ok], key[ok]))]
    bound = []
    for id_, v in zip(missing, vic):
        old = page_of[v]
        if old >= 0:
            slot_of[old] = -1
        slot_of[id_], page_of[v], last_use[v] = v, id_, e
        bound.append((id_, int(v)))
    return slot_of, page_of, last_use, bound


def _top_candidates(scores, lens, P, width, n_max):
    out = []
    for b in range(scores.shape[0]):
        n = min(n_max, -(-int(lens[b]) // P))
        if n - 1 <= width - 1:
            pages = list(range(n))
        else:
            order = sorted(range(n - 1), key=lambda p: (-int(scores[b, p]), p))
            pages = order[:width - 1] + [n - 1]
        out.append(pages)
    return out


@pytest.mark.parametrize("fp8", [False, True])
def test_random_traces_match_an_independent_model(fp8):
    rng = np.random.default_rng(7 + fp8)
    B, n, k = 3, 50, 4
    W = 2 * k + 8
    S = B * W + 5
    w, kv = _kv(B=B, n=n, S=S, k=k, fp8=fp8)
    bt, lens = block_table(w), w.lens
    bt[2, :12] = bt[0, :12]                   # requests 0 and 2 share 12 logical pages
    for step in range(40):
        scores = rng.integers(-50, 50, size=(B, w.pages_per_request)).astype(np.int32)
        # the step: its selection (top k + last) and its ensure
        sel_pages = _top_candidates(scores, lens, w.page_size, k + 1, w.pages_per_request)
        kv.ensure(0, _sel(W, sel_pages), bt)
        pinned = {int(bt[b][p]) for b, ps in enumerate(sel_pages) for p in ps}
        width = int(rng.integers(1, W + 1))
        cand = _top_candidates(scores, lens, w.page_size, width, w.pages_per_request)
        cand_ids = [int(bt[b][p]) for b, ps in enumerate(cand) for p in ps]
        want = _model_prefetch(kv.slot_of[0], kv.page_of[0], kv.last_use[0], int(kv.clock[0]),
                               cand_ids)
        clock = int(kv.clock[0])
        mp, ms, nm, fl = kv.prefetch(0, width, scores, lens, bt)
        assert fl == 0
        assert np.array_equal(kv.slot_of[0], want[0]) and np.array_equal(kv.page_of[0], want[1])
        assert np.array_equal(kv.last_use[0], want[2]) and int(kv.clock[0]) == clock
        assert [(int(a), int(b)) for a, b in zip(mp[:nm], ms[:nm])] == want[3]
        # the pages the step reads stay resident; bijection; pool == mirror
        assert all(kv.slot_of[0][i] >= 0 for i in pinned)
        po, so = kv.page_of[0], kv.slot_of[0]
        bound = np.nonzero(po >= 0)[0]
        assert len(set(po[bound].tolist())) == len(bound) and (so[po[bound]] == bound).all()
        for s in bound:
            assert np.array_equal(kv.k_pool[0, s], kv.k_mirror[0, po[s]])
            assert np.array_equal(kv.v_pool[0, s], kv.v_mirror[0, po[s]])
        # with S >= B*W every candidate fits
        assert all(so[i] >= 0 for i in cand_ids)


def test_attention_from_the_mirror_equals_attention_from_the_pool():
    # the mirror holds the pool's bytes, so once the selection is resident the
    # attention read from the mirror (logical ids as slots) is the same, bit
    # for bit, as the one read from the pool through the remapped table
    w, kv = _kv(B=2, n=40, S=2 * 20, k=5, fp8=True)
    bt, lens = block_table(w), w.lens
    from workloads import queries
    q = queries(w.with_(steps=1), 0)[0]
    sel, n_sel, scores, _, _ = kv.index_topk(0, q, bt, lens)
    kv.ensure(0, sel, bt)
    phys, unresolved = kv.remap(0, sel, bt)
    assert unresolved == 0
    a = kv.decode(0, q, sel, phys, lens)
    b = kv.decode_from_mirror(0, q, sel, bt, lens)
    assert np.array_equal(a, b)
