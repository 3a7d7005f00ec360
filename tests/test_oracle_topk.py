"""Pins for the oracle's top-k page selection.

Checked against (a) the defining property of the selection, on tiny inputs
with many ties, and (b) numpy's lexsort (a library routine): the k best pages
of [0, n-1) by (score desc, page asc), plus the last page, ascending, padded.
"""
import itertools

import numpy as np
import pytest

import oracle


def _select(scores, seq_lens, k, P=4, n_max=None):
    B, n = scores.shape
    n_max = n_max or n
    lay = oracle.OracleLayout(page_size=P, n_q_heads=1, n_kv_heads=1, head_dim=1, fp8=False,
                              n_layers=1, logical_pages=B * n_max, pool_slots=B * n_max,
                              batch=B, max_pages=n_max, block_topk=k)
    lib = oracle._load()
    W = lay.max_sel
    sel = np.empty((B, W), np.int32)
    n_sel = np.empty((B,), np.int32)
    sc = np.full((B, n_max), np.iinfo(np.int32).min, np.int32)
    sc[:, :n] = scores
    import ctypes
    drops = lib.or_select(ctypes.byref(lay.c()), oracle._p(sc),
                          oracle._p(np.ascontiguousarray(seq_lens, np.int32)),
                          oracle._p(sel), oracle._p(n_sel))
    return sel, n_sel, drops, W


def _check_property(row, scores, n, k, W):
    chosen = [p for p in row if p >= 0]
    assert chosen == sorted(chosen) and len(set(chosen)) == len(chosen)
    assert all(p == -1 for p in row[len(chosen):])
    if n == 0:
        assert chosen == []
        return
    if n - 1 <= k:
        assert chosen == list(range(n))
        return
    assert n - 1 in chosen and len(chosen) == k + 1
    top = set(chosen) - {n - 1}
    rest = set(range(n - 1)) - top
    for i in top:
        for j in rest:
            assert scores[i] > scores[j] or (scores[i] == scores[j] and i < j)


def test_bruteforce_all_tie_patterns_small():
    # every score vector over {0,1,2} for n = 6 pages, k = 1..4
    n = 6
    for vals in itertools.product(range(3), repeat=n):
        s = np.array([vals], np.int32)
        for k in (1, 2, 3, 4):
            sel, n_sel, drops, W = _select(s, [n * 4], k)
            _check_property(sel[0].tolist(), list(vals), n, k, W)
            assert drops == 0 and n_sel[0] == min(k + 1, n)


def test_matches_lexsort_on_random_rows():
    rng = np.random.default_rng(7)
    B, n, k = 6, 300, 32
    s = rng.integers(-50, 50, size=(B, n)).astype(np.int32)   # many ties
    lens = np.array([n * 4, n * 4 - 3, 137 * 4, 4 * 33, 4 * 34, 1], np.int32)
    sel, n_sel, drops, W = _select(s, lens, k)
    for b in range(B):
        nb = -(-int(lens[b]) // 4)
        if nb - 1 <= k:
            want = list(range(nb))
        else:
            cand = np.arange(nb - 1)
            order = np.lexsort((cand, -s[b, :nb - 1].astype(np.int64)))
            want = sorted(cand[order[:k]].tolist() + [nb - 1])
        assert sel[b][:n_sel[b]].tolist() == want, b
        assert (sel[b][n_sel[b]:] == -1).all()


def test_extreme_scores_and_edge_lengths():
    i32 = np.iinfo(np.int32)
    s = np.array([[i32.max, i32.min, 0, i32.max, i32.min, -1, 5, 5]], np.int32)
    sel, n_sel, _, _ = _select(s, [8 * 4], k=3)
    assert sel[0][:4].tolist() == [0, 3, 6, 7]
    sel, n_sel, _, _ = _select(s, [0], k=3)           # empty request
    assert n_sel[0] == 0 and (sel[0] == -1).all()
    sel, n_sel, _, _ = _select(s, [1], k=3)           # one token: one page
    assert sel[0][:2].tolist() == [0, -1]
    sel, n_sel, _, _ = _select(s, [3 * 4 + 1], k=3)   # 4 pages, n - 1 == k: all of them
    assert sel[0][:5].tolist() == [0, 1, 2, 3, -1]
    sel, n_sel, _, _ = _select(s, [4 * 4 + 1], k=3)   # 5 pages: top-3 of 0..3, plus 4
    assert sel[0][:5].tolist() == [0, 2, 3, 4, -1]


def test_width_formula():
    assert oracle.max_sel_pages(32) == 72
    assert oracle.max_sel_pages(16) == 40
