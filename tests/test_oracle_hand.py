"""Pins: the hand-worked 4-page example and the hand LRU trace (tests/golden/)."""
import json
import os

import numpy as np
import pytest

import oracle
from workloads import to_bf16_bits

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _hand_state(block_topk, host_tier=False):
    g = _load("hand_example_4page.json")
    lay = oracle.OracleLayout(page_size=2, n_q_heads=1, n_kv_heads=1, head_dim=2, fp8=False,
                              n_layers=1, logical_pages=4, pool_slots=4, batch=1, max_pages=4,
                              block_topk=block_topk)
    kv = oracle.OracleKV(lay, host_tier=host_tier, identity=True)
    k = to_bf16_bits(np.array(g["k_rows"], np.float32).reshape(8, 1, 2))
    v = to_bf16_bits(np.array(g["v_rows"], np.float32).reshape(8, 1, 2))
    assert kv.store(0, k, v, np.arange(8, dtype=np.int64)) == 0
    return g, kv


def test_hand_example_slab_scores_selection_output():
    g, kv = _hand_state(block_topk=2)
    assert kv.slab[0].reshape(4, 2).tolist() == g["slab_codes"]
    assert np.allclose(kv.slab_sum[0].reshape(4, 2) / kv.slab_cnt[0][:, None], g["page_means"])
    q = to_bf16_bits(np.array(g["q"], np.float32).reshape(1, 1, 2))
    bt = np.arange(4, dtype=np.int32).reshape(1, 4)
    sl = np.array([8], np.int32)
    r = kv.step(0, q, bt, sl)
    assert r["scores"][0].tolist() == g["scores"]
    assert r["sel"][0].tolist() == g["selected"]
    assert int(r["n_sel"][0]) == 3
    assert r["phys"][0].tolist() == g["selected"]          # identity pool
    assert r["drops"] == 0 and r["n_miss"] == 0
    np.testing.assert_allclose(r["out"][0, 0], g["out"], rtol=0, atol=1e-9)


def test_hand_example_all_pages_is_dense_attention():
    g, kv = _hand_state(block_topk=3)
    q = to_bf16_bits(np.array(g["q"], np.float32).reshape(1, 1, 2))
    r = kv.step(0, q, np.arange(4, dtype=np.int32).reshape(1, 4), np.array([8], np.int32))
    assert r["sel"][0][:4].tolist() == [0, 1, 2, 3]
    np.testing.assert_allclose(r["out"][0, 0], g["out_all_pages"], rtol=0, atol=1e-9)


def test_hand_example_zero_query_ties_go_to_lower_page():
    g, kv = _hand_state(block_topk=2)
    q = to_bf16_bits(np.zeros((1, 1, 2), np.float32))
    sel, n_sel, scores, drops, bad = kv.index_topk(
        0, q, np.arange(4, dtype=np.int32).reshape(1, 4), np.array([8], np.int32))
    assert scores[0].tolist() == [0, 0, 0, 0]
    assert sel[0].tolist() == g["zero_query_selected"]


def _lru(S, Lp, B, W):
    lay = oracle.OracleLayout(page_size=1, n_q_heads=1, n_kv_heads=1, head_dim=1, fp8=False,
                              n_layers=1, logical_pages=Lp, pool_slots=S, batch=B,
                              max_pages=Lp, block_topk=1, max_sel_override=W)
    return oracle.OracleKV(lay, host_tier=True, identity=False)


def test_hand_lru_trace():
    g = _load("lru_trace_s3.json")
    kv = _lru(S=3, Lp=6, B=1, W=2)
    bt = np.arange(6, dtype=np.int32).reshape(1, 6)
    for st in g["steps"]:
        sel = np.array([st["selected"]], np.int32)
        mp, ms, nm, flags = kv.ensure(0, sel, bt)
        assert flags == 0
        assert mp[:nm].tolist() == st["misses"]
        assert ms[:nm].tolist() == st["miss_slots"]
        assert kv.page_of[0].tolist() == st["page_of"]
        assert kv.last_use[0].tolist() == st["last_use"]
        assert int(kv.clock[0]) == st["clock"]


def test_hand_lru_shared_page_is_one_miss():
    g = _load("lru_trace_s3.json")["shared_page"]
    kv = _lru(S=4, Lp=6, B=2, W=2)
    bt = np.tile(np.arange(6, dtype=np.int32), (2, 1))
    mp, ms, nm, flags = kv.ensure(0, np.array(g["selected"], np.int32), bt)
    assert mp[:nm].tolist() == g["misses"]
    assert ms[:nm].tolist() == g["miss_slots"]
    assert kv.page_of[0].tolist() == g["page_of"]
    assert int(kv.clock[0]) == g["clock"]
