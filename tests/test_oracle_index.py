"""Pins for the oracle's slab (int8 page-mean keys) and indexer scores.

The slab and q8 quantisers are checked against a vectorised numpy float32
restatement (different loop structure, library rint) and against invariants
of symmetric int8 quantisation; the int32 scores against numpy int64 einsum
with the KV heads expanded by np.repeat, which pins the query-head to KV-head
mapping (hq -> hq // G) and catches any transposed operand.
"""
import numpy as np
import pytest

import oracle
from workloads import Workload, bf16_bits_to_f32, block_table, queries, store_batch


def _state(w: Workload):
    lay = oracle.OracleLayout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8,
                              w.n_layers, w.logical_pages, w.slots, w.batch,
                              w.pages_per_request, w.block_topk)
    return oracle.OracleKV(lay, host_tier=w.host_tier, identity=not w.host_tier)


W_SMALL = Workload("pin", batch=3, n_layers=1, ctx=40 * 16 + 5, page_size=16, n_q_heads=8,
                   n_kv_heads=2, head_dim=32, fp8=False, block_topk=6, pool_slots=None,
                   seed=11, seq_lens=(40 * 16 + 5, 17 * 16, 3 * 16 - 1))


def _numpy_slab(k_bits, pos, Lp, P, HD):
    x = bf16_bits_to_f32(k_bits).reshape(-1, HD)
    page = pos // P
    s = np.zeros((Lp, HD), np.float32)
    cnt = np.zeros((Lp,), np.int32)
    for t in range(x.shape[0]):            # token order, one fp32 add each
        s[page[t]] = s[page[t]] + x[t]
        cnt[page[t]] += 1
    codes = np.zeros((Lp, HD), np.int8)
    for p in np.nonzero(cnt)[0]:
        mean = s[p] / np.float32(cnt[p])
        amax = np.abs(mean).max()
        if amax > 0:
            sc = amax / np.float32(127.0)
            codes[p] = np.clip(np.rint(mean / sc), -127, 127).astype(np.int8)
    return s, cnt, codes


def test_slab_matches_numpy_restatement_and_invariants():
    w = W_SMALL
    kv = _state(w)
    k, v, pos = store_batch(w, 0)
    assert kv.store(0, k, v, pos) == 0
    HD = w.n_kv_heads * w.head_dim
    s, cnt, codes = _numpy_slab(k, pos, w.logical_pages, w.page_size, HD)
    assert np.array_equal(kv.slab_cnt[0], cnt)
    assert np.array_equal(kv.slab_sum[0], s)
    assert np.array_equal(kv.slab[0], codes)
    used = cnt > 0
    # symmetric int8: every used page reaches +-127 somewhere, codes in range
    assert (np.abs(kv.slab[0][used].astype(int)).max(axis=1) == 127).all()
    # dequantised codes are within half a step of the mean
    mean = s[used] / cnt[used][:, None]
    step = kv.slab_scale[0][used][:, None]
    assert (np.abs(kv.slab[0][used] * step - mean) <= 0.5 * step * (1 + 1e-6)).all()


def test_store_in_two_calls_equals_one_call():
    w = W_SMALL
    k, v, pos = store_batch(w, 0)
    a, b = _state(w), _state(w)
    a.store(0, k, v, pos)
    cut = 300                                     # mid-page
    b.store(0, k[:cut], v[:cut], pos[:cut])
    b.store(0, k[cut:], v[cut:], pos[cut:])
    for name in ("slab", "slab_sum", "slab_cnt", "slab_scale", "k_pool", "v_pool"):
        assert np.array_equal(getattr(a, name), getattr(b, name)), name


def test_scores_match_numpy_einsum_with_expanded_heads():
    w = W_SMALL
    kv = _state(w)
    k, v, pos = store_batch(w, 0)
    kv.store(0, k, v, pos)
    q = queries(w, 0)[0]
    bt = block_table(w)
    sel, n_sel, scores, drops, bad = kv.index_topk(0, q, bt, w.lens)
    assert bad == 0 and drops == 0
    # q8, numpy float32
    qf = bf16_bits_to_f32(q).reshape(w.batch, -1)
    amax = np.abs(qf).max(axis=1, keepdims=True)
    q8 = np.clip(np.rint(qf / (amax / np.float32(127.0))), -127, 127).astype(np.int64)
    q8 = q8.reshape(w.batch, w.n_q_heads, w.head_dim)
    slab = kv.slab[0].reshape(w.logical_pages, w.n_kv_heads, w.head_dim).astype(np.int64)
    slab_q = np.repeat(slab, w.group, axis=1)          # KV head h serves hq in [h*G, (h+1)*G)
    for b in range(w.batch):
        n = -(-int(w.lens[b]) // w.page_size)
        want = np.einsum("hd,phd->p", q8[b], slab_q[bt[b, :n]])
        assert np.array_equal(scores[b, :n].astype(np.int64), want)
        assert (scores[b, n:] == np.iinfo(np.int32).min).all()


def test_zero_query_and_zero_page_give_zero_scores():
    w = W_SMALL.with_(batch=1, seq_lens=(64,), ctx=64)
    kv = _state(w)
    zeros = np.zeros((64, w.n_kv_heads, w.head_dim), np.uint16)
    kv.store(0, zeros, zeros, np.arange(64, dtype=np.int64))
    assert (kv.slab[0] == 0).all() and (kv.slab_scale[0] == 0).all()
    q = queries(w, 0)[0]
    sel, n_sel, scores, _, _ = kv.index_topk(0, q, block_table(w), w.lens)
    assert (scores[0, :4] == 0).all()
