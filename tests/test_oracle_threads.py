"""The oracle's parallel loops give the same bytes at any thread count.

Each output element (a token's codes, a page's slab row, a score, a
request's selection, a (request, head) attention row) is computed by one
thread in the order the code states, so one thread and every core must agree
exactly, on a workload with ragged requests, a host tier and misses.
"""
import numpy as np

import oracle
from workloads import Workload, block_table, queries, store_batch


def _run(threads):
    w = Workload("threads", batch=3, n_layers=1, ctx=64 * 30 + 7,
                 seq_lens=(64 * 30 + 7, 64 * 11, 200), page_size=64, n_q_heads=8,
                 n_kv_heads=2, head_dim=128, fp8=True, block_topk=6, pool_slots=3 * 20 + 1,
                 steps=3, rho=0.8, walk_c=0.6, seed=31)
    lay = oracle.OracleLayout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8, 1,
                              w.logical_pages, w.slots, w.batch, w.pages_per_request,
                              w.block_topk)
    oracle.set_threads(threads)
    try:
        kv = oracle.OracleKV(lay, host_tier=True, identity=False)
        k, v, pos = store_batch(w, 0)
        assert kv.store(0, k, v, pos) == 0
        qs = queries(w, 0)
        outs = [kv.step(0, qs[t], block_table(w), w.lens) for t in range(w.steps)]
    finally:
        oracle.set_threads(0)
    return kv, outs


def test_results_do_not_depend_on_the_thread_count():
    a, ra = _run(1)
    b, rb = _run(0)
    for name in ("k_pool", "v_pool", "k_scale", "v_scale", "k_mirror", "v_mirror", "slab",
                 "slab_sum", "slab_cnt", "slab_scale", "slot_of", "page_of", "last_use"):
        assert np.array_equal(getattr(a, name), getattr(b, name)), name
    for x, y in zip(ra, rb):
        for key in ("scores", "sel", "n_sel", "miss_page", "miss_slot", "phys", "out"):
            assert np.array_equal(x[key], y[key]), key


def test_store_out_of_order_positions_sum_in_call_order():
    # positions that do not increase take the one-by-one path; its sums equal
    # those of the same tokens stored page by page in the given order
    w = Workload("unordered", batch=1, n_layers=1, ctx=64 * 4, page_size=64, n_q_heads=2,
                 n_kv_heads=1, head_dim=128, fp8=False, block_topk=2, pool_slots=None, seed=32)
    lay = oracle.OracleLayout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8, 1,
                              w.logical_pages, w.slots, w.batch, w.pages_per_request,
                              w.block_topk)
    k, v, pos = store_batch(w, 0)
    order = np.concatenate([np.arange(64, 256), np.arange(0, 64)])   # page 0 last
    one = oracle.OracleKV(lay, host_tier=False, identity=True)
    one.store(0, k[order], v[order], pos[order])
    two = oracle.OracleKV(lay, host_tier=False, identity=True)
    two.store(0, k[64:], v[64:], pos[64:])
    two.store(0, k[:64], v[:64], pos[:64])
    for name in ("slab_sum", "slab_cnt", "slab", "slab_scale", "k_pool", "v_pool"):
        assert np.array_equal(getattr(one, name), getattr(two, name)), name
