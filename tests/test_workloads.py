"""The seeded input generators: determinism, shapes, needle recipe."""
import numpy as np

from workloads import (WORKLOADS, Workload, block_table, bf16_bits_to_f32, needle_pages,
                       query_walk_f32, queries, store_batch, sweep_workload)


def test_presets_have_the_stated_shapes():
    w = WORKLOADS["lru_pressure_64k_fp8"]
    assert (w.batch, w.n_layers, w.pages_per_request, w.slots) == (4, 12, 1024, 320)
    assert w.slots >= w.batch * (2 * w.block_topk + 8)
    w = WORKLOADS["host_tier_196k_fp8"]
    assert (w.pages_per_request, w.slots, w.steps) == (3072, 1635, 64)
    w = WORKLOADS["decode_4k_bf16_resident"]
    assert (w.pages_per_request, w.group) == (256, 8)
    s = sweep_workload(8, True, 0.2)
    assert s.slots == int(np.ceil(0.2 * 8 * 2048)) and s.group == 8


def test_generators_are_deterministic_and_request_major():
    w = Workload("t", batch=2, n_layers=2, ctx=100, page_size=16, n_q_heads=4, n_kv_heads=2,
                 head_dim=16, fp8=False, block_topk=2, pool_slots=None, seed=5,
                 seq_lens=(100, 33))
    k1, v1, p1 = store_batch(w, 1)
    k2, v2, p2 = store_batch(w, 1)
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2) and np.array_equal(p1, p2)
    assert k1.shape == (133, 2, 16) and p1.dtype == np.int64
    assert (np.diff(p1) > 0).all()
    n = w.pages_per_request
    assert p1[100] == n * 16                     # request 1 starts at logical page n
    assert not np.array_equal(store_batch(w, 0)[0], k1)
    bt = block_table(w)
    assert bt.shape == (2, n) and bt[1, 0] == n


def test_query_walk_recipe():
    w = WORKLOADS["lru_pressure_64k_fp8"].with_(batch=1, steps=3)
    qf = query_walk_f32(w, 0)
    rng = np.random.default_rng([w.seed, 0, 2])
    q0 = rng.standard_normal(qf.shape[1:], dtype=np.float32)
    e1 = rng.standard_normal(qf.shape[1:], dtype=np.float32)
    assert np.array_equal(qf[0], q0)
    assert np.array_equal(qf[1], np.float32(0.8) * q0 + np.float32(w.walk_c) * e1)
    assert abs(w.walk_c - 0.6) < 1e-12
    assert queries(w, 0).dtype == np.uint16


def test_needles_shift_the_page_keys_along_the_query():
    w = WORKLOADS["batched_32k_bf16_needles"].with_(n_layers=1, ctx=64 * 40)
    pages = needle_pages(w)
    assert pages.shape == (4, 4) and (pages < w.pages_per_request - 1).all()
    k, v, pos = store_batch(w, 0)
    q = bf16_bits_to_f32(queries(w, 0)[0])                  # [B][Hq][D]
    kf = bf16_bits_to_f32(k).reshape(w.batch, -1, w.n_kv_heads, w.head_dim)
    qh = q.reshape(w.batch, w.n_kv_heads, w.group, -1).sum(2)
    qh /= np.linalg.norm(qh, axis=-1, keepdims=True)
    P = w.page_size
    for b in range(w.batch):
        means = kf[b].reshape(-1, P, w.n_kv_heads, w.head_dim).mean(1)
        proj = (means * qh[b][None]).sum(-1).sum(-1)        # per page
        top = set(np.argsort(-proj)[:4].tolist())
        assert top == set(pages[b].tolist())
