"""Top-k selection under heavy ties, GPU against the oracle, bit-exact.

Scores that tie are ranked by page id (lower first).  Three cases: every
score equal (a zero query), three distinct page keys repeated over hundreds
of pages, and scores spanning the whole int range with duplicates.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.parity import gpu_runner, oracle_state

pytestmark = pytest.mark.gpu


def _run_case(w, k_bits, v_bits, pos, q_bits):
    orc = oracle_state(w)
    run = gpu_runner(w)
    orc.store(0, k_bits, v_bits, pos)
    kd = torch.from_numpy(k_bits.view(np.int16)).view(torch.bfloat16).cuda()[None]
    vd = torch.from_numpy(v_bits.view(np.int16)).view(torch.bfloat16).cuda()[None]
    run.store(0, 1, kd, vd, torch.from_numpy(pos).cuda())
    import sparse_attention_decode_indexer_gb300 as ssa
    qd = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()[None]
    ssa.ssa_index_topk(run.cache, 0, 1, qd, run.block_table, run.seq_lens, run.sel, run.n_sel,
                       run.scores, run.status, run.ws)
    torch.cuda.synchronize()
    sel, n_sel, scores, drops, bad = orc.index_topk(0, q_bits, wl.block_table(w), w.lens)
    assert int(run.status.item()) == 0
    assert np.array_equal(run.scores[0].cpu().numpy(), scores)
    assert np.array_equal(run.sel[0].cpu().numpy(), sel)
    assert np.array_equal(run.n_sel[0].cpu().numpy(), n_sel)
    return sel, scores


def _w(**kw):
    base = dict(batch=3, n_layers=1, ctx=64 * 300, page_size=64, n_q_heads=16, n_kv_heads=2,
                head_dim=128, fp8=False, block_topk=32, pool_slots=None, seed=401,
                seq_lens=(64 * 300, 64 * 257 + 3, 64 * 40))
    base.update(kw)
    return wl.Workload("ties", **base)


def test_zero_query_selects_lowest_pages():
    w = _w()
    k, v, pos = wl.store_batch(w, 0)
    q = np.zeros((w.batch, w.n_q_heads, w.head_dim), np.uint16)
    sel, scores = _run_case(w, k, v, pos, q)
    assert (scores[0, :300] == 0).all()
    assert sel[0][:33].tolist() == list(range(32)) + [299]


def test_three_key_patterns_over_hundreds_of_pages():
    w = _w()
    rng = np.random.default_rng([w.seed, 9])
    pats = rng.standard_normal((3, w.n_kv_heads, w.head_dim)).astype(np.float32)
    k, v, pos = wl.store_batch(w, 0)
    page_pat = rng.integers(0, 3, size=int(pos.max()) // w.page_size + 1)
    kf = pats[page_pat[pos // w.page_size]]                 # every token = its page's pattern
    k = wl.to_bf16_bits(kf)
    q = wl.queries(w, 0)[0]
    sel, scores = _run_case(w, k, v, pos, q)
    assert len(np.unique(scores[0, :299])) <= 3


def test_wide_range_scores_with_duplicates():
    w = _w(seed=402)
    k, v, pos = wl.store_batch(w, 0)
    kf = wl.bf16_bits_to_f32(k).reshape(len(pos), w.n_kv_heads, w.head_dim)
    kf *= np.float32(1000.0)                                # large magnitudes
    pg = pos // w.page_size
    kf[pg % 7 == 0] = kf[0]                                 # many duplicate pages
    q = wl.to_bf16_bits(np.float32(50.0) * wl.query_walk_f32(w, 0)[0])
    _run_case(w, wl.to_bf16_bits(kf), v, pos, q)
