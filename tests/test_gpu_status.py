"""Device-detected problems surface as bits of the caller's status word.

Every input here is one the kernels' own range checks turn into a status bit
(the access is skipped, nothing faults); the tests check the bit and that
valid parts of the same call still produce correct results.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.parity import gpu_runner, prefill

pytestmark = pytest.mark.gpu


def _w(**kw):
    base = dict(batch=2, n_layers=1, ctx=64 * 20, page_size=64, n_q_heads=16, n_kv_heads=2,
                head_dim=128, fp8=True, block_topk=4, pool_slots=2 * 16 + 4, steps=1, rho=0.8,
                walk_c=0.6, seed=301)
    base.update(kw)
    return wl.Workload("status", **base)


def _q(w):
    q = wl.queries(w, 0)[0][None]
    return torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).cuda()


def test_bad_block_table_id_sets_bad_id():
    import sparse_attention_decode_indexer_gb300 as ssa
    w = _w()
    run = gpu_runner(w)
    prefill(w, run, None, [])
    bt = run.block_table.clone()
    bt[1, 3] = w.logical_pages + 5                 # out of range
    ssa.ssa_index_topk(run.cache, 0, 1, _q(w), bt, run.seq_lens, run.sel, run.n_sel, None,
                       run.status, run.ws)
    torch.cuda.synchronize()
    assert int(run.status.item()) & ssa.ST_BAD_ID


def test_unresolved_page_at_decode_is_skipped_and_flagged():
    import sparse_attention_decode_indexer_gb300 as ssa
    w = _w()
    run = gpu_runner(w)
    prefill(w, run, None, [])
    q = _q(w)
    run.step(q)
    torch.cuda.synchronize()
    assert int(run.status.item()) == 0
    phys = run.phys.clone()
    phys[0, 0, 0] = -1                              # a selected page without a slot
    out = torch.empty_like(run.out)
    ssa.ssa_sparse_paged_decode(run.cache, 0, 1, q, run.sel, phys, run.seq_lens, run.sm_scale,
                                out, run.status, run.ws)
    torch.cuda.synchronize()
    assert int(run.status.item()) & ssa.ST_UNRESOLVED
    # request 1 is untouched by the bad entry
    assert torch.equal(out[0, 1], run.out[0, 1])


def test_miss_without_mirror_is_flagged():
    import sparse_attention_decode_indexer_gb300 as ssa
    from sparse_attention_decode_indexer_gb300 import Layout
    from sparse_attention_decode_indexer_gb300.runner import DecodeRunner
    w = _w()
    lay = Layout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8, w.n_layers,
                 w.logical_pages, w.slots, w.batch, w.pages_per_request, w.block_topk)
    run = DecodeRunner(lay, host_tier=False, identity=False, block_table=wl.block_table(w),
                       seq_lens=w.lens)                  # empty pool, no mirror
    run.step(_q(w))
    torch.cuda.synchronize()
    assert int(run.status.item()) & ssa.ST_MISS_NO_MIRROR


def test_non_increasing_store_positions_are_flagged():
    import sparse_attention_decode_indexer_gb300 as ssa
    w = _w(batch=1)
    run = gpu_runner(w)
    k, v, pos = wl.store_batch(w, 0)
    pos = pos.copy()
    pos[10], pos[11] = pos[11], pos[10]              # swap two tokens of one page
    kd = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).cuda()[None]
    vd = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda()[None]
    run.store(0, 1, kd, vd, torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    assert int(run.status.item()) & ssa.ST_BAD_POS


def test_out_of_range_store_position_is_skipped():
    import sparse_attention_decode_indexer_gb300 as ssa
    w = _w(batch=1)
    run = gpu_runner(w)
    k, v, pos = wl.store_batch(w, 0)
    pos = pos.copy()
    pos[-1] = w.logical_pages * w.page_size + 3      # past the logical page space
    kd = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).cuda()[None]
    vd = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda()[None]
    run.store(0, 1, kd, vd, torch.from_numpy(pos).cuda())
    torch.cuda.synchronize()
    assert int(run.status.item()) & ssa.ST_BAD_ID
    assert int(run.cache.slab_cnt[0].sum().item()) == len(pos) - 1


def test_lost_arrival_ends_in_timeout_status_not_a_hang():
    import time
    import sparse_attention_decode_indexer_gb300 as ssa
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    t0 = time.time()
    ssa.ssa_selftest_bounded_wait(status)
    torch.cuda.synchronize()
    dt = time.time() - t0
    assert int(status.item()) == ssa.ST_TIMEOUT
    assert 0.5 < dt < 30.0
    # the context is still usable
    x = torch.arange(10, device="cuda").sum()
    assert int(x.item()) == 45


def test_attention_is_bitwise_deterministic_across_calls():
    # units split across CTAs are merged by whichever piece finishes last;
    # both merge paths do the same arithmetic, so repeated calls agree bit
    # for bit (many units of a few pages, ragged lengths: many merges)
    import sparse_attention_decode_indexer_gb300 as ssa
    w = wl.Workload("det", batch=24, n_layers=2, ctx=64 * 30,
                    seq_lens=tuple(64 * 30 if i % 3 == 0 else (i * 211) % (64 * 30) + 1
                                   for i in range(24)),
                    page_size=64, n_q_heads=16, n_kv_heads=2, head_dim=128, fp8=True,
                    block_topk=8, pool_slots=None, seed=311)
    run = gpu_runner(w)
    prefill(w, run, None, [])
    q = torch.from_numpy(np.stack([wl.queries(w, l)[0] for l in range(2)]).view(np.int16)).view(
        torch.bfloat16).cuda()
    run.step(q)
    torch.cuda.synchronize()
    ref = run.out.clone()
    for _ in range(6):
        out = torch.empty_like(run.out)
        ssa.ssa_sparse_paged_decode(run.cache, 0, 2, q, run.sel, run.phys, run.seq_lens,
                                    run.sm_scale, out, run.status, run.ws)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert int(run.status.item()) == 0
