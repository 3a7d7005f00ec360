"""The indexer's work split, GPU against the oracle, bit-exact.

The score CTAs of a call cover its rows (layer, request): each row is cut
into chunks of whole rounds of pages, as many as one wave of resident CTAs
holds, and the last CTA of a row to finish (an atomic ticket) selects it.
With more rows than the wave holds every row is one CTA and the CTAs run in
several waves.  Cases: ragged request lengths with rows cut into chunks,
512 and 1,152 short rows, 520 rows of 4 KV heads (32 lanes per page).
Scores, selections and counts equal the oracle's for every layer, on two
calls in a row (the tickets return to zero).  FreeToken PR #499, "Why this
works for sparse attention" and "Design": the indexer over the slab and the
fixed-shape selection.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.parity import _u16_to_bf16, gpu_runner, oracle_state

pytestmark = pytest.mark.gpu


def _w(name, **kw):
    base = dict(batch=4, n_layers=2, ctx=64 * 40, page_size=64, n_q_heads=16, n_kv_heads=2,
                head_dim=128, fp8=False, block_topk=8, pool_slots=None, steps=1, seed=160)
    base.update(kw)
    return wl.Workload(name, **base)


def _lens(B, P, n, seed):
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(P * 2, P * n + 1, size=B))


CASES = [
    # few rows, each cut into chunks
    _w("rows_chunked_ragged", batch=3, ctx=64 * 400, seq_lens=_lens(3, 64, 400, 1), seed=161),
    # 8 layers x 64 requests = 512 rows, more than one wave of CTAs holds
    _w("line_two_rows_per_range", batch=64, n_layers=8, ctx=16 * 48, page_size=16,
       n_q_heads=8, n_kv_heads=1, block_topk=4, seq_lens=_lens(64, 16, 48, 2), seed=162),
    # 12 x 96 = 1,152 short rows
    _w("line_many_short_rows", batch=96, n_layers=12, ctx=16 * 12, page_size=16,
       n_q_heads=8, n_kv_heads=1, block_topk=2, seq_lens=_lens(96, 16, 12, 3), seed=163),
    # 4 KV heads (32 lanes per page), 520 rows
    _w("line_4_kv_heads", batch=40, n_layers=13, ctx=32 * 70, page_size=32, n_q_heads=32,
       n_kv_heads=4, block_topk=8, seq_lens=_lens(40, 32, 70, 4), seed=164),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_index_topk_every_layer(w):
    import sparse_attention_decode_indexer_gb300 as ssa
    L = w.n_layers
    orc = oracle_state(w)
    run = gpu_runner(w)
    for l in range(L):
        k, v, pos = wl.store_batch(w, l)
        run.store(l, 1, _u16_to_bf16(k).cuda()[None], _u16_to_bf16(v).cuda()[None],
                  torch.from_numpy(pos).cuda())
        assert orc.store(l, k, v, pos) == 0
    q = np.stack([wl.queries(w, l)[0] for l in range(L)])
    bt = wl.block_table(w)
    for rep in range(2):          # the tickets return to zero: a second call sees the same
        ssa.ssa_index_topk(run.cache, 0, L, _u16_to_bf16(q).cuda(), run.block_table, run.seq_lens,
                           run.sel, run.n_sel, run.scores, run.status, run.ws)
        torch.cuda.synchronize()
        assert int(run.status.item()) == 0
        for l in range(L):
            sel, n_sel, scores, drops, bad = orc.index_topk(l, q[l], bt, w.lens)
            assert drops == 0 and bad == 0
            assert np.array_equal(run.scores[l].cpu().numpy(), scores), f"scores layer {l}"
            assert np.array_equal(run.sel[l].cpu().numpy(), sel), f"sel layer {l}"
            assert np.array_equal(run.n_sel[l].cpu().numpy(), n_sel), f"n_sel layer {l}"
