"""GPU parity of the residency shared by the layers of a call
(ssa_ensure_remap_shared): one LRU state (the first layer's) ensures the union
of every layer's selection, each miss copied into the same slot of every
layer's pool, the remapped table written for every layer.

Each step, against the oracle (its indexer per layer, or_ensure_shared, the
remap of each layer through the shared slot_of, its attention per layer):
scores and selections bit for bit, the shared miss list and count, the
shared state, every layer's remapped table, every layer's pool bytes at the
end, and outputs within tolerance.
"""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from tests.parity import TOL, _u16_to_bf16, gpu_pool_as_oracle_layout, oracle_state, prefill

pytestmark = pytest.mark.gpu


def _w(name, **kw):
    base = dict(batch=2, n_layers=3, ctx=64 * 80 + 21, page_size=64, n_q_heads=16,
                n_kv_heads=2, head_dim=128, fp8=True, block_topk=6, pool_slots=3 * 2 * 20 + 4,
                steps=6, rho=0.8, walk_c=0.6, seed=600)
    base.update(kw)
    return wl.Workload(name, **base)


CASES = [
    _w("fp8_3_layers"),
    _w("bf16_ragged", fp8=False, seq_lens=(64 * 80 + 21, 64 * 33 + 1), seed=601),
    # the pool holds exactly the layers' union of selection widths
    _w("fp8_tight", n_layers=2, batch=3, block_topk=4, pool_slots=2 * 3 * 16, seed=602),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_shared_residency_parity(w):
    from sparse_attention_decode_indexer_gb300 import Layout
    from sparse_attention_decode_indexer_gb300.runner import DecodeRunner
    lay = Layout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8, w.n_layers,
                 w.logical_pages, w.slots, w.batch, w.pages_per_request, w.block_topk)
    run = DecodeRunner(lay, host_tier=True, identity=False, block_table=wl.block_table(w),
                       seq_lens=w.lens, shared_residency=True)
    orc = oracle_state(w)
    L = w.n_layers
    prefill(w, run, orc, oracle_layers=list(range(L)))
    qs = {l: wl.queries(w, l) for l in range(L)}
    bt = wl.block_table(w)
    n_miss = 0
    for t in range(w.steps):
        q = _u16_to_bf16(np.stack([qs[l][t] for l in range(L)])).cuda()
        run.step(q, keep_scores=True)
        torch.cuda.synchronize()
        assert int(run.status.item()) == 0, run.status.item()
        sels = []
        for l in range(L):
            sel, n_sel, scores, drops, bad = orc.index_topk(l, qs[l][t], bt, w.lens)
            assert np.array_equal(run.scores[l].cpu().numpy(), scores)
            assert np.array_equal(run.sel[l].cpu().numpy(), sel)
            sels.append(sel)
        mp, ms, nm, fl = orc.ensure_shared(0, L, np.stack(sels), bt)
        assert fl == 0
        assert int(run.n_miss[0].item()) == nm, f"n_miss step {t}"
        assert np.array_equal(run.miss_page.reshape(-1)[:len(mp)].cpu().numpy(), mp)
        assert np.array_equal(run.miss_slot.reshape(-1)[:len(ms)].cpu().numpy(), ms)
        for name in ("slot_of", "page_of", "last_use"):
            assert np.array_equal(getattr(run.cache, name)[0].cpu().numpy(),
                                  getattr(orc, name)[0]), f"{name} step {t}"
        assert int(run.cache.clock[0].item()) == int(orc.clock[0])
        for l in range(L):
            phys, unresolved = orc.remap_shared(0, l, sels[l], bt)
            assert unresolved == 0
            assert np.array_equal(run.phys[l].cpu().numpy(), phys), f"phys layer {l} step {t}"
            want = orc.decode(l, qs[l][t], sels[l], phys, w.lens)
            err = float(np.abs(run.out[l].float().cpu().numpy() - want).max())
            assert err <= TOL[w.fp8], f"max abs err {err} layer {l} step {t}"
        n_miss += nm
    bound = np.nonzero(orc.page_of[0] >= 0)[0]
    idx = torch.from_numpy(bound).cuda()
    for l in range(L):
        for name, is_v in (("k_pool", False), ("v_pool", True)):
            g = gpu_pool_as_oracle_layout(w, getattr(run.cache, name)[l][idx], is_v)
            assert np.array_equal(g, getattr(orc, name)[l][bound]), f"{name} layer {l}"
    assert n_miss > 0
    print(w.name, "misses", n_miss)
