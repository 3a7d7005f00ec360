"""GPU parity of the zero-copy host-tail attention (ssa_sparse_paged_decode_host_tail).

Selected pages without a pool slot are read straight from the pinned host
mirror inside the attention kernel; resident ones from the pool.  The
residency state must not change.  Expected values: the oracle's attention
over the same selected tokens read from its own mirror (which holds the
pool's bytes for every page), within the tolerance of the other parity tests.
Cases: a pool warmed by two ordinary steps (a mix of resident and host
pages), an empty pool (every page from the host), ragged requests, fp8 and
bf16, several page sizes.
"""
import math

import numpy as np
import pytest
import torch

import workloads as wl
from tests.parity import TOL, _u16_to_bf16, gpu_runner, oracle_state, prefill

pytestmark = pytest.mark.gpu


def _w(name, **kw):
    base = dict(batch=2, n_layers=2, ctx=64 * 100 + 17, page_size=64, n_q_heads=16,
                n_kv_heads=2, head_dim=128, fp8=True, block_topk=12, pool_slots=2 * 32 + 3,
                steps=6, rho=0.9, walk_c=math.sqrt(1 - 0.81), seed=500)
    base.update(kw)
    return wl.Workload(name, **base)


CASES = [
    (_w("fp8_warm_pool"), 2),
    (_w("fp8_cold_pool"), 0),
    (_w("bf16_ragged_warm", fp8=False, seq_lens=(64 * 100 + 17, 64 * 41 + 3), seed=501), 2),
    (_w("fp8_p32_g4", page_size=32, ctx=32 * 150 + 5, n_q_heads=8, n_kv_heads=2, seed=502), 1),
    (_w("bf16_p128", page_size=128, ctx=128 * 60 + 33, fp8=False, block_topk=6,
        pool_slots=2 * 20 + 1, seed=503), 1),
]


@pytest.mark.parametrize("w,warm", CASES, ids=[c[0].name for c in CASES])
def test_host_tail_parity(w, warm):
    import sparse_attention_decode_indexer_gb300 as ssa
    orc = oracle_state(w)
    run = gpu_runner(w)
    prefill(w, run, orc, oracle_layers=list(range(w.n_layers)))
    qs = {l: wl.queries(w, l) for l in range(w.n_layers)}
    bt = wl.block_table(w)
    L = w.n_layers
    for t in range(warm):                 # ordinary steps: the pool holds some pages
        run.step(_u16_to_bf16(np.stack([qs[l][t] for l in range(L)])).cuda())
    torch.cuda.synchronize()
    assert int(run.status.item()) == 0
    host_pages = 0
    for t in range(warm, w.steps):
        q = _u16_to_bf16(np.stack([qs[l][t] for l in range(L)])).cuda()
        before = [x.clone() for x in (run.cache.slot_of, run.cache.page_of, run.cache.last_use,
                                      run.cache.clock)]
        ssa.ssa_index_topk(run.cache, 0, L, q, run.block_table, run.seq_lens, run.sel, run.n_sel,
                           None, run.status, run.ws)
        ssa.ssa_sparse_paged_decode_host_tail(run.cache, 0, L, q, run.sel, run.block_table,
                                              run.seq_lens, run.sm_scale, run.out, run.status,
                                              run.ws)
        torch.cuda.synchronize()
        assert int(run.status.item()) == 0, ssa.status_str(int(run.status.item()))
        for a, b in zip(before, (run.cache.slot_of, run.cache.page_of, run.cache.last_use,
                                 run.cache.clock)):
            assert torch.equal(a, b), "the host-tail attention changed the residency state"
        for l in range(L):
            sel = run.sel[l].cpu().numpy()
            want = orc.decode_from_mirror(l, qs[l][t], sel, bt, w.lens)
            got = run.out[l].float().cpu().numpy()
            err = float(np.abs(got - want).max())
            assert err <= TOL[w.fp8], f"max abs err {err} layer {l} step {t}"
            so = run.cache.slot_of[l].cpu().numpy()
            for b in range(w.batch):
                ids = bt[b][sel[b][sel[b] >= 0]]
                host_pages += int((so[ids] < 0).sum())
    assert host_pages > 0
    print(w.name, "host pages read", host_pages)
