"""Attention over selections the indexer never produces.

The attention kernel cuts its work by the weight min(max_pages, block_topk + 1)
per (layer, request, KV head) and maps each CTA's share onto the row's valid
entries.  Whatever the rows hold, every valid entry must be attended exactly
once: rows with more valid entries than block_topk + 1, fewer, holes of -1
between valid entries, unsorted and repeated page ids, and a row with no valid
entry (zeros).  Compared with the fp64 oracle on the same rows, twice in a row
(the split tickets must come back to zero).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.parity import TOL, _u16_to_bf16, gpu_runner, oracle_state, prefill

pytestmark = pytest.mark.gpu


def _w(name, **kw):
    base = dict(batch=3, n_layers=2, ctx=64 * 30 + 17, page_size=64, n_q_heads=16,
                n_kv_heads=2, head_dim=128, fp8=False, block_topk=4, pool_slots=None, steps=1,
                seed=41)
    base.update(kw)
    return wl.Workload(name, **base)


CASES = [
    _w("sel_bf16_p64"),
    _w("sel_fp8_p32", page_size=32, ctx=32 * 50 + 5, fp8=True, n_q_heads=8, seed=42),
]


def _rows(w: wl.Workload, rng) -> np.ndarray:
    n, W = w.pages_per_request, 2 * w.block_topk + 8
    sel = np.full((w.n_layers, w.batch, W), -1, np.int32)
    for l in range(w.n_layers):
        for b in range(w.batch):
            kind = (l * w.batch + b) % 5
            if kind == 0:                       # every slot valid, unsorted
                sel[l, b] = rng.permutation(n)[:W]
            elif kind == 1:                     # one valid entry
                sel[l, b, 0] = n - 1
            elif kind == 2:                     # valid entries at even slots only
                m = min(n, W // 2)
                sel[l, b, 0:2 * m:2] = rng.choice(n, m, replace=False)
            elif kind == 3:                     # repeated ids at the end of the row
                sel[l, b, W - 3:] = [0, 0, n - 1]
            # kind 4: no valid entry
    return sel


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_decode_over_arbitrary_selections(w):
    import sparse_attention_decode_indexer_gb300 as ssa
    rng = np.random.default_rng([w.seed, 9])
    orc = oracle_state(w)
    run = gpu_runner(w)
    prefill(w, run, orc, list(range(w.n_layers)))
    sel = _rows(w, rng)
    bt = wl.block_table(w)
    phys = np.where(sel >= 0, np.take_along_axis(bt[None], np.maximum(sel, 0), axis=2), -1)
    phys = phys.astype(np.int32)        # resident, identity binding: slot = logical page
    q = np.stack([wl.queries(w, l)[0] for l in range(w.n_layers)])
    qd = _u16_to_bf16(q).cuda()
    sel_d = torch.from_numpy(sel).cuda()
    phys_d = torch.from_numpy(phys).cuda()
    expect = [orc.decode(l, q[l], sel[l], phys[l], w.lens) for l in range(w.n_layers)]
    for rep in range(2):
        out = torch.full_like(run.out, float("nan"))
        ssa.ssa_sparse_paged_decode(run.cache, 0, w.n_layers, qd, sel_d, phys_d, run.seq_lens,
                                    run.sm_scale, out, run.status, run.ws)
        torch.cuda.synchronize()
        assert int(run.status.item()) == 0
        got = out.float().cpu().numpy()
        for l in range(w.n_layers):
            err = float(np.abs(got[l] - expect[l]).max())
            assert err <= TOL[w.fp8], f"rep {rep} layer {l}: max abs err {err}"
        # the request without a valid entry gets zeros
        assert not np.any(got[1, 1]), "empty row must give zeros"
