"""The overlapped step (DecodeRunner with overlap_groups) against the plain one.

The overlapped step makes the same launches as ssa_ensure_remap's step, split
differently: the LRU update for all layers (ssa_ensure_remap_bind), then the
host-link copy per range of layers (ssa_fetch_misses) with each range's
attention on a second stream behind that range's copy.  Each step of a
host-tier workload whose LRU evicts and fetches every step must leave the same
bits as the plain step fed the same queries -- selection, remap, miss lists,
the residency state and the pool -- for uneven splits of the layers, eagerly
and as a CUDA graph replay.  The attention splits a launch's units over its
CTAs by the launch's size, so a range of layers merges its pieces in another
order than the launch over all layers and rounds differently; its outputs
must equal, bit for bit, the same per-range attention launches made after the
plain step, and agree with the plain step's outputs within the oracle parity
tolerance (their parity with the oracle is tested beside the other modes).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from sparse_attention_decode_indexer_gb300 import ssa_sparse_paged_decode
from tests.parity import TOL, _u16_to_bf16, gpu_runner, prefill

pytestmark = pytest.mark.gpu


def _workload(fp8):
    return wl.Workload("overlap_step", batch=3, n_layers=5, ctx=64 * 60, page_size=64,
                       n_q_heads=16, n_kv_heads=2, head_dim=128, fp8=fp8, block_topk=6,
                       pool_slots=3 * 20 + 4, steps=6, rho=0.8, walk_c=0.6,
                       seed=180 + int(fp8))


@pytest.mark.parametrize("groups,graphs,fp8", [(2, False, True), (3, True, True),
                                               (5, False, False), (4, True, False)])
def test_overlapped_step_equals_plain_step(groups, graphs, fp8):
    w = _workload(fp8)
    plain = gpu_runner(w)
    over = gpu_runner(w, overlap_groups=groups)
    over.graphs = graphs
    assert [n for _, n in over.layer_groups()] == sorted(
        [n for _, n in over.layer_groups()], reverse=True)
    assert sum(n for _, n in over.layer_groups()) == w.n_layers
    prefill(w, plain, None, [])
    prefill(w, over, None, [])
    qs = np.stack([wl.queries(w, l) for l in range(w.n_layers)], axis=1)   # [steps][L]...
    q_buf = torch.empty((w.n_layers, w.batch, w.n_q_heads, w.head_dim), dtype=torch.bfloat16,
                        device="cuda")
    misses = 0
    for t in range(w.steps):
        q = _u16_to_bf16(qs[t]).cuda()
        plain.step(q)
        q_buf.copy_(q)
        over.step(q_buf)
        torch.cuda.synchronize()
        assert int(plain.status.item()) == 0 and int(over.status.item()) == 0
        # the plain step's pages and phys, attended range by range
        ref = torch.empty_like(plain.out)
        for l0, n in over.layer_groups():
            sl = slice(l0, l0 + n)
            ssa_sparse_paged_decode(plain.cache, l0, n, q[sl], plain.sel[sl], plain.phys[sl],
                                    plain.seq_lens, plain.sm_scale, ref[sl], plain.status,
                                    plain.ws)
        torch.cuda.synchronize()
        assert torch.equal(ref, over.out), f"out against per-range launches, step {t}"
        diff = (plain.out.float() - over.out.float()).abs().max().item()
        assert diff <= TOL[fp8], f"out against the all-layer launch, step {t}: {diff}"
        for name in ("sel", "n_sel", "phys", "n_miss", "miss_page", "miss_slot"):
            assert torch.equal(getattr(plain, name), getattr(over, name)), f"{name}, step {t}"
        for name in ("slot_of", "page_of", "last_use", "clock", "k_pool", "v_pool"):
            assert torch.equal(getattr(plain.cache, name), getattr(over.cache, name)), \
                f"{name}, step {t}"
        if fp8:
            for name in ("k_scale", "v_scale"):
                assert torch.equal(getattr(plain.cache, name), getattr(over.cache, name)), name
        misses += int(plain.n_miss.sum().item())
    assert misses > 0
    if graphs:
        assert len(over._graphs) == 1
