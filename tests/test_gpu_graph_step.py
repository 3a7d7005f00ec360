"""DecodeRunner.step as a CUDA graph replay (graphs=True) against eager steps.

A serving loop keeps one query buffer and replays the step's launches.  The
first call with that buffer runs the step eagerly and records the launches;
every later call replays them.  Each step of a host-tier workload with
misses (the LRU evicts and fetches every step) must leave the same bits as
an eager runner fed the same queries: output, selection, remap, miss count
and the whole residency state -- in particular the first call must not run
the step twice (the clock advances once per step).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.parity import _u16_to_bf16, gpu_runner, prefill

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fetch", [False, True])
def test_graph_replay_equals_eager_steps(fetch):
    w = wl.Workload("graph_step", batch=3, n_layers=3, ctx=64 * 60, page_size=64, n_q_heads=16,
                    n_kv_heads=2, head_dim=128, fp8=True, block_topk=6, pool_slots=3 * 20 + 4,
                    steps=8, rho=0.8, walk_c=0.6, seed=170)
    eager = gpu_runner(w, fetch_in_attention=fetch)
    graphed = gpu_runner(w, fetch_in_attention=fetch)
    graphed.graphs = True
    prefill(w, eager, None, [])
    prefill(w, graphed, None, [])
    qs = np.stack([wl.queries(w, l) for l in range(w.n_layers)], axis=1)   # [steps][L]...
    q_buf = torch.empty((w.n_layers, w.batch, w.n_q_heads, w.head_dim), dtype=torch.bfloat16,
                        device="cuda")
    misses = 0
    for t in range(w.steps):
        q = _u16_to_bf16(qs[t]).cuda()
        eager.step(q)
        q_buf.copy_(q)
        graphed.step(q_buf)
        torch.cuda.synchronize()
        assert int(eager.status.item()) == 0 and int(graphed.status.item()) == 0
        assert torch.equal(eager.out, graphed.out), f"out, step {t}"
        for name in ("sel", "n_sel", "phys", "n_miss"):
            assert torch.equal(getattr(eager, name), getattr(graphed, name)), f"{name}, step {t}"
        for name in ("slot_of", "page_of", "last_use", "clock"):
            assert torch.equal(getattr(eager.cache, name), getattr(graphed.cache, name)), \
                f"{name}, step {t}"
        misses += int(eager.n_miss.sum().item())
    assert len(graphed._graphs) == 1
    assert misses > 0
