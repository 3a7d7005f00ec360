"""GPU parity of the top-k preload (ssa_prefetch_pages) in a decode loop.

The runner issues each step's preload on a second stream after the step's
remap, overlapping its attention and the next step's indexer; the next
step's ensure waits for it.  The oracle runs the same sequence (step, then
or_prefetch with the step's scores).  Every step: the scores the preload
read, its fetch lists and counts, and then the whole residency state bit
for bit, besides everything the plain parity loop compares; pool bytes of
every bound slot after the last step.
"""
import math

import pytest

import workloads as wl
from tests.parity import run_parity

pytestmark = pytest.mark.gpu


def _w(name, **kw):
    base = dict(batch=2, n_layers=2, ctx=64 * 120 + 9, page_size=64, n_q_heads=16, n_kv_heads=2,
                head_dim=128, fp8=True, block_topk=8, pool_slots=2 * 24 + 5, steps=8, rho=0.9,
                walk_c=math.sqrt(1 - 0.81), seed=400)
    base.update(kw)
    return wl.Workload(name, **base)


CASES = [
    # the pool holds exactly the batch's candidates; wide preload
    (_w("fp8_tight_pool"), 2 * 8 + 8),
    # narrow preload, ragged requests, bf16
    (_w("bf16_ragged", fp8=False, seq_lens=(64 * 120 + 9, 64 * 77 + 40), seed=401), 12),
    # a large pool (most candidates already resident), rho = 0.95
    (_w("fp8_large_pool", batch=1, ctx=64 * 600, block_topk=32, pool_slots=300, rho=0.95,
        walk_c=0.31, steps=10, seed=402), 48),
    # width k + 1: the candidates are the step's own selection (nothing to fetch)
    (_w("fp8_width_k_plus_1", seed=403), 9),
]


@pytest.mark.parametrize("w,width", CASES, ids=[c[0].name for c in CASES])
def test_preload_parity(w, width):
    rep = {}
    run_parity(w, pool_every_step=False, preload_width=width, report=rep)
    if width > w.block_topk + 1:
        assert rep["fetched"] > 0
    else:
        assert rep["fetched"] == 0
    print(w.name, rep)
