"""Stores in pieces of every size: both work splits of the store path.

A call of fewer than 4,096 tokens runs one CTA per token; a longer one runs
one CTA per page-sized chunk of tokens, which handles every run of a page
that starts inside its chunk.  Each case stores a ragged context in pieces
whose edges fall inside pages (so runs start mid-page, cross the chunks'
edges, and continue pages written by an earlier call), once with a long
first call and short ones after it, once the other way round.  After every
call the mirror, the pool of resident pages, the fp8 scales and the slab
equal the oracle's after the same calls, bit for bit (FreeToken PR #499,
"Design": the write-through store; PR #525: the host copy holds the
quantised codes and their scales).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.parity import (_u16_to_bf16, compare_mirror, compare_slab, compare_state,
                          gpu_runner, oracle_state)

pytestmark = pytest.mark.gpu


def _w(name, **kw):
    base = dict(batch=3, n_layers=2, ctx=3000, seq_lens=(3000, 2501, 1699), page_size=64,
                n_q_heads=16, n_kv_heads=2, head_dim=128, fp8=True, block_topk=4,
                pool_slots=None, steps=1, seed=140)
    base.update(kw)
    return wl.Workload(name, **base)


CASES = [
    _w("store_fp8_p64_host_tier", pool_slots=60, seed=141),
    _w("store_bf16_p16_resident", page_size=16, n_kv_heads=1, n_q_heads=8, fp8=False, seed=142),
    _w("store_fp8_p128_h4", page_size=128, n_kv_heads=4, n_q_heads=32, seed=143),
    _w("store_bf16_p32_host_tier", page_size=32, fp8=False, pool_slots=3 * 12 + 40, seed=144),
]
SPLITS = {"long_first": (0.0, 0.7, 0.85, 1.0), "short_first": (0.0, 0.1, 1.0)}


@pytest.mark.parametrize("split", list(SPLITS))
@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_store_in_pieces(w, split):
    fr = SPLITS[split]
    L = w.n_layers
    orc = oracle_state(w)
    run = gpu_runner(w)
    data = [wl.store_batch(w, l) for l in range(L)]
    starts = np.concatenate([[0], np.cumsum(w.lens)[:-1]])
    lens = [int(x) for x in w.lens]
    cuts = [[int(round(f * n)) for f in fr] for n in lens]
    sizes = []
    for i in range(len(fr) - 1):
        idx = np.concatenate([np.arange(s + c[i], s + c[i + 1]) for s, c in zip(starts, cuts)])
        sizes.append(len(idx))
        k = np.stack([data[l][0][idx] for l in range(L)])
        v = np.stack([data[l][1][idx] for l in range(L)])
        pos = data[0][2][idx]
        run.store(0, L, _u16_to_bf16(k).cuda(), _u16_to_bf16(v).cuda(), torch.from_numpy(pos).cuda())
        for l in range(L):
            assert orc.store(l, data[l][0][idx], data[l][1][idx], pos) == 0
        torch.cuda.synchronize()
        assert int(run.status.item()) == 0
        for l in range(L):
            compare_slab(run, orc, l)
            compare_mirror(w, run, orc, l)
            compare_state(w, run, orc, l, check_pool=True)
    # both work splits ran
    assert max(sizes) >= 4096 and min(sizes) < 4096
