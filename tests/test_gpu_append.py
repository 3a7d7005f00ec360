"""The append path of a decode loop: each step stores the token it produced.

A request's context is written in pieces: a prefill of all but its last A
tokens, then one token per request per store call (every layer in one
launch), each followed by a decode step at the new lengths, as a serving loop
runs.  The appends fill partly written pages and open new ones; with a host
tier the page being filled is resident (the last page is always selected) or
not, so the store writes the mirror always and the pool slot when bound.
After every step the library's mirror, pool, fp8 scales, slab and LRU state
equal the oracle's after the same calls, the selection, remap and misses are
bit-exact, and the attention output is within tolerance.  (That the slab of a
context stored in pieces equals the slab of one store of it is pinned on the
CPU side.)
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests.parity import (TOL, _u16_to_bf16, compare_mirror, compare_slab, compare_state,
                          gpu_runner, oracle_state)

pytestmark = pytest.mark.gpu

A = 40   # tokens appended per request, one per step


def _w(name, **kw):
    base = dict(batch=3, n_layers=2, ctx=64 * 30 + 5, seq_lens=(64 * 30 + 5, 64 * 20 + 40, 600),
                page_size=64, n_q_heads=16, n_kv_heads=2, head_dim=128, fp8=False, block_topk=4,
                pool_slots=None, steps=A, rho=0.8, walk_c=0.6, seed=120)
    base.update(kw)
    return wl.Workload(name, **base)


CASES = [
    # host tier with eviction pressure: 90 logical pages, 50 slots
    _w("append_fp8_host_tier", fp8=True, pool_slots=50, seed=121),
    # fully resident: every append also writes its pool slot
    _w("append_bf16_resident", seed=122),
    # 32-token pages, 4 KV heads
    _w("append_fp8_p32_h4", page_size=32, ctx=32 * 40 + 3, seq_lens=(32 * 40 + 3, 32 * 25, 97),
       n_q_heads=16, n_kv_heads=4, fp8=True, pool_slots=3 * 16 + 20, seed=123),
]


def _split(w: wl.Workload, layer: int):
    """The layer's tokens as one prefill (all but the last A of each request)
    and A append calls of one token per request."""
    k, v, pos = wl.store_batch(w, layer)
    starts = np.concatenate([[0], np.cumsum(w.lens)[:-1]])
    pre = np.concatenate([np.arange(s, s + n - A) for s, n in zip(starts, w.lens)])
    steps = [np.array([s + n - A + i for s, n in zip(starts, w.lens)]) for i in range(A)]
    return (k[pre], v[pre], pos[pre]), [(k[i], v[i], pos[i]) for i in steps]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_append_then_decode_each_step(w):
    assert int(w.lens.min()) > A
    L = w.n_layers
    orc = oracle_state(w)
    run = gpu_runner(w)
    parts = [_split(w, l) for l in range(L)]

    def store_all(chunks):
        k = np.stack([c[0] for c in chunks])
        v = np.stack([c[1] for c in chunks])
        pos = chunks[0][2]
        run.store(0, L, _u16_to_bf16(k).cuda(), _u16_to_bf16(v).cuda(), torch.from_numpy(pos).cuda())
        for l in range(L):
            assert orc.store(l, chunks[l][0], chunks[l][1], chunks[l][2]) == 0

    store_all([parts[l][0] for l in range(L)])
    qs = {l: wl.queries(w, l) for l in range(L)}
    bt = wl.block_table(w)
    lens = w.lens - A
    for t in range(A):
        store_all([parts[l][1][t] for l in range(L)])
        lens = lens + 1
        run.seq_lens.copy_(torch.from_numpy(lens.astype(np.int32)))
        q = np.stack([qs[l][t] for l in range(L)])
        run.step(_u16_to_bf16(q).cuda(), keep_scores=True)
        torch.cuda.synchronize()
        assert int(run.status.item()) == 0, f"status {run.status.item()} at step {t}"
        for l in range(L):
            r = orc.step(l, qs[l][t], bt, lens)
            assert r["drops"] == 0 and r["flags"] == 0 and r["unresolved"] == 0
            assert np.array_equal(run.scores[l].cpu().numpy(), r["scores"]), f"scores {l} {t}"
            assert np.array_equal(run.sel[l].cpu().numpy(), r["sel"]), f"sel {l} {t}"
            assert int(run.n_miss[l].item()) == r["n_miss"], f"n_miss {l} {t}"
            assert np.array_equal(run.phys[l].cpu().numpy(), r["phys"]), f"phys {l} {t}"
            err = float(np.abs(run.out[l].float().cpu().numpy() - r["out"]).max())
            assert err <= TOL[w.fp8], f"max abs err {err} layer {l} step {t}"
            if t % 8 == 7 or t == A - 1:
                compare_slab(run, orc, l)
                compare_mirror(w, run, orc, l)
                compare_state(w, run, orc, l, check_pool=True)
