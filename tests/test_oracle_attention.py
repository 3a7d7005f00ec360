"""Pins for the oracle's attention over the selected pages.

The reference values come from torch.nn.functional.scaled_dot_product_attention
in float64 on the CPU (a library routine the oracle does not use), on K/V read
back from the oracle's pool and decoded by torch (bf16 bits -> float, or
float8_e4m3fn codes -> float times the per-token scale).  When block_topk
covers every page the method is plain dense GQA attention; with a real
selection it is dense attention over the gathered tokens of the selected pages.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import Workload, block_table, queries, store_batch


def _state(w):
    lay = oracle.OracleLayout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8,
                              w.n_layers, w.logical_pages, w.slots, w.batch,
                              w.pages_per_request, w.block_topk)
    return oracle.OracleKV(lay, host_tier=w.host_tier, identity=not w.host_tier)


def _decode_pool(kv, layer, w):
    """Pool of one layer as float64 torch tensors [S][Hkv][P][D] (torch decodes)."""
    S, H, P, D = w.slots, w.n_kv_heads, w.page_size, w.head_dim
    out = []
    for pool, scale in ((kv.k_pool[layer], kv.k_scale[layer]), (kv.v_pool[layer], kv.v_scale[layer])):
        raw = torch.from_numpy(pool.copy())
        if w.fp8:
            x = raw.view(torch.float8_e4m3fn).to(torch.float64).view(S, H, P, D)
            x = x * torch.from_numpy(scale.astype(np.float64)).view(S, 1, P, 1)
        else:
            x = raw.view(torch.bfloat16).to(torch.float64).view(S, H, P, D)
        out.append(x)
    return out


def _sdpa_over(kv, layer, w, q_bits, sel, phys):
    K, V = _decode_pool(kv, layer, w)
    q = torch.from_numpy(q_bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)
    q = q.to(torch.float64)                                       # [B][Hq][D]
    outs = []
    for b in range(w.batch):
        ks, vs = [], []
        for p, s in zip(sel[b], phys[b]):
            if p < 0:
                continue
            valid = min(w.page_size, int(w.lens[b]) - int(p) * w.page_size)
            ks.append(K[s, :, :valid])
            vs.append(V[s, :, :valid])
        kk = torch.cat(ks, dim=1).repeat_interleave(w.group, dim=0)   # [Hq][T][D]
        vv = torch.cat(vs, dim=1).repeat_interleave(w.group, dim=0)
        o = F.scaled_dot_product_attention(q[b][:, None, :], kk, vv,
                                           scale=1.0 / math.sqrt(w.head_dim))
        outs.append(o[:, 0, :].numpy())
    return np.stack(outs)


CASES = [
    # dense: block_topk covers every page (ragged last page)
    Workload("dense_bf16", batch=2, n_layers=1, ctx=12 * 16 + 7, page_size=16, n_q_heads=8,
             n_kv_heads=2, head_dim=64, fp8=False, block_topk=64, pool_slots=None, seed=21,
             seq_lens=(12 * 16 + 7, 5 * 16)),
    Workload("dense_fp8", batch=2, n_layers=1, ctx=9 * 32 + 3, page_size=32, n_q_heads=4,
             n_kv_heads=1, head_dim=128, fp8=True, block_topk=64, pool_slots=None, seed=22,
             seq_lens=(9 * 32 + 3, 2 * 32 + 1)),
    # sparse: a real top-k over many pages
    Workload("sparse_bf16", batch=2, n_layers=1, ctx=60 * 16 + 9, page_size=16, n_q_heads=8,
             n_kv_heads=1, head_dim=128, fp8=False, block_topk=8, pool_slots=None, seed=23),
    Workload("sparse_fp8", batch=3, n_layers=1, ctx=50 * 64 + 33, page_size=64, n_q_heads=16,
             n_kv_heads=2, head_dim=128, fp8=True, block_topk=5, pool_slots=None, seed=24),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_attention_matches_sdpa_float64(w):
    kv = _state(w)
    k, v, pos = store_batch(w, 0)
    kv.store(0, k, v, pos)
    q = queries(w, 0)[0]
    r = kv.step(0, q, block_table(w), w.lens)
    if w.block_topk >= w.pages_per_request:
        for b in range(w.batch):
            n = -(-int(w.lens[b]) // w.page_size)
            assert r["sel"][b][:n].tolist() == list(range(n))
    ref = _sdpa_over(kv, 0, w, q, r["sel"], r["phys"])
    np.testing.assert_allclose(r["out"], ref, rtol=0, atol=1e-12)


def test_attention_is_invariant_to_slot_placement():
    """Same pages in a permuted pool (host tier, empty start) give the same output."""
    w = CASES[3]
    a = _state(w)
    wb = w.with_(pool_slots=w.batch * (2 * w.block_topk + 8) + 5)
    b = _state(wb)
    k, v, pos = store_batch(w, 0)
    a.store(0, k, v, pos)
    b.store(0, k, v, pos)
    q = queries(w, 0)[0]
    ra = a.step(0, q, block_table(w), w.lens)
    rb = b.step(0, q, block_table(w), w.lens)
    assert np.array_equal(ra["sel"], rb["sel"])
    assert rb["n_miss"] == int((rb["sel"] >= 0).sum())
    assert not np.array_equal(ra["phys"], rb["phys"])
    np.testing.assert_allclose(ra["out"], rb["out"], rtol=0, atol=1e-13)
