"""GPU parity of the LRU ensure kernel on every one of its code paths.

The ensure kernel (one CTA per layer) picks its path from the shapes:
  * victim keys kept in shared memory, or read from global memory on every
    radix pass (more than 16,384 slots, or id/victim buffers plus keys above
    the per-CTA shared-memory limit);
  * the victim order by all-pairs ranking (up to 1,024 misses in a layer) or
    by a bitonic sort (more);
  * 256 or 1,024 threads;
  * the distinct selected ids from a bitmap over the logical ids, or, when
    the bitmap would be wider than twice the padded selection (ceil(Lp/32) >
    2 * N2), from a bitonic sort of the ids and an adjacent dedup.
Each case below forces one combination with small heads (Hq = Hkv = 1,
16-token pages) so that memory stays small, runs several steps of a
low-correlation query walk from an empty pool (so the pool fills and then
evicts), and checks every step against the oracle bit for bit: selection,
miss lists, slot_of, page_of, last_use, clock and the remapped table; the
pool bytes after the last step; attention within tolerance.
"""
import pytest

import workloads as wl
from tests.parity import run_parity

SMEM_OPTIN = 227 * 1024


def _n2(w):
    n = 2
    while n < w.batch * (2 * w.block_topk + 8):
        n <<= 1
    return n


def _keys_in_smem(w):
    return w.slots <= 16384 and _n2(w) * 12 + w.slots * 4 + 2048 <= SMEM_OPTIN


def _w(name, **kw):
    base = dict(batch=4, n_layers=1, page_size=16, n_q_heads=1, n_kv_heads=1, head_dim=128,
                fp8=True, steps=4, rho=0.3, walk_c=(1 - 0.09) ** 0.5, seed=300)
    base.update(kw)
    return wl.Workload(name, **base)


CASES = {
    # > 16,384 slots: keys re-read from global memory; 8,004 misses in the
    # first step (bitonic victim sort, 1,024 threads); the pool fills in
    # the third step and evicts from then on
    "global_keys_bitonic_victims": _w("global_keys_bitonic_victims", ctx=16 * 5000,
                                      block_topk=2000, pool_slots=16400, seed=301),
    # 8,832 selection entries pad to N2 = 16,384: ids and victims take 192 KiB,
    # so 9,000 slots of keys no longer fit beside them (global keys although
    # S <= 16,384); 4,404 misses in the first step
    "smem_limit_falls_back_to_global_keys": _w("smem_limit_falls_back_to_global_keys",
                                               ctx=16 * 3000, block_topk=1100, pool_slots=9000,
                                               seed=302),
    # keys in shared memory with more than 1,024 misses (bitonic victim sort)
    "smem_keys_bitonic_victims": _w("smem_keys_bitonic_victims", ctx=16 * 2500, block_topk=600,
                                    pool_slots=5000, seed=303),
    # fully resident (identity pool, hits only) with 16,400 slots: keys from
    # global memory and id/victim buffers of exactly 48 KiB (N2 = 4,096),
    # which with the kernel's static shared memory needs the opt-in limit
    "resident_global_keys_48k_buffers": _w("resident_global_keys_48k_buffers",
                                           ctx=16 * 4100, block_topk=500, pool_slots=None,
                                           steps=2, seed=306),
    # one request, top-4: N2 = 16, and 2,000 logical pages need 63 bitmap
    # words > 2 * N2, so the ids are sorted and deduplicated instead
    "id_sort_dedup": _w("id_sort_dedup", batch=1, ctx=16 * 2000, block_topk=4, pool_slots=40,
                        steps=6, rho=0.8, walk_c=0.6, seed=304),
    # the same path in bf16, two requests sharing nothing, ragged lengths
    "id_sort_dedup_bf16_ragged": _w("id_sort_dedup_bf16_ragged", batch=2, ctx=16 * 1500 + 5,
                                    seq_lens=(16 * 1500 + 5, 16 * 1100 + 9), fp8=False,
                                    block_topk=3, pool_slots=30, steps=6, rho=0.8, walk_c=0.6,
                                    seed=305),
}


def test_cases_reach_the_intended_paths():
    c = CASES["global_keys_bitonic_victims"]
    assert c.slots > 16384 and not _keys_in_smem(c)
    assert c.batch * (c.block_topk + 1) > 1024
    c = CASES["smem_limit_falls_back_to_global_keys"]
    assert c.slots <= 16384 and not _keys_in_smem(c) and _n2(c) == 16384
    c = CASES["smem_keys_bitonic_victims"]
    assert _keys_in_smem(c) and c.batch * (c.block_topk + 1) > 1024
    c = CASES["resident_global_keys_48k_buffers"]
    assert c.slots > 16384 and _n2(c) * 12 == 48 * 1024 and not c.host_tier
    for name in ("id_sort_dedup", "id_sort_dedup_bf16_ragged"):
        c = CASES[name]
        assert (c.logical_pages + 31) // 32 > 2 * _n2(c)


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_ensure_path_parity(name):
    w = CASES[name]
    rep = {}
    run_parity(w, pool_every_step=False, report=rep)
    assert rep["misses"] > 0 or not w.host_tier
    if name in ("global_keys_bitonic_victims", "smem_limit_falls_back_to_global_keys",
                "smem_keys_bitonic_victims"):
        assert rep["max_layer_misses"] > 1024
    print(name, rep)
