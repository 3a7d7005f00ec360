"""GPU parity at the full sizes of the synthetic workloads, in the benchmark's
launch configuration: the library runs every layer in one launch per stage;
the oracle (which finishes a layer in seconds) checks sampled layers after
every decode step of the query walk.  Bit-exact selection, remap, miss lists
and LRU state each step; pool bytes at the end; outputs within tolerance.

The throughput sweep (131,072-token requests, 32/4 heads) runs at its full
per-layer sizes for every batch, with one layer so that the oracle's copy of
the host mirror fits the host: 64 and 32 requests over a 20 %-resident pool
(26,215 and 13,108 slots per layer; 2,112 and 1,056 misses in the first step
from the empty pool), and 8 requests fully resident, in bf16 and fp8.
"""
import pytest

import workloads as wl
from tests.parity import run_parity

pytestmark = pytest.mark.gpu


def test_batched_32k_bf16_needles_full():
    w = wl.WORKLOADS["batched_32k_bf16_needles"]
    rep = {}
    run, orc = run_parity(w, oracle_layers=[0, 11], pool_every_step=False, report=rep)
    pages = wl.needle_pages(w)
    for l in (0, 11):
        sel = run.sel[l].cpu().numpy()
        for b in range(w.batch):
            assert set(pages[b].tolist()) <= set(sel[b].tolist())
    print(w.name, rep)


def test_lru_pressure_64k_fp8_full():
    w = wl.WORKLOADS["lru_pressure_64k_fp8"]
    rep = {}
    run_parity(w, oracle_layers=[0, 7], pool_every_step=False, check_mirror=True, report=rep)
    assert rep["misses"] > 0
    print(w.name, rep)


def test_host_tier_196k_fp8_full():
    w = wl.WORKLOADS["host_tier_196k_fp8"]
    rep = {}
    run_parity(w, oracle_layers=[5], pool_every_step=False, report=rep)
    assert rep["misses"] > 0
    print(w.name, rep)


@pytest.mark.parametrize("fp8,frac", [(False, 1.0), (True, 0.2)], ids=["bf16_resident", "fp8_20pct"])
def test_sweep_128k_batch1_full(fp8, frac):
    w = wl.sweep_workload(1, fp8, frac, steps=6)
    rep = {}
    run_parity(w, oracle_layers=[3], pool_every_step=False, report=rep)
    print(w.name, rep)


SWEEP_FULL = [(64, True, 0.2), (64, False, 0.2), (32, True, 0.2), (32, False, 0.2),
              (8, False, 1.0), (8, True, 1.0)]


@pytest.mark.parametrize("batch,fp8,frac", SWEEP_FULL,
                         ids=[f"b{b}_{'fp8' if f else 'bf16'}_{'resident' if r >= 1 else '20pct'}"
                              for b, f, r in SWEEP_FULL])
def test_sweep_128k_full_per_layer_sizes(batch, fp8, frac):
    w = wl.sweep_workload(batch, fp8, frac, steps=3).with_(n_layers=1)
    rep = {}
    run_parity(w, pool_every_step=False, check_mirror=frac < 1.0, report=rep)
    if frac < 1.0:
        assert rep["max_layer_misses"] >= batch * (w.block_topk + 1)   # the cold first step
    print(w.name, rep)


@pytest.mark.parametrize("name", ["lru_pressure_64k_fp8", "host_tier_196k_fp8"])
def test_full_size_misses_fetched_inside_the_attention(name):
    w = wl.WORKLOADS[name]
    if name == "host_tier_196k_fp8":
        w = w.with_(steps=24)
    rep = {}
    run_parity(w, oracle_layers=[0, 5], pool_every_step=False, fetch_in_attention=True,
               report=rep)
    assert rep["misses"] > 0
    print(w.name, rep)
