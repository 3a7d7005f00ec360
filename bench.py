#!/usr/bin/env python
"""Benchmark: the sparse-attention decode step on one GB300 (or N replicas).

One step = one decode step of every layer of the workload: indexer + top-k,
LRU ensure + miss fetch from the pinned host mirror, remap, sparse paged
attention (+ split merge), all layers of the range in one launch per stage.

Default workload: 4 requests x 12 layers, 65,536 tokens each in 64-token
pages, fp8 e4m3 K/V with per-token scales, 16/2 heads, top-32, a pool of 320
GPU slots per layer over a pinned host mirror, queries on a rho = 0.8 random
walk (frequent misses).  Inputs are seeded synthetic data resident in HBM
before timing; L2 is flushed (256 MiB write) between timed steps.

Timing: per stage a captured CUDA graph, CUDA events between stages on the
launching stream; W warm-up steps, then K timed steps.  `e2e` repeats the
metric through the public API (DecodeRunner.step) with the step's queries
copied from pinned host memory and its output copied back inside the timed
region.  Multi-GPU (torchrun): each rank runs an independent replica (the
path shards by request with no collective): weak scaling, max time over ranks.

--impl reference times the plain CPU oracle on the host cores on a bounded
sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "sparse decode layer-steps/s (x batch)"
UNIT = "layer-steps/s"
DEFAULT_WORKLOAD = "lru_pressure_64k_fp8"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-legs", action="store_true",
                    help="skip the preload, host-tail, shared-residency and store legs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="bound on the timed oracle sample")
    ap.add_argument("--kernel", choices=["index", "attention"], default=None,
                    help="time one kernel alone on the workload's shape (a small pool of "
                         "B*W slots with random contents, so that a profiler capture holds "
                         "little device memory) instead of the step")
    ap.add_argument("--host-warmup", type=int, default=-1,
                    help="most untimed steps that warm the host tier after the prefill, stopped "
                         "once the ensure stage plateaus (-1: 300 with a host tier, 0 without)")
    return ap.parse_args()


def get_workload(name: str) -> wl.Workload:
    if name in wl.WORKLOADS:
        return wl.WORKLOADS[name]
    if name.startswith("sweep_"):
        # sweep_<bf16|fp8>_<resident|20pct>_b<B>
        _, kv, res, b = name.split("_")
        return wl.sweep_workload(int(b[1:]), kv == "fp8", 1.0 if res == "resident" else 0.2)
    raise SystemExit(f"unknown workload {name}")


def replica_workload(w: wl.Workload, rank: int, world: int) -> wl.Workload:
    """The path shards by request with no exchange: each rank runs its own
    replica of the workload (same shape, its own seed) -- weak scaling."""
    return w if world == 1 else w.with_(seed=w.seed + 1000 * rank)


def reduce_max(x: float, dist, device) -> float:
    """Max over ranks (the slowest rank sets the job's time)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# DRAM bytes (read + write) of one decode launch on lru_pressure_64k_fp8, from
# the committed ncu capture of the attention kernel on that workload, valid
# only for the kernel sources it was taken on (their SHA-256 below).
DECODE_TRAFFIC = {"workload": "lru_pressure_64k_fp8", "bytes": 53123328 + 245760,
                  "sources": ("sparse_attention_decode_indexer_gb300/csrc/decode.cu",
                              "sparse_attention_decode_indexer_gb300/csrc/common.cuh"),
                  "sha256": "cb8879fca68c63f44cb1b94d6af4f1739193415d1ae9f92d9b2a67cc0fd12727"}


def decode_traffic(workload_name):
    """The captured traffic per launch, or None when the workload differs or the
    kernel sources changed since the capture."""
    import hashlib
    if workload_name != DECODE_TRAFFIC["workload"]:
        return None
    h = hashlib.sha256()
    for f in DECODE_TRAFFIC["sources"]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return DECODE_TRAFFIC["bytes"] if h.hexdigest() == DECODE_TRAFFIC["sha256"] else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes (what the method must move; the dense KV it skips is not
# counted, nor any re-read or split-K partial)
# ---------------------------------------------------------------------------

def n_selected(w: wl.Workload) -> np.ndarray:
    n_b = np.ceil(w.lens / w.page_size).astype(np.int64)
    return np.minimum(n_b, w.block_topk + 1)


def decode_bytes(w: wl.Workload) -> int:
    """Per launch of the attention over all layers: the selected pages' K and V
    (one KV head each, per KV head), fp8 per-token scales, q, out, sel, phys."""
    esz = 1 if w.fp8 else 2
    ns = n_selected(w)
    kv = int(ns.sum()) * w.n_kv_heads * 2 * w.page_size * w.head_dim * esz
    sc = int(ns.sum()) * w.page_size * 8 if w.fp8 else 0
    qo = 2 * w.batch * w.n_q_heads * w.head_dim * 2
    lists = 2 * w.batch * (2 * w.block_topk + 8) * 4
    return w.n_layers * (kv + sc + qo + lists)


def index_bytes(w: wl.Workload) -> int:
    """The slab scan: int8 page keys of every page of every request, plus the
    block-table ids and q."""
    n_b = np.ceil(w.lens / w.page_size).astype(np.int64)
    per_layer = int(n_b.sum()) * (w.n_kv_heads * w.head_dim + 4) + \
        w.batch * w.n_q_heads * w.head_dim * 2
    return w.n_layers * per_layer


def page_fetch_bytes(w: wl.Workload) -> int:
    esz = 1 if w.fp8 else 2
    b = 2 * w.n_kv_heads * w.page_size * w.head_dim * esz
    return b + (2 * w.page_size * 4 if w.fp8 else 0)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# the CPU oracle on a bounded sample (reported baseline; also --impl reference)
# ---------------------------------------------------------------------------

def _oracle_state(w: wl.Workload):
    """The oracle's state for layer 0 of the workload after its prefill."""
    import oracle
    lay = oracle.OracleLayout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8,
                              1, w.logical_pages, w.slots, w.batch, w.pages_per_request,
                              w.block_topk)
    orc = oracle.OracleKV(lay, host_tier=w.host_tier, identity=not w.host_tier)
    k, v, pos = wl.store_batch(w.with_(n_layers=1), 0)
    orc.store(0, k, v, pos)
    return orc


def _oracle_leg(w: wl.Workload, orc, seconds: float, threads: int, t_start: int):
    """Decode steps of layer 0 (every request) through the oracle with the
    given thread count, for about `seconds`; per-stage and total rates."""
    import oracle
    oracle.set_threads(threads)
    one = w.with_(n_layers=1)
    qs = wl.queries(one.with_(steps=max(w.steps, 64)) if w.rho is not None else one, 0)
    bt = wl.block_table(w)
    stage_s = {"index_topk": 0.0, "ensure": 0.0, "remap": 0.0, "decode": 0.0}
    steps = 0
    t0 = time.perf_counter()
    while True:
        q = qs[(t_start + steps) % len(qs)]
        ta = time.perf_counter()
        sel, _, _, _, _ = orc.index_topk(0, q, bt, w.lens)
        tb = time.perf_counter()
        orc.ensure(0, sel, bt)
        tc = time.perf_counter()
        phys, _ = orc.remap(0, sel, bt)
        td = time.perf_counter()
        orc.decode(0, q, sel, phys, w.lens)
        te = time.perf_counter()
        for name, dt in (("index_topk", tb - ta), ("ensure", tc - tb), ("remap", td - tc),
                         ("decode", te - td)):
            stage_s[name] += dt
        steps += 1
        if te - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    used = oracle.threads()
    oracle.set_threads(0)
    return {"value": steps * w.batch / dt, "steps": steps, "seconds": dt, "threads": used,
            "stage_ms_per_step": {k: 1e3 * v / steps for k, v in stage_s.items()}}


def cpu_oracle_sample(w: wl.Workload, seconds: float):
    """The oracle as it stands, on the host cores, on a bounded sample (layer 0
    of the workload, every request; the prefill is not timed): once on one
    thread, once with its independent loops spread over every core (the
    headline figure).  Per-stage times for both."""
    import oracle
    oracle.build()
    orc = _oracle_state(w)
    single = _oracle_leg(w, orc, seconds / 2, 1, 0)
    multi = _oracle_leg(w, orc, seconds / 2, 0, single["steps"])
    return {"value": multi["value"], "unit": UNIT, "cores": multi["threads"], "kind": "oracle",
            "sample": f"layer 0 of {w.name}, all {w.batch} requests, {multi['steps']} decode "
                      f"steps (index, select, ensure+copy, remap, fp64 attention) on "
                      f"{multi['threads']} threads in {multi['seconds']:.1f} s; prefill not timed",
            "stage_ms_per_step": multi["stage_ms_per_step"],
            "single_thread": {"value": single["value"], "unit": UNIT, "cores": 1,
                              "steps": single["steps"],
                              "stage_ms_per_step": single["stage_ms_per_step"]}}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def build_runner(w: wl.Workload, rank: int, prefill_now: bool = True):
    import torch
    from sparse_attention_decode_indexer_gb300 import Layout
    from sparse_attention_decode_indexer_gb300.runner import DecodeRunner
    lay = Layout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8, w.n_layers,
                 w.logical_pages, w.slots, w.batch, w.pages_per_request, w.block_topk)
    run = DecodeRunner(lay, host_tier=w.host_tier, identity=not w.host_tier,
                       block_table=wl.block_table(w), seq_lens=w.lens)
    if prefill_now:
        prefill(w, run)
    return run


def draws_on_device(w: wl.Workload) -> bool:
    """Inputs drawn on the device (torch's Philox generator) where drawing them
    on the host would take minutes and tens of GB of host memory: more than
    4 GiB of bf16 K+V per layer (the 32- and 64-request sweeps).  Same
    distributions (N(0, 1) K, V; the same query walk), other random numbers."""
    return int(w.lens.sum()) * w.n_kv_heads * w.head_dim * 4 > (4 << 30)


def prefill(w: wl.Workload, run):
    """Store every layer's K/V of the workload through ssa_store_kv_mirror."""
    import torch
    if draws_on_device(w):
        assert w.needles == 0
        bt = torch.from_numpy(wl.block_table(w)).cuda()
        P, HD = w.page_size, (w.n_kv_heads, w.head_dim)
        per_req = int(w.lens.max())
        chunk = max(1, (1 << 30) // (per_req * w.n_kv_heads * w.head_dim * 4))
        for l in range(w.n_layers):
            g = torch.Generator(device="cuda")
            g.manual_seed(w.seed * 1000003 + l)
            for b0 in range(0, w.batch, chunk):
                bs = range(b0, min(w.batch, b0 + chunk))
                pos = torch.cat([bt[b][torch.arange(int(w.lens[b]), device="cuda") // P] * P +
                                 torch.arange(int(w.lens[b]), device="cuda") % P
                                 for b in bs]).to(torch.int64)
                T = int(pos.numel())
                kd = torch.randn((1, T) + HD, generator=g, device="cuda").to(torch.bfloat16)
                vd = torch.randn((1, T) + HD, generator=g, device="cuda").to(torch.bfloat16)
                run.store(l, 1, kd, vd, pos)
                del kd, vd, pos
    else:
        for l in range(w.n_layers):
            k, v, pos = wl.store_batch(w, l)
            kd = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).cuda()[None]
            vd = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).cuda()[None]
            run.store(l, 1, kd, vd, torch.from_numpy(pos).cuda())
            del kd, vd
    torch.cuda.synchronize()
    st = int(run.status.item())
    if st != 0:
        raise RuntimeError(f"store status {st}")


def queries_all(w: wl.Workload, n_steps: int):
    """[n_steps][L][B][Hq][D] bf16 queries of the walk, on the device."""
    import torch
    if draws_on_device(w):
        shape = (w.batch, w.n_q_heads, w.head_dim)
        out = torch.empty((n_steps, w.n_layers) + shape, dtype=torch.bfloat16, device="cuda")
        for l in range(w.n_layers):
            g = torch.Generator(device="cuda")
            g.manual_seed(w.seed * 1000003 + 500 + l)
            q = torch.randn(shape, generator=g, device="cuda")
            out[0, l] = q.to(torch.bfloat16)
            for t in range(1, n_steps):
                q = w.rho * q + w.walk_c * torch.randn(shape, generator=g, device="cuda")
                out[t, l] = q.to(torch.bfloat16)
        return out
    ww = w.with_(steps=n_steps)
    q_np = np.stack([wl.queries(ww, l) for l in range(w.n_layers)], axis=1)
    return torch.from_numpy(q_np.view(np.int16)).view(torch.bfloat16).cuda()


def host_link_rates(torch, ssa, page_chunk: int, scatter_chunks: int) -> dict:
    """SM-driven reads of pinned host memory (ssa_host_read_probe), beside the
    copy engine: a sequential stream of 64 KiB chunks over 1 GiB, and a
    scatter of `scatter_chunks` page-sized chunks at random offsets (fresh
    offsets each repetition), the access pattern of one step's miss fetch."""
    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    src.fill_(1)
    dst = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = {}

    def timed(offsets, chunk, lpt):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        ssa.ssa_host_read_probe(src, dst, offsets, chunk, lpt)
        e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e-3

    seq = torch.arange(0, n, 65536, dtype=torch.int64, device="cuda")
    for lpt in (8, 16):
        timed(seq, 65536, lpt)
        best = min(timed(seq, 65536, lpt) for _ in range(4))
        out[f"sm_read_seq_gbs_lpt{lpt}"] = n / best / 1e9
    rng = np.random.default_rng(11)
    n_pages = n // page_chunk
    # every chunk lies inside the 1 GiB source, and the copies fit the 1 GiB dst
    for cnt in sorted({max(1, min(scatter_chunks, n_pages, 65535)), min(4096, n_pages)}):
        ts = []
        for _ in range(5):
            offs = rng.choice(n_pages, size=cnt, replace=False).astype(np.int64) * page_chunk
            ts.append(timed(torch.from_numpy(offs).cuda(), page_chunk, 8))
        out[f"sm_read_scatter_{cnt}x{page_chunk}B_gbs"] = cnt * page_chunk / statistics.median(ts) / 1e9
    del src, dst
    return out


def h2d_peak_gbs(torch) -> float:
    n = 256 << 20
    src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(n, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(6):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        e1.synchronize()
        best = max(best, n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    return best


def run_ours(args, rank: int, world: int, dist):
    import torch
    import sparse_attention_decode_indexer_gb300 as ssa

    w = replica_workload(get_workload(args.workload), rank, world)
    W, K = args.warmup, args.steps
    H_max = args.host_warmup if args.host_warmup >= 0 else (300 if w.host_tier else 0)
    run = build_runner(w, rank, prefill_now=False)   # graphs first, then one prefill
    n_total = H_max + W + 4 * K + (10 * K + 140 + len(OVERLAP_GROUPS) * (K + 12) + 20
                                   if w.host_tier else 0)
    q_all = queries_all(w, n_total)
    q_cur = q_all[0].clone()
    flush_w = torch.empty(64 << 20, dtype=torch.float32, device="cuda")  # 256 MiB > L2
    flush_r = torch.zeros(64 << 20, dtype=torch.float32, device="cuda")

    def flush_l2():
        # write 256 MiB (evicts the step's data), then read another 256 MiB so
        # the lines left in L2 are clean: the timed kernels do not pay for
        # writing back the flush itself
        flush_w.zero_()
        flush_r.sum()

    L = w.n_layers
    c = run.cache

    def st_index():
        ssa.ssa_index_topk(c, 0, L, q_cur, run.block_table, run.seq_lens, run.sel, run.n_sel,
                           None, run.status, run.ws)

    def st_ensure():
        # ensure (LRU state + miss copy) with the remap fused into the LRU kernel
        ssa.ssa_ensure_remap(c, 0, L, run.sel, run.block_table, run.phys, run.miss_page,
                             run.miss_slot, run.n_miss, run.status, run.ws)

    def st_decode():
        ssa.ssa_sparse_paged_decode(c, 0, L, q_cur, run.sel, run.phys, run.seq_lens,
                                    run.sm_scale, run.out, run.status, run.ws)

    stages = [("index_topk", st_index), ("ensure_remap", st_ensure), ("decode", st_decode)]
    # one eager step (function attributes, lazy init), then capture the step:
    # one graph with timing events between its stages (events recorded from
    # inside the graph), or, where this torch cannot record events in a
    # graph, one graph per stage with events between the replays
    for _, f in stages:
        f()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    launches_per_step = 0
    try:
        # the timed step: events only at its two ends, so the stages keep
        # their programmatic (PDL) edges; the stage breakdown comes from a
        # second graph with events between the stages
        pev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
        g_plain = torch.cuda.CUDAGraph()
        n0 = ssa.launch_count()
        with torch.cuda.graph(g_plain, stream=s):
            pev[0].record()
            for _, f in stages:
                f()
            pev[1].record()
        launches_per_step = ssa.launch_count() - n0
        sev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(stages) + 1)]
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step, stream=s):
            sev[0].record()
            for i, (_, f) in enumerate(stages):
                f()
                sev[i + 1].record()
        graphs = None
        timing_mode = ("one CUDA graph per step, events at its ends; stage times from a second "
                       "graph with events between the stages")
    except Exception:
        g_plain = None
        torch.cuda.synchronize()
        g_step = None
        graphs = []
        for name, f in stages:
            g = torch.cuda.CUDAGraph()
            n0 = ssa.launch_count()
            with torch.cuda.graph(g, stream=s):
                f()
            launches_per_step += ssa.launch_count() - n0
            graphs.append(g)
        timing_mode = "one CUDA graph per stage, CUDA events between the replays"
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()

    def replay_plain():
        """One decode step; returns its time (ms)."""
        if g_plain is not None:
            g_plain.replay()
            pev[1].synchronize()
            return pev[0].elapsed_time(pev[1])
        return sum(replay_step(ev))

    def replay_step(timed_events=None):
        """One decode step; returns per-stage times (ms) when timed_events."""
        if g_step is not None:
            g_step.replay()
            if timed_events is None:
                return None
            sev[-1].synchronize()
            return [sev[i].elapsed_time(sev[i + 1]) for i in range(len(stages))]
        if timed_events is None:
            for g in graphs:
                g.replay()
            return None
        timed_events[0].record()
        for i, g in enumerate(graphs):
            g.replay()
            timed_events[i + 1].record()
        timed_events[-1].synchronize()
        return [timed_events[i].elapsed_time(timed_events[i + 1]) for i in range(len(stages))]

    # the eager step ran on the empty cache: reset the state, then prefill once
    ssa.ssa_lru_init(c, identity=not w.host_tier)
    prefill(w, run)
    miss_acc = torch.zeros(L, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()

    # host tier: the miss fetch over the host link runs far slower in the
    # first steps after a prefill and keeps speeding up for tens of steps;
    # untimed steps of the same query walk until it settles -- at least 100,
    # then until the median ensure time of the last 20 steps is within 3 % of
    # the 20 before (at most H_max) -- the count recorded in the config
    H = 0
    ens_us = []
    warm_ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
    while H < H_max:
        flush_l2()                         # the same conditions as the timed steps
        q_cur.copy_(q_all[H])
        ens_us.append(replay_step(warm_ev)[1] * 1e3)   # the ensure_remap stage
        H += 1
        if H >= 100:
            last, prev = statistics.median(ens_us[-20:]), statistics.median(ens_us[-40:-20])
            if last >= 0.97 * prev:
                break
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms, stage_rows = [], []
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
    for t in range(W + K):
        flush_l2()
        q_cur.copy_(q_all[H + t])
        ms = replay_plain()
        if t >= W:
            step_ms.append(ms)
            miss_acc += run.n_miss
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    st = int(run.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st}: {ssa.status_str(st)}")
    # the stage breakdown: the same step with events between its stages
    stage_miss = torch.zeros(L, dtype=torch.int64, device="cuda")
    for t in range(K):
        flush_l2()
        q_cur.copy_(q_all[H + W + K + t])
        stage_rows.append(replay_step(ev))
        stage_miss += run.n_miss
    torch.cuda.synchronize()
    stage_ms = {name: [r[i] for r in stage_rows] for i, (name, _) in enumerate(stages)}
    total_s = reduce_max(sum(step_ms) * 1e-3, dist, "cuda")
    units = L * w.batch * K * world
    value = units / total_s
    misses = int(miss_acc.sum().item())

    # per-layer launches (4 calls per layer, layer after layer), one graph per step
    g_pl = torch.cuda.CUDAGraph()
    run.step(q_cur, per_layer=True)
    torch.cuda.synchronize()
    with torch.cuda.graph(g_pl, stream=s):
        run.step(q_cur, per_layer=True)
    torch.cuda.synchronize()
    pl_ms = []
    for t in range(K):
        flush_l2()
        q_cur.copy_(q_all[H + W + 2 * K + t])
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g_pl.replay()
        e1.record()
        torch.cuda.synchronize()
        pl_ms.append(e0.elapsed_time(e1))

    # end to end through the public API, host buffers in and out
    e2e = None
    if not args.no_e2e:
        q_host = q_all[H + W + 3 * K:H + W + 4 * K].cpu().pin_memory()
        out_host = torch.empty((K,) + tuple(run.out.shape), dtype=torch.bfloat16,
                               pin_memory=True)
        q_dev = torch.empty_like(q_cur)
        # the step as a serving loop runs it: one query buffer, the step's
        # launches captured once (on this untimed first call) and replayed
        run.graphs = True
        q_dev.copy_(q_host[0])
        run.step(q_dev)
        torch.cuda.synchronize()
        e2e_ms = []
        for t in range(K):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            q_dev.copy_(q_host[t], non_blocking=True)
            out = run.step(q_dev)
            out_host[t].copy_(out, non_blocking=True)
            e1.record()
            e1.synchronize()
            e2e_ms.append(e0.elapsed_time(e1))
        run.graphs = False                 # the legs below run eager steps on many q buffers
        tot = reduce_max(sum(e2e_ms) * 1e-3, dist, "cuda")
        e2e = {"value": units / tot, "unit": UNIT,
               "h2d_bytes_per_step": int(q_host[0].numel() * 2),
               "d2h_bytes_per_step": int(out_host[0].numel() * 2),
               "ms_per_step": 1e3 * tot / K,
               "path": "DecodeRunner.step (the step's C-ABI calls as one CUDA graph replay, captured "
                       "on an untimed first call) + pinned H2D q / D2H out"}

    preload = host_tail = fetch = overlap = None
    if w.host_tier:
        fetch = time_fetch_in_attention(w, run, q_all, q_cur, H + W + 12 * K + 100, K, flush_l2)
    if w.host_tier and not args.no_legs:
        overlap = time_overlap(w, run, q_all, q_cur, H + W + 14 * K + 130, K, flush_l2)
        preload = time_preload(w, run, q_all, H + W + 4 * K, K, flush_l2)
        host_tail = time_host_tail(w, run, q_all, H + W + 8 * K + 8, K, flush_l2)
    if rank != 0:
        return None
    shared = (time_shared(w, run, q_all, H + W + 10 * K + 16, K, flush_l2)
              if w.host_tier and not args.no_legs else None)
    store = time_store(w, run) if not args.no_legs else None
    peak, peak_kind = load_peaks()
    dec_ms = statistics.mean(stage_ms["decode"])
    dec_bytes = decode_bytes(w)
    achieved = dec_bytes / (dec_ms * 1e-3) / 1e9
    idx_ms = statistics.mean(stage_ms["index_topk"])
    ens_ms = statistics.mean(stage_ms["ensure_remap"])
    miss_bytes = misses * page_fetch_bytes(w) / K
    stage_miss_bytes = int(stage_miss.sum().item()) * page_fetch_bytes(w) / K
    h2d = h2d_peak_gbs(torch)
    esz = 1 if w.fp8 else 2
    head_page = w.n_kv_heads * w.page_size * w.head_dim * esz     # one tensor of one page
    link = host_link_rates(torch, ssa, head_page, max(1, int(round(2 * misses / K))))
    uva_peak = max(v for k, v in link.items() if k.startswith("sm_read_seq"))
    miss_gbs = stage_miss_bytes / (ens_ms * 1e-3) / 1e9
    # pages the step selects (every layer and request): those already bound
    # are the ones the pool kept from earlier steps, fetched by no one now
    sel_per_step = w.n_layers * int(n_selected(w).sum())
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": 1e3 * total_s / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 K/V codes (QK e4m3, PV f16 tensor-core MMAs), f32 accumulate; int8 indexer"
                 if w.fp8 else "bf16 tensor-core MMA, f32 accumulate; int8 indexer",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "layers": w.n_layers, "ctx": w.ctx,
                   "page_size": w.page_size, "heads": f"{w.n_q_heads}/{w.n_kv_heads}",
                   "head_dim": w.head_dim, "kv": "fp8_e4m3" if w.fp8 else "bf16",
                   "block_topk": w.block_topk, "pool_slots": w.slots,
                   "host_tier": w.host_tier, "layers_per_launch": w.n_layers,
                   "l2": "flushed between timed steps (256 MiB write + 256 MiB read)",
                   "inputs": ("K/V and queries drawn on the device (torch Philox), N(0,1) "
                              "rounded to bf16" if draws_on_device(w) else
                              "K/V and queries from the seeded numpy generators (workloads)"),
                   "host_warmup_steps": H,
                   "timing": timing_mode},
        "roofline": {"kernel": "ssa_sparse_paged_decode (decode_kernel: attention and split merge)",
                     "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"hbm_gbs of {peak_kind}",
                     "traffic": decode_traffic(w.name), "alg_bytes_per_launch": dec_bytes,
                     "avg_launch_us": 1e3 * dec_ms},
        "stages_us": {k: 1e3 * statistics.mean(v) for k, v in stage_ms.items()},
        "index_roofline": {"alg_bytes": index_bytes(w),
                           "achieved_gbs": index_bytes(w) / (idx_ms * 1e-3) / 1e9},
        "miss": {"pages_per_step": misses / K, "bytes_per_step": miss_bytes,
                 "selected_pages_per_step": sel_per_step,
                 "resident_fraction": 1.0 - (misses / K) / sel_per_step,
                 "gbs_over_ensure_stage": stage_miss_bytes / (ens_ms * 1e-3) / 1e9,
                 "h2d_copy_engine_peak_gbs": h2d,
                 "frac_of_h2d_peak": miss_gbs / h2d if h2d else None,
                 "sm_read_peak_gbs": uva_peak,
                 "frac_of_sm_read_peak": miss_gbs / uva_peak if uva_peak else None,
                 "host_link": link,
                 "note": "the ensure_remap stage is the LRU state kernel (remap fused) plus the copy kernel",
                 "warmup_ensure_us": ({"first": ens_us[0], "step_10": ens_us[min(9, len(ens_us) - 1)],
                                       "last_20_median": statistics.median(ens_us[-20:])}
                                      if ens_us else None)},
        "per_layer_sequential": {"value": L * w.batch * K / (sum(pl_ms) * 1e-3),
                                 "ms_per_step": statistics.mean(pl_ms),
                                 "note": "4 calls per layer, layer after layer, one graph"},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if store is not None:
        line["store"] = store
    if fetch is not None:
        line["fetch_in_attention"] = fetch
    if overlap is not None:
        line["copy_attention_overlap"] = overlap
    if preload is not None:
        line["preload"] = preload
    if host_tail is not None:
        line["host_tail"] = host_tail
    if shared is not None:
        line["shared_residency"] = shared
    return line, w


def time_preload(w: wl.Workload, run, q_all, t0: int, K: int, flush_l2):
    """The top-k preload against plain steps, both through DecodeRunner.step
    (eager launches, the preload on a second stream).  Two timings per
    variant: (a) one step per timed region, L2 flushed before it, the region
    closed only once the step's preload is done too, so the preload overlaps
    the step's attention and nothing else; (b) K steps back to back in one
    region, where the preload also overlaps the next step's indexer."""
    import torch
    width = 2 * w.block_topk + 8          # the widest preload the buffers take
    main = torch.cuda.current_stream()
    out = {"width": width}
    t = t0
    for name, wdt in (("plain", 0), ("preload", width)):
        run.enable_preload(wdt)
        for _ in range(3):                 # warm the variant
            run.step(q_all[t]); t += 1
        torch.cuda.synchronize()
        ms, miss, fetched = [], 0, 0
        for _ in range(K):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run.step(q_all[t]); t += 1
            if wdt:
                main.wait_stream(run.side)
            e1.record()
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
            miss += int(run.n_miss.sum().item())
            fetched += int(run.n_fetch.sum().item()) if wdt else 0
        flush_l2()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            run.step(q_all[t]); t += 1
        if wdt:
            main.wait_stream(run.side)
        e1.record()
        torch.cuda.synchronize()
        out[name] = {"ms_per_step": statistics.mean(ms),
                     "value": w.n_layers * w.batch / (statistics.mean(ms) * 1e-3),
                     "back_to_back_ms_per_step": e0.elapsed_time(e1) / K,
                     "sync_misses_per_step": miss / K,
                     "preloaded_pages_per_step": fetched / K}
    run.enable_preload(0)
    p, b = out["preload"], out["plain"]
    out["sync_miss_fraction_hidden"] = (1.0 - p["sync_misses_per_step"] / b["sync_misses_per_step"]
                                        if b["sync_misses_per_step"] else None)
    out["step_time_ratio"] = p["ms_per_step"] / b["ms_per_step"]
    out["back_to_back_ratio"] = p["back_to_back_ms_per_step"] / b["back_to_back_ms_per_step"]
    out["note"] = ("eager DecodeRunner.step with and without ssa_prefetch_pages on a second "
                   "stream; (a) per-step regions after an L2 flush, closed after the preload; "
                   "(b) K steps back to back")
    return out


OVERLAP_GROUPS = (2, 4)


def time_overlap(w: wl.Workload, run, q_all, q_cur, t0: int, K: int, flush_l2):
    """The overlapped step (DecodeRunner overlap_groups = G: the LRU update
    for all layers, then the host-link copy per range of layers with each
    range's attention on a second stream behind it) for several G, timed as
    the headline step: one CUDA graph per step with events at its ends, L2
    flushed before each replay."""
    import torch
    t = t0
    s = torch.cuda.Stream()
    res = {}
    for G in OVERLAP_GROUPS:
        if G > w.n_layers:
            continue
        run.overlap_groups = G
        q_cur.copy_(q_all[t]); t += 1
        run.step(q_cur)                            # eager once, then captured
        torch.cuda.synchronize()
        s.wait_stream(torch.cuda.current_stream())
        pev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pev[0].record()
            run.step(q_cur)
            pev[1].record()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for _ in range(10):
            flush_l2()
            q_cur.copy_(q_all[t]); t += 1
            g.replay()
        torch.cuda.synchronize()
        ms, miss = [], 0
        for _ in range(K):
            flush_l2()
            q_cur.copy_(q_all[t]); t += 1
            g.replay()
            pev[1].synchronize()
            ms.append(pev[0].elapsed_time(pev[1]))
            miss += int(run.n_miss.sum().item())
        st = int(run.status.item())
        if st != 0:
            raise RuntimeError(f"device status {st} in the overlap leg (G={G})")
        step_ms = statistics.mean(ms)
        res[str(G)] = {"ms_per_step": step_ms, "value": w.n_layers * w.batch / (step_ms * 1e-3),
                       "layer_groups": [n for _, n in run.layer_groups()],
                       "misses_per_step": miss / K}
    run.overlap_groups = 0
    best = min(res, key=lambda k: res[k]["ms_per_step"])
    return {"groups": res, "best": int(best),
            "note": "ssa_ensure_remap_bind (all layers), then per layer range ssa_fetch_misses "
                    "with that range's attention on a second stream behind it; graph per step, "
                    "L2 flushed before each"}


def time_fetch_in_attention(w: wl.Workload, run, q_all, q_cur, t0: int, K: int, flush_l2):
    """The miss fetch folded into the attention (ssa_ensure_remap_deferred +
    ssa_sparse_paged_decode_fetch) against the headline step's copy-then-
    attend, timed the same way: one CUDA graph per step with events at its
    ends, L2 flushed before each replay; stage times from a second graph
    with events between the stages."""
    import torch
    import sparse_attention_decode_indexer_gb300 as ssa
    L, c = w.n_layers, run.cache

    def st_index():
        ssa.ssa_index_topk(c, 0, L, q_cur, run.block_table, run.seq_lens, run.sel, run.n_sel,
                           None, run.status, run.ws)

    def st_state():
        ssa.ssa_ensure_remap_deferred(c, 0, L, run.sel, run.block_table, run.phys,
                                      run.miss_page, run.miss_slot, run.n_miss, run.status,
                                      run.ws)

    def st_attend():
        ssa.ssa_sparse_paged_decode_fetch(c, 0, L, q_cur, run.sel, run.phys, run.block_table,
                                          run.seq_lens, run.sm_scale, run.out, run.status,
                                          run.ws)

    stages = [("index_topk", st_index), ("ensure_state", st_state), ("decode_fetch", st_attend)]
    for _, f in stages:
        f()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    pev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
    g_plain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_plain, stream=s):
        pev[0].record()
        for _, f in stages:
            f()
        pev[1].record()
    sev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(stages) + 1)]
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=s):
        sev[0].record()
        for i, (_, f) in enumerate(stages):
            f()
            sev[i + 1].record()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    t = t0
    for _ in range(20):                        # the host link settles as for the headline
        flush_l2()
        q_cur.copy_(q_all[t]); t += 1
        g_plain.replay()
    torch.cuda.synchronize()
    ms, miss = [], 0
    for _ in range(K):
        flush_l2()
        q_cur.copy_(q_all[t]); t += 1
        g_plain.replay()
        pev[1].synchronize()
        ms.append(pev[0].elapsed_time(pev[1]))
        miss += int(run.n_miss.sum().item())
    rows = []
    for _ in range(K):
        flush_l2()
        q_cur.copy_(q_all[t]); t += 1
        g_step.replay()
        sev[-1].synchronize()
        rows.append([sev[i].elapsed_time(sev[i + 1]) for i in range(len(stages))])
    st = int(run.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st} in the fetch-in-attention leg")
    step_ms = statistics.mean(ms)
    return {"ms_per_step": step_ms, "value": L * w.batch / (step_ms * 1e-3),
            "stages_us": {name: 1e3 * statistics.mean(r[i] for r in rows)
                          for i, (name, _) in enumerate(stages)},
            "misses_per_step": miss / K,
            "note": "index -> ensure state + remap (misses marked) -> attention that reads the "
                    "marked pages from the host mirror and writes them into their slots; "
                    "graph per step, L2 flushed before each"}


def time_host_tail(w: wl.Workload, run, q_all, t0: int, K: int, flush_l2):
    """Zero-copy host-tail attention against ensure-then-attend, both eager,
    one step per timed region after an L2 flush.  The zero-copy step is the
    indexer plus ssa_sparse_paged_decode_host_tail: pages without a slot are
    read from the host mirror inside the attention, the pool stays as the LRU
    left it (a frozen HBM head).  Host pages per step are counted from sel and
    slot_of after each step."""
    import torch
    import sparse_attention_decode_indexer_gb300 as ssa
    L, c = w.n_layers, run.cache
    t = t0

    def zero_copy(q):
        ssa.ssa_index_topk(c, 0, L, q, run.block_table, run.seq_lens, run.sel, run.n_sel, None,
                           run.status, run.ws)
        ssa.ssa_sparse_paged_decode_host_tail(c, 0, L, q, run.sel, run.block_table,
                                              run.seq_lens, run.sm_scale, run.out, run.status,
                                              run.ws)

    out = {}
    for name, fn in (("ensure_then_attend", lambda q: run.step(q)), ("zero_copy", zero_copy)):
        for _ in range(3):
            fn(q_all[t]); t += 1
        torch.cuda.synchronize()
        ms, host = [], 0
        for _ in range(K):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn(q_all[t]); t += 1
            e1.record()
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
            sel = run.sel.long()
            bt = run.block_table.long()
            ids = torch.gather(bt.unsqueeze(0).expand(L, -1, -1), 2, sel.clamp(min=0))
            slot = torch.gather(c.slot_of.long(), 1, ids.reshape(L, -1)).reshape(ids.shape)
            host += int(((sel >= 0) & (slot < 0)).sum().item())
        out[name] = {"ms_per_step": statistics.mean(ms),
                     "value": L * w.batch / (statistics.mean(ms) * 1e-3),
                     "host_pages_per_step": host / K}
    # a host page is one (layer, request) page: K and V of every KV head (+ scales)
    out["zero_copy"]["host_bytes_per_step"] = (out["zero_copy"]["host_pages_per_step"] *
                                               page_fetch_bytes(w))
    out["ratio"] = out["zero_copy"]["ms_per_step"] / out["ensure_then_attend"]["ms_per_step"]
    out["note"] = ("eager steps, L2 flushed before each; zero_copy = indexer + host-tail "
                   "attention over the pool as the LRU left it (not updated), "
                   "ensure_then_attend = DecodeRunner.step")
    st = int(run.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st} in the host-tail leg")
    return out


def time_shared(w: wl.Workload, run, q_all, t0: int, K: int, flush_l2, warm: int = 40):
    """Residency shared by all layers (ssa_ensure_remap_shared: one LRU, each
    miss copied for every layer) against per-layer residency, both eager
    DecodeRunner steps with an L2 flush before each.  The residency state is
    emptied first and each mode warmed for `warm` steps (the first fetches
    after an empty pool run far slower over the host link).  Run last: it
    leaves the cache in shared mode."""
    import torch
    L, B, W, S = w.n_layers, w.batch, 2 * w.block_topk + 8, w.slots
    if L * B * W > 16384 or S < min(L * B * W, w.logical_pages):
        return {"not_applicable": f"pool of {S} slots < {L} layers x {B * W} selection "
                                  f"entries (the union the shared state must hold)"}
    c = run.cache
    out = {}
    t = t0
    for name, shared in (("per_layer", False), ("shared", True)):
        torch.cuda.synchronize()
        for a, v in ((c.slot_of, -1), (c.page_of, -1), (c.last_use, -1), (c.clock, 0)):
            a.fill_(v)                             # an empty pool for each mode
        run.shared_residency = shared
        for _ in range(warm):
            flush_l2()
            run.step(q_all[t]); t += 1
        torch.cuda.synchronize()
        ms, miss = [], 0
        for _ in range(K):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run.step(q_all[t]); t += 1
            e1.record()
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
            miss += int(run.n_miss[0].item()) if shared else int(run.n_miss.sum().item())
        per_miss = page_fetch_bytes(w) * (L if shared else 1)
        out[name] = {"ms_per_step": statistics.mean(ms),
                     "value": L * B / (statistics.mean(ms) * 1e-3),
                     "misses_per_step": miss / K,
                     "miss_bytes_per_step": miss / K * per_miss}
    out["ratio"] = out["shared"]["ms_per_step"] / out["per_layer"]["ms_per_step"]
    out["note"] = ("eager DecodeRunner.step after an emptied pool and %d warm steps per mode; "
                   "a shared miss copies the page for every layer" % warm)
    st = int(run.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st} in the shared-residency leg")
    return out


def time_store(w: wl.Workload, run, chunk: int = 4096, n_append: int = 50):
    """The store path on the filled cache, after every decode measurement:
    the per-step append (one token per request, every layer in one call) and
    a prefill chunk of `chunk` tokens per request (every layer in one call).
    Positions already stored are stored again: the kernels do the same work
    as on first store (the slab sums it leaves are not used afterwards)."""
    import torch
    L, B, P = w.n_layers, w.batch, w.page_size
    bt = wl.block_table(w)
    lens = w.lens.astype(np.int64)
    g = torch.Generator(device="cuda").manual_seed(5)

    def positions(tok):                     # tok[b]: token indices of request b
        return torch.from_numpy(np.concatenate(
            [bt[b][t // P].astype(np.int64) * P + t % P for b, t in enumerate(tok)])).cuda()

    def kv(T):
        shape = (L, T, w.n_kv_heads, w.head_dim)
        return (torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16),
                torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16))

    def timed(k, v, pos, per_graph, reps):
        """ms per call: `per_graph` calls captured in one CUDA graph (as a
        serving loop captures its step), replayed between events"""
        run.store(0, L, k, v, pos)          # warm
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            for _ in range(per_graph):
                run.store(0, L, k, v, pos)
        torch.cuda.current_stream().wait_stream(s)
        g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) / per_graph)
        return statistics.median(ts)

    mirror_per_tok = w.n_kv_heads * w.head_dim * 2 * (1 if w.fp8 else 2) + (8 if w.fp8 else 0)
    k, v = kv(B)
    app_ms = timed(k, v, positions([np.array([n - 1]) for n in lens]), 8, n_append)
    n_chunk = [np.arange(min(chunk, int(n))) for n in lens]
    T = sum(len(t) for t in n_chunk)
    k, v = kv(T)
    pre_ms = timed(k, v, positions(n_chunk), 1, 5)
    torch.cuda.synchronize()
    return {
        "append": {"tokens_per_call": B, "layers_per_call": L, "us_per_call": 1e3 * app_ms,
                   "timing": f"graphs of 8 calls, median of {n_append} replays"},
        "prefill_chunk": {"tokens_per_request": chunk, "tokens_per_call": T, "layers_per_call": L,
                          "ms_per_call": pre_ms, "tokens_per_s": T * L / (pre_ms * 1e-3),
                          "mirror_write_gbs": T * L * mirror_per_tok / (pre_ms * 1e-3) / 1e9},
        "note": "ssa_store_kv_mirror captured in CUDA graphs, on the filled cache after the "
                "decode measurements; positions stored again (same work as a first store)",
    }


def kernel_probe(args) -> dict:
    """One kernel of the step alone, on the workload's shape: the indexer over
    a random slab, or the attention over a random pool of B*W slots with k+1
    selected pages per request (ascending, the last page included) bound to
    slots b*W + i.  The pool is small, so an ncu capture of the launch holds
    little device memory; the work per launch is the step's.  Returns the
    median of --steps timed calls (after --warmup), L2 flushed before each."""
    import torch
    import sparse_attention_decode_indexer_gb300 as ssa
    from sparse_attention_decode_indexer_gb300.runner import DecodeRunner
    w = get_workload(args.workload)
    L, B, n, P, k = w.n_layers, w.batch, w.pages_per_request, w.page_size, w.block_topk
    W = 2 * k + 8
    lay = ssa.Layout(P, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8, L, B * n, B * W, B, n, k)
    bt = torch.arange(B * n, dtype=torch.int32).reshape(B, n)
    run = DecodeRunner(lay, host_tier=False, identity=True, block_table=bt,
                       seq_lens=[n * P] * B)
    c = run.cache
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    q = torch.randn((L, B, w.n_q_heads, w.head_dim), generator=g,
                    device="cuda").to(torch.bfloat16)
    if args.kernel == "index":
        c.slab.copy_(torch.randint(-127, 128, c.slab.shape, generator=g, device="cuda",
                                   dtype=torch.int32).to(torch.int8))

        def call():
            ssa.ssa_index_topk(c, 0, L, q, run.block_table, run.seq_lens, run.sel, run.n_sel,
                               None, run.status, run.ws)
        nbytes = index_bytes(w)
    else:
        if w.fp8:
            for pool in (c.k_pool, c.v_pool):      # finite e4m3 codes of both signs
                codes = torch.randint(0, 126, pool.shape, generator=g, device="cuda",
                                      dtype=torch.int32)
                sign = torch.randint(0, 2, pool.shape, generator=g, device="cuda",
                                     dtype=torch.int32) * 128
                pool.copy_((codes + sign).to(torch.uint8))
            for sc in (c.k_scale, c.v_scale):
                sc.copy_(torch.rand(sc.shape, generator=g, device="cuda") * 0.01 + 0.001)
        else:
            for pool in (c.k_pool, c.v_pool):
                pool.copy_(torch.randn(pool.numel() // 2, generator=g, device="cuda")
                           .to(torch.bfloat16).view(torch.uint8).view(pool.shape))
        sel = torch.full((L, B, W), -1, dtype=torch.int32)
        phys = torch.full((L, B, W), -1, dtype=torch.int32)
        gh = torch.Generator().manual_seed(w.seed)
        for l in range(L):
            for b in range(B):
                pages = torch.randperm(n - 1, generator=gh)[:k]
                pages = torch.sort(torch.cat([pages, torch.tensor([n - 1])])).values
                sel[l, b, :k + 1] = pages.int()
                phys[l, b, :k + 1] = torch.arange(b * W, b * W + k + 1, dtype=torch.int32)
        sel, phys = sel.cuda(), phys.cuda()

        def call():
            ssa.ssa_sparse_paged_decode(c, 0, L, q, sel, phys, run.seq_lens, run.sm_scale,
                                        run.out, run.status, run.ws)
        nbytes = decode_bytes(w)
    flush = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    ts = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            ts.append(e0.elapsed_time(e1) * 1e3)
    st = int(run.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st}: {ssa.status_str(st)}")
    us = statistics.median(ts)
    peak, kind = load_peaks()
    return {"kernel": args.kernel, "workload": w.name, "us_per_call": us,
            "alg_bytes": nbytes, "achieved_gbs": nbytes / (us * 1e-6) / 1e9,
            "frac": nbytes / (us * 1e-6) / 1e9 / peak, "peak_gbs": peak, "peak_kind": kind,
            "note": "one kernel alone on the workload's shape, random contents, small pool; "
                    "median of the timed calls, L2 flushed before each"}


def main():
    args = parse_args()
    if args.kernel:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        print(json.dumps(kernel_probe(args)))
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = get_workload(args.workload)
    if args.impl == "reference":
        if rank != 0:
            return
        cb = cpu_oracle_sample(w, args.cpu_seconds * max(1, min(args.steps, 5)) / 5)
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                # one step = every layer of every request, at the sample's rate
                "ms_per_step": 1e3 * w.n_layers * w.batch / cb["value"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64 attention, int32 indexer", "data": "synthetic",
                "config": {"workload": w.name}, "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    res = run_ours(args, rank, world, dist)
    if rank == 0:
        line, w = res
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_oracle_sample(w, args.cpu_seconds)
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
