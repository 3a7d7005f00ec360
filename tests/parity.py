"""Run the oracle and the CUDA library side by side on one seeded workload.

Used by the GPU parity tests and by the smoke check.  Inputs come only from
``workloads``; expected values come only from ``oracle``.  Bit-exact checks:
scores, selection, n_sel, remapped table, miss lists, LRU state, slab, and the
pool/mirror bytes of every bound slot.  Attention outputs: max-abs error
against the fp64 oracle within TOL (bf16 1e-2, fp8 3e-2).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as wl

TOL = {False: 1e-2, True: 3e-2}


def oracle_state(w: wl.Workload, layers=None) -> oracle.OracleKV:
    lay = oracle.OracleLayout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8,
                              w.n_layers, w.logical_pages, w.slots, w.batch,
                              w.pages_per_request, w.block_topk)
    return oracle.OracleKV(lay, host_tier=w.host_tier, identity=not w.host_tier)


def gpu_runner(w: wl.Workload, preload_width: int = 0, fetch_in_attention: bool = False,
               overlap_groups: int = 0):
    from sparse_attention_decode_indexer_gb300 import Layout
    from sparse_attention_decode_indexer_gb300.runner import DecodeRunner
    lay = Layout(w.page_size, w.n_q_heads, w.n_kv_heads, w.head_dim, w.fp8, w.n_layers,
                 w.logical_pages, w.slots, w.batch, w.pages_per_request, w.block_topk)
    return DecodeRunner(lay, host_tier=w.host_tier, identity=not w.host_tier,
                        block_table=wl.block_table(w), seq_lens=w.lens,
                        preload_width=preload_width, fetch_in_attention=fetch_in_attention,
                        overlap_groups=overlap_groups)


def _u16_to_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def prefill(w: wl.Workload, run, orc, oracle_layers):
    """Store every layer on the GPU; store the sampled layers in the oracle."""
    for l in range(w.n_layers):
        k, v, pos = wl.store_batch(w, l)
        kd = _u16_to_bf16(k).cuda()[None]
        vd = _u16_to_bf16(v).cuda()[None]
        run.store(l, 1, kd, vd, torch.from_numpy(pos).cuda())
        if l in oracle_layers:
            assert orc.store(l, k, v, pos) == 0
    torch.cuda.synchronize()


def gpu_pool_as_oracle_layout(w: wl.Workload, pool: torch.Tensor, is_v: bool) -> np.ndarray:
    """The library stores fp8 V d-major ([Hkv][D][P] per page); the oracle keeps
    [Hkv][P][D].  Return the library's bytes rearranged to the oracle's layout."""
    a = pool.cpu().numpy()
    if w.fp8 and is_v:
        n = a.shape[0]
        a = a.reshape(n, w.n_kv_heads, w.head_dim, w.page_size).transpose(0, 1, 3, 2)
        a = np.ascontiguousarray(a).reshape(n, w.n_kv_heads * w.page_size * w.head_dim)
    return a


def compare_state(w, run, orc, l, check_pool=True):
    c = run.cache
    assert np.array_equal(c.slot_of[l].cpu().numpy(), orc.slot_of[l]), "slot_of"
    assert np.array_equal(c.page_of[l].cpu().numpy(), orc.page_of[l]), "page_of"
    assert np.array_equal(c.last_use[l].cpu().numpy(), orc.last_use[l]), "last_use"
    assert int(c.clock[l].item()) == int(orc.clock[l]), "clock"
    if not check_pool:
        return
    bound = np.nonzero(orc.page_of[l] >= 0)[0]
    for name, is_v in (("k_pool", False), ("v_pool", True)):
        g = gpu_pool_as_oracle_layout(w, getattr(c, name)[l][torch.from_numpy(bound).cuda()], is_v)
        assert np.array_equal(g, getattr(orc, name)[l][bound]), name
    if w.fp8:
        for name in ("k_scale", "v_scale"):
            g = getattr(c, name)[l].cpu().numpy()[bound]
            assert np.array_equal(g, getattr(orc, name)[l][bound]), name


def compare_slab(run, orc, l):
    c = run.cache
    assert np.array_equal(c.slab_cnt[l].cpu().numpy(), orc.slab_cnt[l]), "slab_cnt"
    assert np.array_equal(c.slab_sum[l].cpu().numpy(), orc.slab_sum[l]), "slab_sum"
    assert np.array_equal(c.slab_scale[l].cpu().numpy(), orc.slab_scale[l]), "slab_scale"
    assert np.array_equal(c.slab[l].cpu().numpy(), orc.slab[l]), "slab"


def compare_mirror(w, run, orc, l):
    c = run.cache
    if c.k_mirror is None:
        return
    k = c.k_mirror[l].numpy()
    v = c.v_mirror[l].numpy()
    if w.fp8:
        n = v.shape[0]
        v = np.ascontiguousarray(v.reshape(n, w.n_kv_heads, w.head_dim, w.page_size)
                                 .transpose(0, 1, 3, 2)).reshape(n, w.n_kv_heads * w.page_size
                                                                 * w.head_dim)
    assert np.array_equal(k, orc.k_mirror[l]), "k_mirror"
    assert np.array_equal(v, orc.v_mirror[l]), "v_mirror"
    if w.fp8:
        assert np.array_equal(c.k_scale_mirror[l].numpy(), orc.k_scale_m[l]), "k_scale_mirror"
        assert np.array_equal(c.v_scale_mirror[l].numpy(), orc.v_scale_m[l]), "v_scale_mirror"


def run_parity(w: wl.Workload, oracle_layers=None, steps=None, per_layer=False,
               check_pool=True, check_mirror=True, report=None, pool_every_step=True,
               preload_width=0, fetch_in_attention=False, overlap_groups=0):
    """Run ``steps`` decode steps of ``w`` on both sides and compare.

    The library always runs every layer (one launch per stage covers them
    all, as the benchmark does); the oracle runs ``oracle_layers``.  With
    pool_every_step=False the pool bytes are compared after the last step
    only (the residency state is still compared after every step)."""
    oracle_layers = list(range(w.n_layers)) if oracle_layers is None else list(oracle_layers)
    steps = w.steps if steps is None else steps
    orc = oracle_state(w)
    run = gpu_runner(w, preload_width, fetch_in_attention, overlap_groups)
    prefill(w, run, orc, oracle_layers)
    assert int(run.status.item()) == 0, f"status {run.status.item()}"
    for l in oracle_layers:
        compare_slab(run, orc, l)
        if check_mirror:
            compare_mirror(w, run, orc, l)
        compare_state(w, run, orc, l, check_pool)
    qs = {l: wl.queries(w, l) for l in range(w.n_layers)}
    bt = wl.block_table(w)
    max_err = 0.0
    misses = 0
    max_layer_misses = 0
    fetched = 0
    for t in range(steps):
        q = np.stack([qs[l][t] for l in range(w.n_layers)])
        qd = _u16_to_bf16(q).cuda()
        run.step(qd, per_layer=per_layer, keep_scores=True)
        torch.cuda.synchronize()
        assert int(run.status.item()) == 0, f"status {run.status.item()} at step {t}"
        for l in oracle_layers:
            r = orc.step(l, qs[l][t], bt, w.lens)
            assert r["drops"] == 0 and r["flags"] == 0 and r["unresolved"] == 0
            g_scores = (run.last_scores if preload_width else run.scores)[l].cpu().numpy()
            assert np.array_equal(g_scores, r["scores"]), f"scores layer {l} step {t}"
            assert np.array_equal(run.sel[l].cpu().numpy(), r["sel"]), f"sel layer {l} step {t}"
            assert np.array_equal(run.n_sel[l].cpu().numpy(), r["n_sel"]), "n_sel"
            nm = int(run.n_miss[l].item())
            assert nm == r["n_miss"], f"n_miss {nm} vs {r['n_miss']} layer {l} step {t}"
            assert np.array_equal(run.miss_page[l].cpu().numpy(), r["miss_page"]), "miss_page"
            assert np.array_equal(run.miss_slot[l].cpu().numpy(), r["miss_slot"]), "miss_slot"
            g_phys = run.phys[l].cpu().numpy()
            if fetch_in_attention:
                # the pages this step bound are marked -2 - slot for the attention to fetch:
                # exactly the oracle's misses
                marked = g_phys <= -2
                g_phys = np.where(marked, -2 - g_phys, g_phys)
                ids = np.where(r["sel"] >= 0, bt[np.arange(w.batch)[:, None],
                                                 np.maximum(r["sel"], 0)], -1)
                assert set(ids[marked].tolist()) == set(r["miss_page"][:r["n_miss"]].tolist())
            assert np.array_equal(g_phys, r["phys"]), f"phys layer {l} step {t}"
            if preload_width:
                g_sc = run.last_scores[l].cpu().numpy()
                assert np.array_equal(g_sc, r["scores"]), f"preload scores layer {l} step {t}"
                fp, fs, fn, ffl = orc.prefetch(l, preload_width, r["scores"], w.lens, bt)
                assert ffl == 0
                assert int(run.n_fetch[l].item()) == fn, f"n_fetch layer {l} step {t}"
                assert np.array_equal(run.fetch_page[l].cpu().numpy(), fp), "fetch_page"
                assert np.array_equal(run.fetch_slot[l].cpu().numpy(), fs), "fetch_slot"
                fetched += fn
            compare_state(w, run, orc, l,
                          check_pool and (pool_every_step or t == steps - 1))
            out = run.out[l].float().cpu().numpy()
            err = float(np.abs(out - r["out"]).max())
            max_err = max(max_err, err)
            assert err <= TOL[w.fp8], f"max abs err {err} layer {l} step {t}"
            misses += nm
            max_layer_misses = max(max_layer_misses, nm)
    if report is not None:
        report.update(max_err=max_err, misses=misses, max_layer_misses=max_layer_misses,
                      fetched=fetched)
    return run, orc
