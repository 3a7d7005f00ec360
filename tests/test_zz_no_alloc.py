"""ssa_index_topk_static_scratch: the indexer + top-k call for callers that
cannot allocate device memory (a plugin whose host program owns every device
allocation, a serving loop that must not allocate after start-up).  Its score
scratch is a fixed array inside the library instead of a caller workspace.

Called through the C ABI and compared with ssa_index_topk, which takes a
workspace, on two calls in a row (the second reuses the array the first left
behind), and with the oracle's selection directly (the call runs its own pair
of kernels, a score kernel and a separate select kernel).  Selection results
are integers, so the comparisons are exact.  The file runs last so that a
failure here leaves every other test already run.
"""
import ctypes

import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu


def _w():
    return wl.Workload("noalloc", batch=3, n_layers=2, ctx=64 * 120 + 11,
                       seq_lens=(64 * 120 + 11, 64 * 90, 64 * 100 + 63), page_size=64,
                       n_q_heads=16, n_kv_heads=2, head_dim=128, fp8=True, block_topk=16,
                       pool_slots=3 * 40 + 7, steps=2, rho=0.8, walk_c=0.6, seed=202)


def test_static_scratch_matches_workspace_entry_point_on_two_calls():
    import torch
    import sparse_attention_decode_indexer_gb300 as ssa
    from tests.parity import gpu_runner, oracle_state, prefill

    w = _w()
    run = gpu_runner(w)
    orc = oracle_state(w)
    prefill(w, run, orc, oracle_layers=list(range(w.n_layers)))
    bt = wl.block_table(w)
    L = ssa.lib()
    fn = L.ssa_index_topk_static_scratch
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ssa.SsaLayout), ctypes.POINTER(ssa.SsaCache), ctypes.c_int,
                   ctypes.c_int] + [ctypes.c_void_p] * 7
    q_all = np.stack([wl.queries(w, l) for l in range(w.n_layers)], axis=1)   # [steps][L]...
    sel_b = torch.full_like(run.sel, -7)
    nsel_b = torch.full_like(run.n_sel, -7)
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    for t in range(2):
        q = torch.from_numpy(q_all[t].view(np.int16)).view(torch.bfloat16).cuda()
        ssa.ssa_index_topk(run.cache, 0, w.n_layers, q, run.block_table, run.seq_lens, run.sel,
                           run.n_sel, None, run.status, run.ws)
        rc = fn(ctypes.byref(run.cache._lay), ctypes.byref(run.cache.c), 0, w.n_layers,
                ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(run.block_table.data_ptr()),
                ctypes.c_void_p(run.seq_lens.data_ptr()), ctypes.c_void_p(sel_b.data_ptr()),
                ctypes.c_void_p(nsel_b.data_ptr()), ctypes.c_void_p(status.data_ptr()),
                ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, ssa.status_str(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and int(run.status.item()) == 0
        assert torch.equal(sel_b, run.sel), f"call {t}"
        assert torch.equal(nsel_b, run.n_sel), f"call {t}"
        assert (run.n_sel == w.block_topk + 1).all()
        for l in range(w.n_layers):
            o_sel, o_nsel, _, drops, bad = orc.index_topk(l, q_all[t][l], bt, w.lens)
            assert drops == 0 and bad == 0
            assert np.array_equal(sel_b[l].cpu().numpy(), o_sel), f"call {t} layer {l}"
            assert np.array_equal(nsel_b[l].cpu().numpy(), o_nsel), f"call {t} layer {l}"


def test_static_scratch_rejects_calls_beyond_its_size():
    import sparse_attention_decode_indexer_gb300 as ssa
    L = ssa.lib()
    fn = L.ssa_index_topk_static_scratch
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ssa.SsaLayout), ctypes.POINTER(ssa.SsaCache), ctypes.c_int,
                   ctypes.c_int] + [ctypes.c_void_p] * 7
    # 12 layers x 64 requests x 2,048 pages = 1.5 M scores > 1 M entries
    lay = ssa.Layout(64, 32, 4, 128, True, 12, 64 * 2048, 64 * 2048, 64, 2048, 32).c()
    p = ctypes.c_void_p(0x10000)
    cache = ssa.SsaCache(*([p] * 16))
    rc = fn(ctypes.byref(lay), ctypes.byref(cache), 0, 12, p, p, p, p, p, p, None)
    assert rc == -6
    assert "static score scratch" in ssa.status_str(rc)
