"""The C-ABI boundary, on the CPU: the library builds, loads, exports every
symbol include/ssa.h declares, and rejects bad arguments on the host with the
documented codes before anything reaches a GPU (no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "ssa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ssa_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    from sparse_attention_decode_indexer_gb300 import build
    build.build()
    import sparse_attention_decode_indexer_gb300 as m
    return m


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 10
    lib = ctypes.CDLL(L.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(L.EXPORTS) == set(names)


def _layout(L, **kw):
    base = dict(page_size=64, n_q_heads=16, n_kv_heads=2, head_dim=128, fp8=True, n_layers=2,
                logical_pages=100, pool_slots=80, batch=1, max_pages=100, block_topk=32)
    base.update(kw)
    return L.Layout(**base)


def _fake_cache(L, mirror=True):
    p = ctypes.c_void_p(0x10000)
    c = L.SsaCache(*([p] * 16))
    if not mirror:
        c.k_mirror = c.v_mirror = c.k_scale_mirror = c.v_scale_mirror = None
    return c


def test_workspace_size_and_layout_checks(L):
    lib = L.lib()
    good = _layout(L).c()
    assert lib.ssa_workspace_size(ctypes.byref(good)) > 0
    for bad in (dict(head_dim=64), dict(page_size=48), dict(n_q_heads=17),
                dict(n_q_heads=32, n_kv_heads=2), dict(batch=0), dict(block_topk=0)):
        lay = _layout(L, **bad).c()
        assert lib.ssa_workspace_size(ctypes.byref(lay)) == 0, bad
    lay = _layout(L).c()
    lay.max_sel = 71                          # must be 2k + 8
    assert lib.ssa_workspace_size(ctypes.byref(lay)) == 0
    lay = _layout(L).c()
    lay.kv_dtype = 7
    assert lib.ssa_workspace_size(ctypes.byref(lay)) == 0


def test_host_side_errors_are_returned_before_any_launch(L):
    lib = L.lib()
    lay = _layout(L).c()
    c = _fake_cache(L)
    p = ctypes.c_void_p(0x10000)
    # null outputs
    assert lib.ssa_index_topk(ctypes.byref(lay), ctypes.byref(c), 0, 1, p, p, p, None, p, p, p,
                              p, None) == -1
    # layer range past the cache
    assert lib.ssa_remap_block_table(ctypes.byref(lay), ctypes.byref(c), 1, 2, p, p, p, p,
                                     None) == -1
    # pool smaller than one batch selection: 80 < 72 * 2
    lay2 = _layout(L, batch=2, logical_pages=200, max_pages=100).c()
    assert lib.ssa_ensure_resident(ctypes.byref(lay2), ctypes.byref(c), 0, 1, p, p, p, p, p, p,
                                   p, None) == -2
    # unsupported dtype
    lay3 = _layout(L).c()
    lay3.kv_dtype = 9
    assert lib.ssa_store_kv_mirror(ctypes.byref(lay3), ctypes.byref(c), 0, 1, p, p, p, 4, p,
                                   None) == -3
    # a partial mirror
    c2 = _fake_cache(L)
    c2.v_scale_mirror = None
    assert lib.ssa_ensure_resident(ctypes.byref(lay), ctypes.byref(c2), 0, 1, p, p, p, p, p, p,
                                   p, None) == -4


def test_status_strings(L):
    assert L.status_str(0) == "ok"
    assert "pool_slots" in L.status_str(-2)
    assert L.status_str(1 | 8) == "drop|unresolved"
    assert L.status_str(32) == "timeout"
    assert L.status_str(64 | 2) == "bad_id|internal"


def test_binding_refuses_to_run_without_the_library(tmp_path, monkeypatch):
    import sparse_attention_decode_indexer_gb300 as m
    monkeypatch.setattr(m, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(RuntimeError):
        m.lib()


def test_more_host_side_rejections(L):
    """The remaining documented host-side rejections, each before any launch."""
    lib = L.lib()
    p = ctypes.c_void_p(0x10000)
    c = _fake_cache(L)
    UNSUPPORTED, INVALID = -3, -1
    # KV heads: a power of two, at most 8
    for bad in (dict(n_q_heads=6, n_kv_heads=3), dict(n_q_heads=16, n_kv_heads=16)):
        lay = _layout(L, **bad).c()
        assert lib.ssa_workspace_size(ctypes.byref(lay)) == 0, bad
        assert lib.ssa_store_kv_mirror(ctypes.byref(lay), ctypes.byref(c), 0, 1, p, p, p, 4, p,
                                       None) == UNSUPPORTED, bad
    # a batch selection the LRU cannot sort in shared memory: 256 * 72 > 16,384
    lay = _layout(L, batch=256, logical_pages=25600, pool_slots=25600, max_pages=100).c()
    assert lib.ssa_workspace_size(ctypes.byref(lay)) == 0
    # more pages per request than the select keeps on chip
    lay = _layout(L, logical_pages=50000, pool_slots=50000, max_pages=50000).c()
    assert lib.ssa_workspace_size(ctypes.byref(lay)) == 0
    lay = _layout(L).c()
    # attention without its workspace
    assert lib.ssa_sparse_paged_decode(ctypes.byref(lay), ctypes.byref(c), 0, 1, p, p, p, p,
                                       0.088, p, p, None, None) == INVALID
    # store: a negative token count, or tokens without their data
    assert lib.ssa_store_kv_mirror(ctypes.byref(lay), ctypes.byref(c), 0, 1, p, p, p, -1, p,
                                   None) == INVALID
    assert lib.ssa_store_kv_mirror(ctypes.byref(lay), ctypes.byref(c), 0, 1, None, p, p, 4, p,
                                   None) == INVALID
    # ensure with neither a workspace nor the miss outputs
    assert lib.ssa_ensure_resident(ctypes.byref(lay), ctypes.byref(c), 0, 1, p, p, None, None,
                                   None, p, None, None) == INVALID
    # an fp8 cache without its scale banks
    c2 = _fake_cache(L)
    c2.k_scale = None
    assert lib.ssa_sparse_paged_decode(ctypes.byref(lay), ctypes.byref(c2), 0, 1, p, p, p, p,
                                       0.088, p, p, p, None) == INVALID


def test_split_ensure_host_side_rejections(L):
    """ssa_ensure_remap_bind / ssa_fetch_misses: the lists are required, the
    fetch needs the mirror, the layer range and the pool size are checked --
    all on the host, before any launch."""
    lib = L.lib()
    p = ctypes.c_void_p(0x10000)
    c = _fake_cache(L)
    lay = _layout(L).c()
    INVALID, SMALL, NO_MIRROR = -1, -2, -4
    # bind: every list and phys required
    for i in range(4):
        args = [p, p, p, p]
        args[i] = None
        assert lib.ssa_ensure_remap_bind(ctypes.byref(lay), ctypes.byref(c), 0, 1, p, p,
                                         args[0], args[1], args[2], args[3], p, None) == INVALID
    # bind: the pool must hold one batch selection (80 < 2 * 72)
    lay2 = _layout(L, batch=2, logical_pages=200, max_pages=100).c()
    assert lib.ssa_ensure_remap_bind(ctypes.byref(lay2), ctypes.byref(c), 0, 1, p, p, p, p, p,
                                     p, p, None) == SMALL
    # fetch: lists required, range inside the cache, a full mirror
    assert lib.ssa_fetch_misses(ctypes.byref(lay), ctypes.byref(c), 0, 1, None, p, p, p,
                                None) == INVALID
    assert lib.ssa_fetch_misses(ctypes.byref(lay), ctypes.byref(c), 1, 2, p, p, p, p,
                                None) == INVALID
    c2 = _fake_cache(L, mirror=False)
    assert lib.ssa_fetch_misses(ctypes.byref(lay), ctypes.byref(c2), 0, 1, p, p, p, p,
                                None) == NO_MIRROR


def test_variant_calls_host_side_rejections(L):
    """The documented host-side rejections of the step's variant calls (fused
    ensure, deferred ensure and fetch-mode attention, host-tail attention,
    shared residency, top-k preload, the static-scratch indexer, the host-link
    probe), each returned before any launch."""
    lib = L.lib()
    p = ctypes.c_void_p(0x10000)
    c = _fake_cache(L)
    nomir = _fake_cache(L, mirror=False)
    lay = _layout(L).c()
    INVALID, UNSUPPORTED, NO_MIRROR, SCRATCH = -1, -3, -4, -6
    by = ctypes.byref
    # the fused ensure needs phys
    assert lib.ssa_ensure_remap(by(lay), by(c), 0, 1, p, p, None, p, p, p, p, p, None) == INVALID
    # deferred ensure: phys required, and the attention will fetch from the mirror
    assert lib.ssa_ensure_remap_deferred(by(lay), by(c), 0, 1, p, p, None, p, p, p, p, p,
                                         None) == INVALID
    assert lib.ssa_ensure_remap_deferred(by(lay), by(nomir), 0, 1, p, p, p, p, p, p, p, p,
                                         None) == NO_MIRROR
    # fetch-mode attention: block table and mirror required
    assert lib.ssa_sparse_paged_decode_fetch(by(lay), by(c), 0, 1, p, p, p, None, p, 0.088, p,
                                             p, p, None) == INVALID
    assert lib.ssa_sparse_paged_decode_fetch(by(lay), by(nomir), 0, 1, p, p, p, p, p, 0.088, p,
                                             p, p, None) == NO_MIRROR
    # host-tail attention: block table, slot_of and mirror required
    assert lib.ssa_sparse_paged_decode_host_tail(by(lay), by(c), 0, 1, p, p, None, p, 0.088, p,
                                                 p, p, None) == INVALID
    assert lib.ssa_sparse_paged_decode_host_tail(by(lay), by(nomir), 0, 1, p, p, p, p, 0.088, p,
                                                 p, p, None) == NO_MIRROR
    noslot = _fake_cache(L)
    noslot.slot_of = None
    assert lib.ssa_sparse_paged_decode_host_tail(by(lay), by(noslot), 0, 1, p, p, p, p, 0.088,
                                                 p, p, p, None) == INVALID
    # shared residency: the union of a call's selections is sorted in shared
    # memory, at most 16,384 entries (2 layers x 128 requests x 72 > 16,384)
    big = _layout(L, batch=128, logical_pages=20000, pool_slots=20000, max_pages=100).c()
    assert lib.ssa_ensure_remap_shared(by(big), by(c), 0, 2, p, p, p, p, p, p, p, p,
                                       None) == UNSUPPORTED
    assert lib.ssa_ensure_remap_shared(by(lay), by(c), 0, 1, p, p, None, p, p, p, p, p,
                                       None) == INVALID
    # top-k preload: width in [1, max_sel], scores and a workspace required
    for width in (0, 73):
        assert lib.ssa_prefetch_pages(by(lay), by(c), 0, 1, p, p, p, width, p, p, p, p, p,
                                      None) == INVALID, width
    assert lib.ssa_prefetch_pages(by(lay), by(c), 0, 1, None, p, p, 8, p, p, p, p, p,
                                  None) == INVALID
    assert lib.ssa_prefetch_pages(by(lay), by(c), 0, 1, p, p, p, 8, p, p, p, p, None,
                                  None) == INVALID
    # the static-scratch indexer: n_layers * batch * max_pages above its scratch
    huge = _layout(L, n_layers=2, batch=64, logical_pages=64 * 10000, pool_slots=64 * 72,
                   max_pages=10000).c()
    assert lib.ssa_workspace_size(by(huge)) > 0          # a layout the library accepts
    assert lib.ssa_index_topk_static_scratch(by(huge), by(c), 0, 2, p, p, p, p, p, p,
                                             None) == SCRATCH
    # the host-link probe: aligned buffers, chunk a multiple of 16 bytes, 4/8/16 loads
    assert lib.ssa_host_read_probe(p, p, p, 4, 24, 8, None) == INVALID
    assert lib.ssa_host_read_probe(p, p, p, 4, 4096, 6, None) == INVALID
    assert lib.ssa_host_read_probe(ctypes.c_void_p(0x10008), p, p, 4, 4096, 8, None) == INVALID
    assert lib.ssa_host_read_probe(p, p, p, 0, 4096, 8, None) == INVALID
