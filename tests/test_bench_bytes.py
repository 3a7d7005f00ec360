"""The bench's algorithmic bytes, the numerator of its roofline figures.

Per request-layer the method must move the int8 slab of every page
(n * (Hkv * D + 4)), the selected pages' K and V (n_sel * P * Hkv * D * 2
bytes of codes, bf16 twice that), the fp8 per-token scales (n_sel * P * 8),
and q, out, sel, phys.  The totals below are those figures for the three
fixed workloads as first worked out by hand, to 2-3 significant figures and
from rounded inputs (host_tier_196k_fp8 came to 1.92 MB per request-layer;
the exact count is 1.910), so they agree within 1 %; the hand count of the
second test is exact.
"""
import bench
import workloads as wl

# workload: (MB per request-layer, MB per step), worked out by hand
PRINTED = {
    "batched_32k_bf16_needles": (2.31, 110.7),
    "host_tier_196k_fp8": (1.92, 23.0),
    "lru_pressure_64k_fp8": (1.38, 66.1),
}


def test_step_bytes_match_the_printed_table():
    for name, (per_rl, per_step) in PRINTED.items():
        w = wl.WORKLOADS[name]
        total = bench.decode_bytes(w) + bench.index_bytes(w)
        assert abs(total / 1e6 - per_step) <= 0.01 * per_step, (name, total)
        assert abs(total / (w.n_layers * w.batch) / 1e6 - per_rl) <= 0.01 * per_rl, (name, total)


def test_decode_bytes_by_hand_for_the_bench_workload():
    # lru_pressure_64k_fp8: 4 requests x 12 layers, 1,024 pages each, top-32 + last
    # = 33 pages, 2 KV heads, P = 64, D = 128, e4m3 codes
    w = wl.WORKLOADS["lru_pressure_64k_fp8"]
    kv = 33 * 2 * 2 * 64 * 128               # K and V codes of the selected pages
    scales = 33 * 64 * 8                      # two fp32 scales per token
    q_out = 2 * 16 * 128 * 2                  # q in, out, bf16
    lists = 2 * 72 * 4                        # sel and phys, W = 2 * 32 + 8
    assert bench.decode_bytes(w) == 12 * 4 * (kv + scales + q_out + lists)
    slab = 1024 * (2 * 128 + 4)
    assert bench.index_bytes(w) == 12 * (4 * slab + 4 * 16 * 128 * 2)
    # one missed page: K and V codes of both KV heads plus the two scale banks
    assert bench.page_fetch_bytes(w) == 2 * 2 * 64 * 128 + 2 * 64 * 4
