"""Host logic of the overlapped step: the split of a call's layers into ranges
(one copy call and one attention call per range).  No GPU."""
import pytest

from sparse_attention_decode_indexer_gb300.runner import split_layers


@pytest.mark.parametrize("L", [1, 2, 5, 12, 61])
@pytest.mark.parametrize("G", [0, 1, 2, 3, 4, 5, 6, 12, 100])
def test_ranges_cover_the_layers_in_order(L, G):
    r = split_layers(L, G)
    assert len(r) == max(1, min(G, L))
    # contiguous, in order, covering [0, L) exactly once
    assert r[0][0] == 0
    for (a0, an), (b0, _) in zip(r, r[1:]):
        assert b0 == a0 + an
    assert r[-1][0] + r[-1][1] == L
    sizes = [n for _, n in r]
    assert all(n >= 1 for n in sizes)
    # near-equal, the larger ranges first
    assert max(sizes) - min(sizes) <= 1
    assert sizes == sorted(sizes, reverse=True)


def test_examples():
    assert split_layers(12, 2) == [(0, 6), (6, 6)]
    assert split_layers(5, 3) == [(0, 2), (2, 2), (4, 1)]
    assert split_layers(12, 5) == [(0, 3), (3, 3), (6, 2), (8, 2), (10, 2)]
