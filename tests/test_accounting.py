"""Storage accounting (host arithmetic) against the figures the pages print."""
import os

import pytest

from cross_context_kv_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "storage_accounting.txt")
GIB = 1 << 30


def _rows():
    rows = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *vals = line.split()
                rows[key] = [float(v) for v in vals]
    return rows


def test_full_dimensional_anchor_pool_is_the_printed_50_gib():
    L, n, H, D, V, N, gib = _rows()["kvcmas_pool"]
    pool = acc.anchor_pool_bytes(int(L), int(n), int(H), int(D), int(V), int(N))
    assert pool["total"] == gib * GIB
    # 20 base caches of 512 MiB and 80 corrections of 512 MiB
    assert pool["bases"] == 10 * GIB and pool["corrections"] == 40 * GIB
    assert acc.kv_cache_bytes(int(L), int(n), int(H), int(D)) == 512 << 20


def test_low_rank_pool_stores_two_factors_per_layer_and_plane():
    L, n, H, D, V, N, _ = (int(x) for x in _rows()["kvcmas_pool"])
    r = 32
    one = acc.anchor_state_bytes(L, n, H, D, rank=r)
    # A is n x r and Bt is (H*D) x r per layer and plane, bf16
    assert one == L * 2 * (n * r + H * D * r) * 2 == 20 << 20
    pool = acc.anchor_pool_bytes(L, n, H, D, V, N, rank=r)
    assert pool["total"] == V * (1 + N) * one
    full = acc.anchor_pool_bytes(L, n, H, D, V, N)["total"]
    assert full / pool["total"] == pytest.approx(25.6)
    # the factors cost less than the dense state exactly when r < n H D / (n + H D)
    assert acc.anchor_state_bytes(L, n, H, D, rank=819) < acc.anchor_state_bytes(L, n, H, D)
    assert acc.anchor_state_bytes(L, n, H, D, rank=820) > acc.anchor_state_bytes(L, n, H, D)


@pytest.mark.parametrize("name", ["td_7b", "td_14b"])
def test_master_mirror_round_cost_and_reduction_as_printed(name):
    N, R, copies, reduction, mirror_pct = _rows()[name]
    c = acc.mirror_round_copies(int(N), R)
    assert round(c, 1) == copies
    # the page divides by the rounded cost
    assert round(N / round(c, 1), 1) == reduction
    assert acc.mirror_memory_reduction(int(N), R) == pytest.approx(N / c)
    assert round(100 / R) == mirror_pct


def test_mirror_cost_limits():
    assert acc.mirror_round_copies(1, 3.0) == 1.0          # a lone master
    assert acc.mirror_round_copies(10, 1.0) == 10.0        # incompressible mirrors: dense
    assert acc.mirror_memory_reduction(10, 1e12) == pytest.approx(10.0)
    with pytest.raises(ValueError):
        acc.mirror_round_copies(0, 2.0)


def test_diff_bytes_count_every_buffer():
    # 2 siblings, 1 layer, 64 tokens of 1 x 16 in 16-token blocks: 8 blocks, 3 dirty
    stored = acc.diff_stored_bytes(2, 1, 64, 1, 16, 16, entries=3)
    payload = 3 * 2 * 16 * 16 * 2
    assert stored == payload + 4 * 1 + 8 * 9
    split = acc.diff_stored_bytes(2, 1, 64, 1, 16, 16, entries=5, planes_per_entry=1, lists=2)
    assert split == 5 * 16 * 16 * 2 + 2 * (4 + 8 * 9)
    # nothing dirty: only the index remains; everything dirty: a little above dense
    dense = 2 * acc.kv_cache_bytes(1, 64, 1, 16)
    assert acc.diff_stored_bytes(2, 1, 64, 1, 16, 16, entries=8) > dense
    assert acc.diff_compression(2, 1, 64, 1, 16, 16, entries=8) < 1.0
