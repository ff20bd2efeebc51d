"""The stream-K schedule choice (host logic, no GPU): the invariants the
kernel relies on and the cost model's decisions on the shapes it was
calibrated on.

The kernel deals units [floor(U c / G), floor(U (c+1) / G)) of the split tiles
to cluster c; an owner counts its contributors as the clusters after it whose
ranges start inside the tile, which is only right if no range is empty, i.e.
U >= G.  These tests walk that partition in Python for many tile counts."""
import itertools

import pytest

import dense_gemm_blackwell_tcgen05_gb300 as g


def ranges(plan, kt, unit):
    ku = -(-kt // unit)
    U = plan["sk_tiles"] * ku
    G = plan["clusters"]
    return [(U * c // G, U * (c + 1) // G) for c in range(G)], ku


CASES = list(itertools.product([1, 5, 37, 75, 76, 77, 151, 152, 153, 300, 1024],
                               [76, 148, 152], [1, 2, 3, 17, 128], [1, 4]))


@pytest.mark.parametrize("mode", [g.STREAMK_AUTO, g.STREAMK_ALWAYS])
def test_partition_invariants(mode):
    for tiles, resident, kt, unit in CASES:
        p = g.gemm_streamk_plan(tiles, resident, kt, unit, mode)
        assert p["dp_tiles"] + p["sk_tiles"] == tiles
        ku = -(-kt // unit)
        if p["sk_tiles"] == 0:
            assert p["clusters"] == min(tiles, resident)
            continue
        assert ku >= 2 and tiles % resident != 0
        assert p["clusters"] <= resident
        if p["dp_tiles"]:
            # whole waves first, on every resident cluster
            assert p["clusters"] == resident
            assert p["dp_tiles"] % resident == 0
            assert p["sk_tiles"] == tiles % resident + resident
        rs, ku = ranges(p, kt, unit)
        assert all(b > a for a, b in rs), (tiles, resident, kt, unit, "empty range")
        # every unit of every split tile is dealt exactly once, in order
        assert rs[0][0] == 0 and rs[-1][1] == p["sk_tiles"] * ku
        assert all(rs[i][1] == rs[i + 1][0] for i in range(len(rs) - 1))
        # each split tile has exactly one owner (the range holding its first unit)
        for t in range(p["sk_tiles"]):
            owners = [c for c, (a, b) in enumerate(rs) if a <= t * ku < b]
            assert len(owners) == 1


def test_always_splits_every_partial_wave():
    for tiles, resident, kt, unit in CASES:
        p = g.gemm_streamk_plan(tiles, resident, kt, unit, g.STREAMK_ALWAYS)
        splittable = tiles % resident != 0 and -(-kt // unit) >= 2
        assert (p["sk_tiles"] > 0) == splittable


def test_never_is_data_parallel():
    for tiles, resident, kt, unit in CASES:
        p = g.gemm_streamk_plan(tiles, resident, kt, unit, g.STREAMK_NEVER)
        assert p == {"dp_tiles": tiles, "sk_tiles": 0, "clusters": min(tiles, resident)}


def test_cost_model_decisions():
    plan = lambda *a: g.gemm_streamk_plan(*a, g.STREAMK_AUTO)
    # 1024 x 1024 x 16384 bf16 on 152 one-CTA clusters: 32 tiles of 256 K-tiles
    assert plan(32, 152, 256, 1)["sk_tiles"] == 32
    # 300 x 520 x 1040: 17 K-tiles, the fix-up costs more than the split saves
    assert plan(9, 152, 17, 1)["sk_tiles"] == 0
    # full waves: nothing to balance
    assert plan(304, 152, 128, 1)["sk_tiles"] == 0
    # an almost full last wave saves less than the fix-up costs
    assert plan(144, 76, 128, 1)["sk_tiles"] == 0


def test_plan_argument_checks():
    bad = [(-1, 76, 8, 1, 0), (8, 0, 8, 1, 0), (8, 76, -1, 1, 0), (8, 76, 8, 0, 0), (8, 76, 8, 1, 3)]
    for args in bad:
        with pytest.raises(g.GemmError):
            g.gemm_streamk_plan(*args)
    assert g.gemm_streamk_plan(0, 76, 8, 1) == {"dp_tiles": 0, "sk_tiles": 0, "clusters": 0}
