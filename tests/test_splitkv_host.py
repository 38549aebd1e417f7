"""Host-side checks (no GPU) of the schedule with key-range splits (option FLAG_SPLIT_KV).

The split schedule ("An Optimal Mapper Meets a Real GPU", "Experiment one": split the key
reduction only coarsely; STAGE_D.md, section 2, "Merge": merging partial results is exact
only over disjoint key sets): a query tile may be split in two disjoint key ranges, one per
CTA of a cluster of two (CTAs 2c and 2c + 1), each range at least 3 key tiles (384 keys).
Every query tile must be computed exactly once: either as a plain item on one CTA, or as a
split item listed by both CTAs of one cluster, at the head of both lists, in the same order.
"""
import math

import pytest

import scaled_dot_product_sdpa_gb300 as gb


def _tiles(B, H, L, d, causal, r):
    BH, nQ, dvs = B * H, math.ceil(L / 128), (d // 256 if d > 256 else 1)
    return nQ - r // (BH * dvs) if causal else nQ


def _check(B, H, L, d, causal, grid):
    sched = gb.attn_debug_schedule(B, H, L, d, causal, grid, gb.FLAG_SPLIT_KV)
    assert sched is not None and len(sched) == grid
    n_items = B * H * math.ceil(L / 128) * (d // 256 if d > 256 else 1)
    plain, split = [], {}
    for c, lst in enumerate(sched):
        heads = [v for v in lst if v >= n_items]
        # split items come first
        assert lst[:len(heads)] == heads, f"CTA {c}: a split item after a plain one"
        for pos, v in enumerate(heads):
            split.setdefault(v, []).append((c, pos))
        plain += [v for v in lst if v < n_items]
    for v, where in split.items():
        (c0, p0), (c1, p1) = where  # exactly two CTAs ...
        assert c0 % 2 == 0 and c1 == c0 + 1 and p0 == p1, f"split item {v} at {where}"  # ... of one cluster
        n = _tiles(B, H, L, d, causal, v - n_items)
        assert n // 2 >= 3, f"split item with {n} key tiles: a part shorter than 3 tiles"
    covered = sorted(plain + [v - n_items for v in split])
    assert covered == list(range(n_items)), "every query tile exactly once"
    return sched, split


@pytest.mark.parametrize("B,H,L,d,causal,grid", [
    (1, 4, 4096, 128, True, 152), (1, 8, 4096, 128, True, 152), (1, 1, 16384, 128, True, 152),
    (1, 8, 2048, 512, True, 152), (1, 2, 2048, 64, False, 152), (1, 32, 1024, 128, True, 152),
    (1, 3, 1500, 64, True, 6), (1, 2, 1100, 512, False, 2), (2, 3, 2000, 128, True, 16),
])
def test_split_schedule_covers_every_tile_once(B, H, L, d, causal, grid):
    _check(B, H, L, d, causal, grid)


def test_split_schedule_splits_the_long_tiles_of_an_underfilled_grid():
    """4 heads x 32 query tiles (1 to 32 key tiles) on 152 SMs: without splits the longest
    tile alone (32 steps) sets the makespan; splitting the long ones roughly halves it."""
    sched, split = _check(1, 4, 4096, 128, True, 152)
    assert len(split) >= 8
    plain = gb.attn_debug_plan(1, 4, 4096, 128, True, 152, flags=gb.FLAG_SINGLE_TILE)
    sp = gb.attn_debug_plan(1, 4, 4096, 128, True, 152, flags=gb.FLAG_SPLIT_KV)
    assert sp["kind"] == 3 and plain["kind"] == 0
    assert sp["makespan"] < 0.7 * plain["makespan"]
    # the automatic plan takes the split kernel here ...
    assert gb.attn_debug_plan(1, 4, 4096, 128, True, 152)["kind"] == 3
    # ... but not for the workloads whose tiles are all short or whose grid is full
    for B, H, L, d in [(1, 8, 128, 64), (1, 16, 512, 64), (8, 32, 512, 128)]:
        assert gb.attn_debug_plan(B, H, L, d, True, 152)["kind"] != 3


def test_split_schedule_never_splits_short_tiles():
    """Tiles of fewer than 6 key tiles are never split (each part at least 384 keys)."""
    sched, split = _check(1, 16, 512, 64, True, 152)
    assert not split
    sched, split = _check(1, 8, 640, 128, True, 152)  # 5 key tiles at most
    assert not split


def test_split_flag_validation():
    with pytest.raises(gb.GbattnError):
        gb.attn_debug_plan(1, 2, 2048, 256, True, 152, flags=gb.FLAG_SPLIT_KV)  # no d = 256 variant
    with pytest.raises(gb.GbattnError):
        gb.attn_debug_plan(1, 2, 2048, 128, True, 152, flags=gb.FLAG_SPLIT_KV | gb.FLAG_SINGLE_TILE)
    with pytest.raises(gb.GbattnError):
        gb.attn_debug_schedule(1, 2, 2048, 128, True, 7, gb.FLAG_SPLIT_KV)  # odd CTA count
