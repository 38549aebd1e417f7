"""Host-side checks of the static work schedule (no GPU): every work item is assigned to
exactly one CTA, lists run longest item first (shortest first in the two-tile kernel at
head_dim 128 when L <= 512, where every item lies within one 512-query block), and the
longest-processing-time-first assignment keeps the busiest CTA close to the lower bound."""
import math

import pytest

import scaled_dot_product_sdpa_gb300 as gb


def _kind(d, flags):
    if flags & 8:
        return "dsplit"  # one item per head and query tile, dealt to clusters of two CTAs
    return "single" if d > 128 or flags & 3 else "pair"


def _units(B, H, L, d, causal, flags, r):
    """Work units of item r, from the item numbering documented with the kernels."""
    BH, nQ, nQB = B * H, math.ceil(L / 128), math.ceil(L / 256)
    kind = _kind(d, flags)
    if kind == "pair":
        if not causal:
            return 2 * nQ
        qb = nQB - 1 - r // BH
        return (2 * qb + 1) + min(2 * qb + 2, nQ)
    dvs = d // 256 if d > 256 and kind == "single" else 1
    if not causal:
        return nQ
    return nQ - 1 - r // (BH * dvs) + 1


def _n_items(B, H, L, d, flags):
    BH, nQ, nQB = B * H, math.ceil(L / 128), math.ceil(L / 256)
    kind = _kind(d, flags)
    if kind == "pair":
        return BH * nQB
    if kind == "dsplit":
        return BH * nQ
    return BH * nQ * (d // 256 if d > 256 else 1)


def _fixed_order(n, grid):
    """The kernels' own order when no table is passed: CTA c takes items c, 2G-1-c,
    2G+c, ... (G = grid) below n."""
    lists = [[] for _ in range(grid)]
    p = 0
    while p * grid < n:
        for c in range(grid):
            r = p * grid + ((grid - 1 - c) if p & 1 else c)
            if r < n:
                lists[c].append(r)
        p += 1
    return lists


def _schedule(B, H, L, d, causal, grid, flags):
    """The per-CTA item lists a launch runs: the table, or the fixed order when the host
    passes none (at most one item per CTA, where the two coincide)."""
    sched = gb.attn_debug_schedule(B, H, L, d, causal, grid, flags)
    if sched is None:
        n = _n_items(B, H, L, d, flags)
        assert n <= grid, "only a launch of at most one item per CTA runs without a table"
        sched = _fixed_order(n, grid)
    return sched


CASES = [(8, 32, 512, 128, True, 0), (1, 32, 1024, 128, True, 0), (1, 16, 512, 64, True, 0),
         (1, 8, 128, 64, False, 0), (1, 8, 2048, 512, True, 0), (8, 32, 512, 128, True, 2),
         (2, 3, 1000, 64, False, 0), (1, 5, 777, 128, True, 1), (1, 8, 2048, 512, True, 2),
         (2, 3, 1000, 512, False, 8)]


@pytest.mark.parametrize("B,H,L,d,causal,flags", CASES)
@pytest.mark.parametrize("grid", [1, 7, 152])
def test_every_item_exactly_once(B, H, L, d, causal, flags, grid):
    n = _n_items(B, H, L, d, flags)
    sched = _schedule(B, H, L, d, causal, min(grid, n), flags)
    flat = sorted(i for lst in sched for i in lst)
    assert flat == list(range(n))


@pytest.mark.parametrize("B,H,L,d,causal,flags", CASES)
def test_lists_run_longest_first_and_balance(B, H, L, d, causal, flags):
    n = _n_items(B, H, L, d, flags)
    grid = min(152, n)
    sched = _schedule(B, H, L, d, causal, grid, flags)
    cost = [_units(B, H, L, d, causal, flags, r) for r in range(n)]
    shortest_first = _kind(d, flags) == "pair" and math.ceil(L / 256) <= 2 and d == 128
    for lst in sched:
        c = [cost[r] for r in lst]
        assert c == sorted(c, reverse=not shortest_first)
    loads = [sum(cost[r] for r in lst) for lst in sched]
    lower = max(sum(cost) / grid, max(cost))
    # LPT is within 4/3 of the optimum on costs; allow the per-item overhead term too.
    assert max(loads) <= 4.0 / 3.0 * lower + max(cost)


def test_single_tile_case_d_balances_to_the_mean():
    """caseD as single-tile items (1-4 units each): the busiest CTA is within one item
    of the mean load (2560 units over 152 CTAs = 16.8)."""
    sched = gb.attn_debug_schedule(8, 32, 512, 128, True, 152, gb.FLAG_SINGLE_TILE)
    loads = [sum(_units(8, 32, 512, 128, True, 2, r) for r in lst) for lst in sched]
    assert sum(loads) == 2560
    assert max(loads) <= 17 + 4


def test_too_many_items_falls_back_to_fixed_order():
    assert gb.attn_debug_schedule(1, 4000, 128, 64, False, 152, 0) is None


@pytest.mark.parametrize("B,H,L,d,causal,flags", [(1, 8, 128, 64, False, 0), (1, 16, 512, 64, True, 2),
                                                  (1, 32, 1024, 128, True, 0), (1, 3, 700, 512, True, 0)])
def test_one_item_per_cta_passes_no_table(B, H, L, d, causal, flags):
    """With at most one item per CTA the longest-first assignment is the kernels' own
    order (CTA c takes item c, items numbered longest first), so no table is built and
    the kernels read none; with one CTA fewer the table is back."""
    n = _n_items(B, H, L, d, flags)
    assert gb.attn_debug_schedule(B, H, L, d, causal, n, flags) is None
    cost = [_units(B, H, L, d, causal, flags, r) for r in range(n)]
    assert cost == sorted(cost, reverse=True)
    if n > 1:
        sched = gb.attn_debug_schedule(B, H, L, d, causal, n - 1, flags)
        assert sched is not None and sorted(i for lst in sched for i in lst) == list(range(n))


def test_schedule_rejects_bad_arguments():
    with pytest.raises(gb.GbattnError):
        gb.attn_debug_schedule(1, 1, 128, 48, False, 4)
    with pytest.raises(gb.GbattnError):
        gb.attn_debug_schedule(1, 1, 128, 64, False, 0)
