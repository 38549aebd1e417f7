"""Host-side checks of the launch planner (attn_debug_plan; no GPU needed): which kernel
variant a launch uses, with how many work items and CTAs.

Kernels (include/gbattn.h, attn_fwd_ex): 0 single-tile (items: one 128-row query tile
per value-column half), 1 two-tile (items: 256-row query blocks), 3 single-tile with
key-range splits over clusters of two CTAs (the same items, some split).  The item counts below
follow from those definitions alone."""
import math

import pytest

import scaled_dot_product_sdpa_gb300 as gb

SM = 152


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from scaled_dot_product_sdpa_gb300 import build
    gb.load_library(build.build())


def _items(kind, B, H, L, d):
    nQ, nQB = math.ceil(L / 128), math.ceil(L / 256)
    if kind == 1:
        return B * H * nQB
    if kind == 2:
        return B * H * nQ
    return B * H * nQ * (d // 256 if d > 256 else 1)


SHAPES = [(1, 8, 128, 64, False), (1, 16, 512, 64, True), (1, 32, 1024, 128, True), (8, 32, 512, 128, True),
          (1, 8, 2048, 512, True), (2, 3, 1000, 64, False), (1, 4, 4096, 128, True), (4, 64, 2048, 64, False)]


@pytest.mark.parametrize("B,H,L,d,causal", SHAPES)
@pytest.mark.parametrize("flags,kind", [(2, 0), (1, 0), (4, 1)])
def test_flags_force_the_variant(B, H, L, d, causal, flags, kind):
    if d > 128 and flags in (1, 4):
        with pytest.raises(gb.GbattnError):
            gb.attn_debug_plan(B, H, L, d, causal, SM, flags=flags)
        return
    p = gb.attn_debug_plan(B, H, L, d, causal, SM, flags=flags)
    n = _items(kind, B, H, L, d)
    assert (p["kind"], p["items"], p["grid"]) == (kind, n, min(SM, n))


@pytest.mark.parametrize("B,H,L,d,causal", SHAPES)
def test_auto_plan(B, H, L, d, causal):
    p = gb.attn_debug_plan(B, H, L, d, causal, SM)
    if d == 512:  # the head_dim split only on request: clusters of two CTAs
        q = gb.attn_debug_plan(B, H, L, d, causal, SM, flags=gb.FLAG_DSPLIT)
        n = _items(2, B, H, L, d)
        assert (q["kind"], q["items"], q["grid"]) == (2, n, min(SM // 2, n))
    # Key-range splits (head_dim 64, 128, 512) replace the choice below when their schedule
    # is more than 10% shorter.
    split = gb.attn_debug_plan(B, H, L, d, causal, SM, flags=gb.FLAG_SPLIT_KV)["makespan"] if d != 256 else -1
    if d > 128:
        best = gb.attn_debug_plan(B, H, L, d, causal, SM, flags=gb.FLAG_SINGLE_TILE)["makespan"]
        if 0 <= split < 0.9 * best:
            assert (p["kind"], p["makespan"]) == (3, split)
        else:
            assert (p["kind"], p["makespan"]) == (0, best)
        return
    pair = gb.attn_debug_plan(B, H, L, d, causal, SM, flags=4)
    if pair["items"] >= 2 * SM:
        assert p["kind"] == 1  # enough blocks: the two-tile kernel, whose K/V reuse is highest
        return
    # Few blocks: the kernel with the shorter estimated schedule.
    alternatives = [gb.attn_debug_plan(B, H, L, d, causal, SM, flags=f)["makespan"] for f in (4, 2)]
    best = min(m for m in alternatives if m >= 0)
    if 0 <= split < 0.9 * best:
        assert (p["kind"], p["makespan"]) == (3, split)
    else:
        assert p["makespan"] == best and p["kind"] in (0, 1)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_dsplit_flag_only_at_512(d):
    with pytest.raises(gb.GbattnError):
        gb.attn_debug_plan(1, 2, 256, d, True, SM, flags=gb.FLAG_DSPLIT)


def test_dsplit_flag_alone():
    assert gb.attn_debug_plan(1, 2, 256, 512, True, SM, flags=gb.FLAG_DSPLIT)["kind"] == 2
    for other in (1, 2, 4):
        with pytest.raises(gb.GbattnError):
            gb.attn_debug_plan(1, 2, 256, 512, True, SM, flags=gb.FLAG_DSPLIT | other)


def test_grid_limit_caps_the_ctas():
    p = gb.attn_debug_plan(1, 32, 1024, 128, True, SM, flags=2, grid_limit=7)
    assert p["grid"] == 7 and p["items"] == 256


def test_rejects_bad_arguments():
    for kw in ({"sm_count": 0}, {"sm_count": 100000}, {"grid_limit": -1}):
        args = dict(B=1, H=2, L=256, d=64, causal=True, sm_count=SM)
        args.update(kw)
        with pytest.raises(gb.GbattnError):
            gb.attn_debug_plan(**args)
    with pytest.raises(gb.GbattnError):
        gb.attn_debug_plan(1, 2, 256, 96, True, SM)


# ----------------------------------------------------------------------------- decode
@pytest.mark.parametrize("B,H,L,d", [(8, 32, 8192, 128), (1, 8, 1 << 20, 128), (1, 1, 1, 64), (1, 1, 5, 64),
                                     (2, 3, 300, 64), (1, 1, 65, 512), (1, 2, 1000, 256), (64, 64, 4096, 64),
                                     (1, 1, 1 << 20, 512), (1, 1, 100000, 64), (2, 2, 40000, 128)])
@pytest.mark.parametrize("max_ranks", [8, 16])
@pytest.mark.parametrize("grouped", [False, True])
def test_decode_plan_covers_every_key(B, H, L, d, max_ranks, grouped):
    """Every key is owned by exactly one CTA of its head's clusters: the ranges
    [c*kpr, (c+1)*kpr) of the head's groups*ranks CTAs tile [0, L) (the last ones may be
    empty), in whole key tiles, with power-of-two clusters no larger than allowed, no more
    CTAs per head than key tiles, and one cluster per head without a workspace."""
    pl = gb.attn_debug_decode_plan(B, H, L, d, 152, max_ranks, grouped=grouped)
    r, kpr, g = pl["ranks"], pl["keys_per_rank"], pl["groups"]
    kt = 8192 // d
    tiles = -(-L // kt)
    assert r & (r - 1) == 0 and 1 <= r <= min(max_ranks, {64: 16, 128: 16, 256: 8, 512: 4}[d]) and r <= tiles
    assert 1 <= g <= 32 and (grouped or g == 1) and g * r <= max(tiles, r) and (g == 1 or r <= 8)
    assert kpr % kt == 0 and kpr > 0
    assert g * r * kpr >= L
    assert kpr <= -(-tiles // (g * r)) * kt


def test_decode_plan_fills_the_gpu():
    """Few heads get the widest clusters, and with a workspace several clusters per head
    (up to one wave of two CTAs per SM); many heads stay at one CTA per head."""
    assert gb.attn_debug_decode_plan(1, 8, 1 << 20, 128, 152, 16)["ranks"] == 16
    assert gb.attn_debug_decode_plan(1, 8, 1 << 20, 128, 152, 8)["ranks"] == 8
    assert gb.attn_debug_decode_plan(8, 32, 8192, 128, 152, 16)["ranks"] == 1  # 256 heads fill the wave
    assert gb.attn_debug_decode_plan(1, 64, 8192, 128, 152, 16)["ranks"] == 4  # 256 CTAs <= 304
    assert gb.attn_debug_decode_plan(1, 128, 8192, 128, 152, 16)["ranks"] == 2
    assert gb.attn_debug_decode_plan(64, 64, 4096, 64, 152, 16)["ranks"] == 1
    p = gb.attn_debug_decode_plan(1, 8, 1 << 20, 128, 152, 16, grouped=True)
    assert (p["ranks"], p["groups"]) == (2, 19)  # 8 heads x 19 clusters x 2 CTAs = 304: two per SM
    p = gb.attn_debug_decode_plan(1, 12, 1 << 18, 128, 152, 16, grouped=True)
    assert (p["ranks"], p["groups"]) == (2, 12)
    p = gb.attn_debug_decode_plan(1, 4, 1 << 20, 128, 152, 16, grouped=True)
    assert (p["ranks"], p["groups"]) == (8, 9)  # clusters of two would need 38 per head
    p = gb.attn_debug_decode_plan(1, 1, 100000, 64, 152, 16, grouped=True)
    assert (p["ranks"], p["groups"]) == (8, 32)
    assert gb.attn_debug_decode_plan(8, 32, 8192, 128, 152, 16, grouped=True)["groups"] == 1


def test_decode_plan_validation():
    with pytest.raises(gb.GbattnError):
        gb.attn_debug_decode_plan(1, 1, 128, 96, 152)
    with pytest.raises(gb.GbattnError):
        gb.attn_debug_decode_plan(1, 1, 128, 64, 152, 32)
    with pytest.raises(gb.GbattnError):
        gb.attn_debug_decode_plan(1, 1, 0, 64, 152)


@pytest.mark.parametrize("B,H,L,d,kind", [
    # 512 two-tile items (3.4 per SM): the single-tile kernel's 1024 items spread more evenly
    (4, 16, 2048, 64, 0), (2, 16, 4096, 64, 0), (4, 8, 4096, 64, 0), (2, 32, 2048, 64, 0),
    # 1024 or 256 two-tile items: the two-tile kernel
    (8, 16, 2048, 64, 1), (4, 16, 1024, 64, 1), (2, 16, 2048, 128, 1), (8, 16, 512, 128, 1),
])
def test_non_causal_plan_compares_whole_item_rounds(B, H, L, d, kind):
    """Non-causal items are all alike, so with enough items for the two-tile kernel the
    planner still compares the two kernels' busiest CTAs, in whole items (measured on
    GB300: these choices were the faster kernel)."""
    assert gb.attn_debug_plan(B, H, L, d, False, 152)["kind"] == kind


def test_causal_plan_with_many_items_stays_two_tile():
    for B, H, L, d in [(8, 32, 512, 128), (16, 16, 512, 128), (1, 32, 4096, 128), (8, 32, 512, 64)]:
        assert gb.attn_debug_plan(B, H, L, d, True, 152)["kind"] == 1
