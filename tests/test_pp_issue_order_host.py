"""Host-side model (no GPU) of the two-tile forward kernel's MMA issue order and its ring,
to check the one parity test the issuer makes ahead of its own consumption.

The issuer (attn_fwd_pp.cuh, PPIssuer) consumes ring positions in the producer's load
order, item by item K_0, V_0, K_1, V_1, ... for the n1 key tiles of an item, and issues
per item  QK0_0, QK1_0, then for each key tile j:  PV0_j, QK0_{j+1}, PV1_j, QK1_{j+1}.
When slot 0 has issued its last PV of an item, the next item's QK0_0 becomes "pending" and
is issued from inside the issuer's later waits as soon as a parity test of the FULL barrier
of its K_0 stage (ring position side_base) succeeds.  An mbarrier parity test is only
unambiguous if the barrier is at most one phase behind: the stage's previous use, position
side_base - NST, must already have completed -- which holds once the issuer has consumed
it.  Otherwise (that position not yet landed) the test reports the phase two back as done
and the QK would run on a stage still being filled.

The model replays the issue order and checks that invariant at the first moment the
issuer polls.  It holds for every item the kernel's decoding produces (pp_decode: causal
n0 = 2qb + 1, n1 = min(2qb + 2, nQ); otherwise n0 = n1 = nQ), and fails for items whose
slot 1 needs three or more key tiles beyond slot 0's -- the (i, nQ - 1 - i) pairing of a
removed experiment, whose launch ended in a GPU fault.
"""
import itertools
import math
import random

import pytest


def ring_stages(d: int) -> int:
    """NST of PPCfg: 224 KB of tiles, two Q buffers and one O staging tile of 128 x d fp16,
    at most 12 stages."""
    tile = 128 * d * 2
    return min(12, (224 * 1024 - 3 * tile) // tile)


def first_polls_are_safe(items, nst):
    """Replay the issue order of `items` ((n0, n1) pairs, n1 >= n0 >= 1) on one CTA; return
    a list of (item index, side_base, previous use, consumed?) for every pending QK0_0, at
    the first wait after it becomes pending."""
    consumed = set()
    base = 0
    out = []
    pending_check = None  # (il, side_base) to check at the next wait

    def wait():  # every wait polls the pending QK's stage first
        nonlocal pending_check
        if pending_check is not None:
            il, sb = pending_check
            prev = sb - nst
            out.append((il, sb, prev, prev < 0 or prev in consumed))
            pending_check = None

    def qk(j, item_base):
        wait()
        consumed.add(item_base + 2 * j)

    def pv(j):
        wait()
        consumed.add(base + 2 * j + 1)

    qk(0, 0)
    qk(0, 0)  # QK1_0 (same K tile)
    for il, (n0, n1) in enumerate(items):
        has_next = il + 1 < len(items)
        next_base = base + 2 * n1
        side = False
        for j in range(n1):
            if j < n0:
                pv(j)
                if j + 1 < n0:
                    qk(j + 1, base)
                elif has_next:
                    side = True
                    pending_check = (il + 1, next_base)
            pv(j)
            if j + 1 < n1:
                qk(j + 1, base)
        if not has_next:
            break
        if side:
            qk(0, next_base)  # the pending QK0_0, at the latest here
        qk(0, next_base)      # QK1_0
        base = next_base
    return out


def decode(nQ, qb, causal):
    return (2 * qb + 1, min(2 * qb + 2, nQ)) if causal else (nQ, nQ)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("L", [256, 300, 512, 640, 1024, 2048, 4096])
@pytest.mark.parametrize("causal", [True, False])
def test_retained_items_poll_safely(d, L, causal):
    """Every sequence of the kernel's own items (all orders a schedule can give a CTA)."""
    nst = ring_stages(d)
    nQ, nQB = math.ceil(L / 128), math.ceil(L / 256)
    kinds = [decode(nQ, qb, causal) for qb in range(nQB)]
    rng = random.Random(L * d + causal)
    seqs = [list(p) for p in itertools.product(kinds, repeat=min(3, len(kinds)))]
    seqs += [[rng.choice(kinds) for _ in range(rng.randint(2, 12))] for _ in range(200)]
    for seq in seqs:
        for il, sb, prev, ok in first_polls_are_safe(seq, nst):
            assert ok, f"{seq}: item {il}'s K_0 stage polled before position {prev} was consumed"


def test_paired_tiles_would_poll_too_early():
    """The removed pairing of query tiles (i, nQ - 1 - i) at L = 512 (nQ = 4), head_dim 128
    (4 ring stages): item (0, 3) has n0 = 1, n1 = 4, and the next item's K_0 stage is polled
    while its previous use, K_2 of the current item, has not been consumed (possibly not
    even loaded)."""
    nst = ring_stages(128)
    assert nst == 4
    paired = [(1, 4), (2, 3)]  # (0, 3) and (1, 2) as (n0, n1)
    bad = [r for r in first_polls_are_safe(paired + paired, nst) if not r[3]]
    assert bad, "the model should show the unsafe poll"
    il, sb, prev, _ = bad[0]
    assert (il, sb, prev) == (1, 8, 4)
