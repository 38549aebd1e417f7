"""Host-side model (no GPU) of the backward dQ kernel's barrier protocol between its MMA
thread, the tensor pipe and the elementwise threads (attn_bwd.cuh, attn_bwd_dq_kernel).

Per step s (global step g) of an item the tensor pipe runs S(g) = Q K^T into S buffer g&1,
dP(g) = dO V^T into the dP columns and dQ += dS(g) K.  The elementwise threads read S(g)
(for P) and dP(g), write dS(g) (fp16) over dP(g) and signal DSFULL.  The MMA thread
issues, per item, S(g), dP(g), S(g+1), then per step: dQ(g) once DSFULL(g) is complete,
then dP(g+1) into the columns dQ(g) has just read, then S(g+2) into S buffer g&1.

A variant that was measured and not kept writes dS(g) over S(g) instead, hands the dP
columns back as soon as they are read (DPREAD), and issues dP(g+1) once DPREAD(g) is
complete, before waiting for DSFULL(g).

An mbarrier parity wait is only unambiguous while the barrier is at most one phase away
from the waited phase: waiting for phase k, the barrier must have completed k or k+1
phases; at k+2 the wait never returns.  Arrivals carry no phase either: an arrival meant
for phase k must land while the barrier has completed exactly k phases.  The model runs
the three roles under randomly skewed schedules (the tensor pipe and each role stalled or
racing at random) and checks both rules at every scheduling step, plus every tensor-memory
read and overwrite (a region is only overwritten once its content has been consumed).

In the kernel, dS(g+1) needs dP(g+1), which is issued only after the wait for dS(g), so
one DSFULL barrier suffices.  In the variant dP(g+1) is issued before that wait, so the
elementwise threads can finish dS(g+1) before the wait looks, and one barrier can then
be two phases ahead of it.  The variant needs one DSFULL barrier per step parity.  The
model shows that the kernel's protocol and the two-barrier variant hold, and that it
finds the gap in the one-barrier variant.
"""
import random

import pytest


class Bar:
    def __init__(self, count):
        self.count = count
        self.arrived = 0
        self.done = 0  # completed phases


class Model:
    """variant: "kernel" (the protocol above), "early_dp" (the variant, two DSFULL
    barriers) or "early_dp_one_barrier"."""

    def __init__(self, items, nthreads, variant, rng):
        self.items = items
        self.nt = nthreads
        self.early = variant != "kernel"
        self.two = variant == "early_dp"
        self.rng = rng
        self.bars = {"SFULL0": Bar(1), "SFULL1": Bar(1), "DPFULL": Bar(1), "IDONE": Bar(1),
                     "DSFULL0": Bar(nthreads), "DSFULL1": Bar(nthreads), "DPREAD": Bar(nthreads)}
        # tensor memory, per thread lane: (content tag, consumed?)
        self.tmem = {}
        for t in range(nthreads):
            for r in ("S0", "S1", "DP", "DQ"):
                self.tmem[(r, t)] = (None, True)
        self.pipe = []  # in-order queue of ("mma", fn) / ("commit", bar, phase)
        self.errors = []

    # ---- barrier rules
    def arrive(self, name, phase):
        b = self.bars[name]
        if b.done != phase:
            self.errors.append(f"arrival for phase {phase} on {name} at {b.done} completed phases")
        b.arrived += 1
        if b.arrived == b.count:
            b.arrived = 0
            b.done += 1

    def check_wait(self, name, phase):
        d = self.bars[name].done
        if d not in (phase, phase + 1):
            self.errors.append(f"wait for phase {phase} on {name} at {d} completed phases")
            return False
        return True

    # ---- tensor memory rules
    def write(self, region, t, tag, rmw_expect=None):
        old, consumed = self.tmem[(region, t)]
        if rmw_expect is not None:
            if old != rmw_expect:
                self.errors.append(f"{tag} accumulates onto {old} in {region}[{t}], expected {rmw_expect}")
        elif not consumed:
            self.errors.append(f"{tag} overwrites unconsumed {old} in {region}[{t}]")
        self.tmem[(region, t)] = (tag, False)

    def read(self, region, t, tag):
        old, _ = self.tmem[(region, t)]
        if old != tag:
            self.errors.append(f"read of {tag} in {region}[{t}] found {old}")
        self.tmem[(region, t)] = (old, True)

    def ds_bar(self, g):
        return (f"DSFULL{g & 1}", g >> 1) if self.two else ("DSFULL0", g)

    # ---- roles (generators yielding ("wait", bar, phase) or None for a plain step)
    def mma_thread(self):
        g = 0

        def issue_s(gg):
            def run():
                for t in range(self.nt):
                    self.write(f"S{gg & 1}", t, ("S", gg))
            self.pipe.append(("mma", run))
            self.pipe.append(("commit", f"SFULL{gg & 1}", gg >> 1))

        def issue_dp(gg):
            def run():
                for t in range(self.nt):
                    self.write("DP", t, ("dP", gg))
            self.pipe.append(("mma", run))
            self.pipe.append(("commit", "DPFULL", gg))

        def issue_dq(gg, first):
            def run():
                for t in range(self.nt):
                    self.read(f"S{gg & 1}" if self.early else "DP", t, ("dS", gg))
                    self.write("DQ", t, ("dQ", gg), None if first else ("dQ", gg - 1))
            self.pipe.append(("mma", run))

        for it, n in enumerate(self.items):
            issue_s(g)
            yield None
            issue_dp(g)
            yield None
            if n > 1:
                issue_s(g + 1)
                yield None
            for s in range(n):
                if self.early and s + 1 < n:
                    yield ("wait", "DPREAD", g)
                    issue_dp(g + 1)
                    yield None
                yield ("wait",) + self.ds_bar(g)
                issue_dq(g, s == 0)
                yield None
                if not self.early and s + 1 < n:
                    issue_dp(g + 1)
                    yield None
                if s + 2 < n:
                    issue_s(g + 2)
                    yield None
                g += 1
            self.pipe.append(("commit", "IDONE", it))
            yield None

    def elementwise_thread(self, t):
        g = 0
        for it, n in enumerate(self.items):
            for s in range(n):
                yield ("wait", f"SFULL{g & 1}", g >> 1)
                self.read(f"S{g & 1}", t, ("S", g))
                yield None
                yield ("wait", "DPFULL", g)
                self.read("DP", t, ("dP", g))
                if self.early:
                    self.arrive("DPREAD", g)
                yield None
                self.write(f"S{g & 1}" if self.early else "DP", t, ("dS", g))
                self.arrive(*self.ds_bar(g))
                yield None
                g += 1
            yield ("wait", "IDONE", it)
            self.read("DQ", t, ("dQ", g - 1))
            yield None

    def run(self, max_steps=200000):
        roles = {"mma": self.mma_thread()}
        for t in range(self.nt):
            roles[f"t{t}"] = self.elementwise_thread(t)
        pending = {k: None for k in roles}  # current wait of each role
        finished = set()
        names = list(roles) + ["pipe"]
        weights = {}

        def reweight():
            for k in names:
                weights[k] = 10 ** self.rng.uniform(-3, 0)

        reweight()
        for step in range(max_steps):
            if step % 37 == 0:
                reweight()
            for k, w in pending.items():
                if w is not None and k not in finished:
                    self.check_wait(w[1], w[2])
            runnable = []
            for k in roles:
                if k in finished:
                    continue
                w = pending[k]
                if w is None or self.bars[w[1]].done >= w[2] + 1:
                    runnable.append(k)
            if self.pipe:
                runnable.append("pipe")
            if not runnable:
                return len(finished) == len(roles)
            k = self.rng.choices(runnable, [weights[x] for x in runnable])[0]
            if k == "pipe":
                op = self.pipe.pop(0)
                if op[0] == "mma":
                    op[1]()
                else:
                    self.arrive(op[1], op[2])
                continue
            try:
                pending[k] = next(roles[k])
            except StopIteration:
                finished.add(k)
                pending[k] = None
        return False


def dq_items(B, H, L, causal):
    """Step counts of the dQ kernel's items in list order (query tile qt of a head sees key
    tiles 0..qt when causal), longest first as the kernel walks them."""
    n = (L + 127) // 128
    out = []
    for grp in range(n):
        qt = n - 1 - grp if causal else grp
        out += [qt + 1 if causal else n] * (B * H)
    return out


def run_many(variant, seeds, nthreads=3):
    bad = []
    for seed in seeds:
        rng = random.Random(seed)
        # one CTA's items: a mix of 1..4-step items as in an 8x32x512 causal launch
        items = [rng.choice([1, 2, 3, 4]) for _ in range(rng.randint(2, 7))]
        m = Model(items, nthreads, variant, rng)
        ok = m.run()
        if m.errors or not ok:
            bad.append((seed, items, m.errors[:3], ok))
    return bad


def test_item_lists_match_the_kernel_decoding():
    assert dq_items(1, 1, 512, True) == [4, 3, 2, 1]
    assert dq_items(2, 1, 300, False) == [3] * 6
    assert sorted(set(dq_items(8, 32, 512, True))) == [1, 2, 3, 4]


def test_kernel_protocol_holds():
    bad = run_many("kernel", range(300))
    assert not bad, bad[:2]


def test_early_dp_variant_with_two_dsfull_barriers_holds():
    bad = run_many("early_dp", range(300))
    assert not bad, bad[:2]


def test_early_dp_variant_with_one_dsfull_barrier_is_caught():
    # the wait can fall two phases behind: the model must find it
    bad = run_many("early_dp_one_barrier", range(300))
    assert bad, "the model did not find the two-phase gap of a single DSFULL barrier"
    assert any("DSFULL" in e for _, _, errs, _ in bad for e in errs)


@pytest.mark.parametrize("variant", ["kernel", "early_dp"])
@pytest.mark.parametrize("items", [[1], [4], [1, 1, 1], [4, 1, 4, 1], [2, 3, 1, 4, 2]])
def test_every_role_finishes(items, variant):
    for seed in range(20):
        m = Model(items, 2, variant, random.Random(seed))
        assert m.run(), (items, seed)
        assert not m.errors, m.errors[:3]
