"""CPU replay of the bf16 prefill pair kernel's barrier protocol.

Restated from the kernel (tc_prefill_pair_kernel): two CTAs, E (even: issues
the MMAs) and O (odd).  Per tile segment each CTA's producer loads its query
rows into buffer seg % 2 (after the commit that empties it two segments
back), and per pair of pages its page into stage g % S (after the commit
that emptied the stage S pairs back).  O's forwarder waits for O's query
rows and each of O's stages and arrives on E's "peer" barriers.  E's waiter
waits, per pair, for E's stage, the peer stage and the accumulator buffer
g % 2 (freed by every epilogue warp of both CTAs two pairs back) and raises
a counter.  E's issuing thread waits for both CTAs' query rows at each
segment and for the counter at each pair; its MMAs complete in order, later,
and each commit arrives on the same barrier in both CTAs once every MMA
issued before it has completed.  The epilogue warps of both CTAs wait for
each pair's accumulator buffer and arrive on E's accumulator-empty barrier.

An mbarrier wait is on a phase's parity, so a waiter must never fall two
phases behind the barrier it waits on (the parity would then say "not
complete" forever).  Random schedules check that no wait is ever overtaken
that way and that every role finishes.
"""

import random

import pytest

S = 5          # page stages a CTA (kP2Stages)
ACC = 2        # accumulator buffers (kP2AccBufs)
QB = 2         # query buffers (kP2QBufs)
EPI = 2        # epilogue warps modelled per CTA (the kernel's 8 behave alike)


class Barrier:
    def __init__(self, name, count):
        self.name, self.count, self.arrived, self.phases = name, count, 0, 0

    def arrive(self):
        self.arrived += 1
        assert self.arrived <= self.count, self.name
        if self.arrived == self.count:
            self.arrived = 0
            self.phases += 1

    def done(self, phase):
        """Phase `phase` (0-based) has completed; a parity wait would see it."""
        assert self.phases <= phase + 1, f"{self.name}: waiter for phase {phase} overtaken ({self.phases})"
        return self.phases > phase


def roles(segments):
    """Generators for every role; each yields a predicate to wait on, or None to
    yield the scheduler."""
    bars = {}

    def bar(name, count=1):
        if name not in bars:
            bars[name] = Barrier(name, count)
        return bars[name]

    for x in "EO":
        for s in range(S):
            bar(f"k_full{x}{s}"), bar(f"k_empty{x}{s}")
        for b in range(QB):
            bar(f"q_full{x}{b}"), bar(f"q_empty{x}{b}")
        for a in range(ACC):
            bar(f"acc_full{x}{a}")
    for s in range(S):
        bar(f"k_peerE{s}")
    for b in range(QB):
        bar(f"q_peerE{b}")
    for a in range(ACC):
        bar(f"acc_emptyE{a}", 2 * EPI)
    state = {"ready": 0, "issued": 0, "completed": 0, "commits": []}
    total = sum(segments)
    copies = []  # in-flight copies: barriers to arrive on when they land

    def producer(x):
        gc = 0
        for seg, ng in enumerate(segments):
            if seg >= QB:
                b = bars[f"q_empty{x}{seg % QB}"]
                yield lambda b=b, ph=seg // QB - 1: b.done(ph)
            copies.append(bars[f"q_full{x}{seg % QB}"])
            for _ in range(ng):
                if gc >= S:
                    b = bars[f"k_empty{x}{gc % S}"]
                    yield lambda b=b, ph=gc // S - 1: b.done(ph)
                copies.append(bars[f"k_full{x}{gc % S}"])
                gc += 1
                yield None

    def forwarder():
        gc = 0
        for seg, ng in enumerate(segments):
            b = bars[f"q_fullO{seg % QB}"]
            yield lambda b=b, ph=seg // QB: b.done(ph)
            bars[f"q_peerE{seg % QB}"].arrive()
            for _ in range(ng):
                b = bars[f"k_fullO{gc % S}"]
                yield lambda b=b, ph=gc // S: b.done(ph)
                bars[f"k_peerE{gc % S}"].arrive()
                gc += 1

    def waiter():
        for gc in range(total):
            for name in (f"k_fullE{gc % S}", f"k_peerE{gc % S}"):
                b = bars[name]
                yield lambda b=b, ph=gc // S: b.done(ph)
            if gc >= ACC:
                b = bars[f"acc_emptyE{gc % ACC}"]
                yield lambda b=b, ph=gc // ACC - 1: b.done(ph)
            state["ready"] = gc + 1

    def issuer():
        gc = 0
        for seg, ng in enumerate(segments):
            for name in (f"q_fullE{seg % QB}", f"q_peerE{seg % QB}"):
                b = bars[name]
                yield lambda b=b, ph=seg // QB: b.done(ph)
            for _ in range(ng):
                yield lambda g=gc: state["ready"] >= g + 1
                state["issued"] += 1
                # commits fire when every MMA issued before them has completed
                state["commits"].append((state["issued"], [f"k_empty{x}{gc % S}" for x in "EO"]))
                state["commits"].append((state["issued"], [f"acc_full{x}{gc % ACC}" for x in "EO"]))
                gc += 1
            state["commits"].append((state["issued"], [f"q_empty{x}{seg % QB}" for x in "EO"]))

    def epilogue(x):
        for gc in range(total):
            b = bars[f"acc_full{x}{gc % ACC}"]
            yield lambda b=b, ph=gc // ACC: b.done(ph)
            bars[f"acc_emptyE{gc % ACC}"].arrive()

    gens = [producer("E"), producer("O"), forwarder(), waiter(), issuer()]
    gens += [epilogue(x) for x in "EO" for _ in range(EPI)]
    return gens, bars, state, copies


def run(segments, rng):
    gens, bars, state, copies = roles(segments)
    waiting = [None] * len(gens)
    live = list(range(len(gens)))
    steps = 0
    while live:
        steps += 1
        assert steps < 200000, "no progress (deadlock)"
        # asynchronous work: a copy lands, an MMA completes, a commit fires
        r = rng.random()
        if copies and r < 0.3:
            copies.pop(rng.randrange(len(copies))).arrive()  # copies land in any order
            continue
        if state["completed"] < state["issued"] and r < 0.5:
            state["completed"] += 1
        while state["commits"] and state["commits"][0][0] <= state["completed"]:
            for name in state["commits"].pop(0)[1]:
                bars[name].arrive()
        runnable = [i for i in live if waiting[i] is None or waiting[i]()]
        if not runnable:
            if not copies and state["completed"] == state["issued"] and not state["commits"]:
                raise AssertionError("deadlock: " + repr([i for i in live]))
            continue
        i = rng.choice(runnable)
        try:
            waiting[i] = next(gens[i])
        except StopIteration:
            live.remove(i)
    return state


@pytest.mark.parametrize("seed", range(8))
def test_pair_protocol_random_schedules(seed):
    rng = random.Random(seed)
    for _ in range(25):
        segments = [rng.randint(1, 12) for _ in range(rng.randint(1, 6))]
        st = run(segments, rng)
        assert st["issued"] == sum(segments) and st["ready"] == sum(segments)


def test_parity_check_catches_an_overtaken_wait():
    """The checker itself: a barrier two phases ahead of its waiter fails."""
    b = Barrier("x", 1)
    b.arrive()
    b.arrive()
    with pytest.raises(AssertionError):
        b.done(0)
