"""CPU replay of the E4M3 prefill pair kernel's barrier protocol.

Restated from the kernel (tc_prefill_fp8_kernel): two CTAs, E (even: issues
the MMAs) and O (odd).  Per CTA: the producer copies its query rows into
buffer seg % 2 (after the commit that empties it two segments back) and, per
pair of pages, its page's codes and both pages' scales into raw stage
g % RS (after the converters have emptied it); the converters (CONV warps,
each arriving once) turn the query rows to f16 and write the rows' powers of
two (after every epilogue warp has read the ones of two segments back), and
per pair turn the raw page into f16 operand stage g % OS (after the commit
that freed it) and copy the scales into ring slot g % R (after the epilogue
warps have read it).  O's forwarder tells E when O's query rows and each of
O's operand stages are ready.  E's waiter counts the pairs whose two operand
stages are ready and whose accumulator buffer g % 2 is free; E's issuing
thread waits for both CTAs' query rows at each segment and for the count at
each pair; its MMAs complete in order, later, and each commit arrives on the
same barrier in both CTAs once every MMA issued before it has completed.
The epilogue warps of both CTAs read the powers of two at each segment and
per pair wait for the accumulator buffer and the scale slot, then free both.

Besides the barrier phases (a waiter must never fall two phases behind), the
replay tracks what each buffer holds: a converter's writes, the MMA's reads
of an operand stage and the epilogue's reads of the powers of two and the
scales must see the right pair's or segment's data.  Removing any of the
waits that guard a buffer's reuse makes some random schedule fail, except
the scale-slot wait, which the operand and accumulator waits already imply
for the kernel's ring depth.
"""

import random

import pytest

RS, OS, R = 3, 3, 8      # raw stages, operand stages, scale slots
ACC, QB = 2, 2           # accumulator buffers, query buffers
CONV, EPI = 2, 2         # converter and epilogue warps modelled per CTA


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
        assert self.phases <= phase + 1, f"{self.name}: waiter for phase {phase} overtaken ({self.phases})"
        return self.phases > phase


def roles(segments, drop=None, ring=R):
    """Generators for every role; each yields a predicate to wait on, or None.
    `drop` names one reuse wait to leave out (the check of the checker);
    `ring` is the number of scale slots."""
    R = ring
    bars = {}

    def bar(name, count=1):
        bars[name] = Barrier(name, count)

    for x in "EO":
        for s in range(RS):
            bar(f"raw_full{x}{s}"), bar(f"raw_empty{x}{s}", CONV)
        for s in range(OS):
            bar(f"op_full{x}{s}", CONV), bar(f"op_empty{x}{s}")
        for s in range(R):
            bar(f"sc_full{x}{s}", CONV), bar(f"sc_empty{x}{s}", EPI)
        for b in range(QB):
            bar(f"q_full{x}{b}"), bar(f"q_conv{x}{b}", CONV), bar(f"q_empty{x}{b}")
            bar(f"inv_free{x}{b}", EPI)
        for a in range(ACC):
            bar(f"acc_full{x}{a}")
    for s in range(OS):
        bar(f"op_peerE{s}")
    for b in range(QB):
        bar(f"q_peerE{b}")
    for a in range(ACC):
        bar(f"acc_emptyE{a}", 2 * EPI)
    # what each buffer holds: the pair or segment whose data was written last
    data = {f"{kind}{x}{i}": None for x in "EO" for kind, n in (("op", OS), ("ring", R), ("inv", QB))
            for i in range(n)}
    state = {"ready": 0, "issued": 0, "completed": 0, "commits": [], "mma_reads": []}
    total = sum(segments)
    copies = []

    def wait(name, phase):
        b = bars[name]
        return lambda: b.done(phase)

    def producer(x):
        gc = 0
        for seg, ng in enumerate(segments):
            if seg >= QB:
                yield wait(f"q_empty{x}{seg % QB}", seg // QB - 1)
            copies.append(bars[f"q_full{x}{seg % QB}"])
            for _ in range(ng):
                if gc >= RS:
                    yield wait(f"raw_empty{x}{gc % RS}", gc // RS - 1)
                copies.append(bars[f"raw_full{x}{gc % RS}"])
                gc += 1
                yield None

    def converter(x, cw):
        gc = 0
        for seg, ng in enumerate(segments):
            qb = seg % QB
            yield wait(f"q_full{x}{qb}", seg // QB)
            if seg >= QB and drop != "inv_free":
                yield wait(f"inv_free{x}{qb}", seg // QB - 1)
            data[f"inv{x}{qb}"] = seg  # this warp's rows' powers of two
            yield None
            bars[f"q_conv{x}{qb}"].arrive()
            for _ in range(ng):
                yield wait(f"raw_full{x}{gc % RS}", gc // RS)
                if gc >= OS and drop != "op_empty":
                    yield wait(f"op_empty{x}{gc % OS}", gc // OS - 1)
                if gc >= R and drop != "sc_empty":
                    yield wait(f"sc_empty{x}{gc % R}", gc // R - 1)
                data[f"op{x}{gc % OS}"] = gc
                data[f"ring{x}{gc % R}"] = gc
                yield None
                for name in (f"op_full{x}{gc % OS}", f"raw_empty{x}{gc % RS}", f"sc_full{x}{gc % R}"):
                    bars[name].arrive()
                gc += 1

    def forwarder():
        gc = 0
        for seg, ng in enumerate(segments):
            yield wait(f"q_convO{seg % QB}", seg // QB)
            bars[f"q_peerE{seg % QB}"].arrive()
            for _ in range(ng):
                yield wait(f"op_fullO{gc % OS}", gc // OS)
                bars[f"op_peerE{gc % OS}"].arrive()
                gc += 1

    def waiter():
        for gc in range(total):
            yield wait(f"op_fullE{gc % OS}", gc // OS)
            yield wait(f"op_peerE{gc % OS}", gc // OS)
            if gc >= ACC and drop != "acc_empty":
                yield wait(f"acc_emptyE{gc % ACC}", gc // ACC - 1)
            state["ready"] = gc + 1

    def issuer():
        gc = 0
        for seg, ng in enumerate(segments):
            yield wait(f"q_convE{seg % QB}", seg // QB)
            yield wait(f"q_peerE{seg % QB}", seg // QB)
            for _ in range(ng):
                yield lambda g=gc: state["ready"] >= g + 1
                state["issued"] += 1
                # the MMA reads both CTAs' operand stages until it completes
                state["mma_reads"].append((state["issued"], gc))
                state["commits"].append((state["issued"], [f"op_empty{x}{gc % OS}" for x in "EO"]))
                state["commits"].append((state["issued"], [f"acc_full{x}{gc % ACC}" for x in "EO"]))
                gc += 1
            state["commits"].append((state["issued"], [f"q_empty{x}{seg % QB}" for x in "EO"]))

    def epilogue(x):
        gc = 0
        for seg, ng in enumerate(segments):
            qb = seg % QB
            yield wait(f"q_conv{x}{qb}", seg // QB)
            assert data[f"inv{x}{qb}"] == seg, f"powers of two of segment {seg} overwritten"
            bars[f"inv_free{x}{qb}"].arrive()
            for _ in range(ng):
                yield wait(f"acc_full{x}{gc % ACC}", gc // ACC)
                yield wait(f"sc_full{x}{gc % R}", gc // R)
                yield None
                assert data[f"ring{x}{gc % R}"] == gc, f"scales of pair {gc} overwritten"
                bars[f"acc_emptyE{gc % ACC}"].arrive()
                bars[f"sc_empty{x}{gc % R}"].arrive()
                gc += 1

    gens = [producer("E"), producer("O"), forwarder(), waiter(), issuer()]
    gens += [converter(x, cw) for x in "EO" for cw in range(CONV)]
    gens += [epilogue(x) for x in "EO" for _ in range(EPI)]
    return gens, bars, state, copies, data


def run(segments, rng, drop=None, ring=R):
    gens, bars, state, copies, data = roles(segments, drop, ring)
    waiting = [None] * len(gens)
    live = list(range(len(gens)))
    steps = 0
    while live:
        steps += 1
        assert steps < 400000, "no progress (deadlock)"
        r = rng.random()
        if copies and r < 0.3:
            copies.pop(rng.randrange(len(copies))).arrive()  # copies land in any order
            continue
        if state["completed"] < state["issued"] and r < 0.5:
            # an MMA completes: it read the operand stages of its pair until now
            done = state["completed"] + 1
            for n, g in state["mma_reads"]:
                if n == done:
                    for x in "EO":
                        assert data[f"op{x}{g % OS}"] == g, f"operands of pair {g} overwritten"
            state["completed"] = done
        while state["commits"] and state["commits"][0][0] <= state["completed"]:
            for name in state["commits"].pop(0)[1]:
                bars[name].arrive()
        runnable = [i for i in live if waiting[i] is None or waiting[i]()]
        if not runnable:
            if not copies and state["completed"] == state["issued"] and not state["commits"]:
                raise AssertionError("deadlock: " + repr(live))
            continue
        i = rng.choice(runnable)
        try:
            waiting[i] = next(gens[i])
        except StopIteration:
            live.remove(i)
    return state


@pytest.mark.parametrize("seed", range(6))
def test_fp8_pair_protocol_random_schedules(seed):
    rng = random.Random(seed)
    for _ in range(20):
        segments = [rng.randint(1, 12) for _ in range(rng.randint(1, 6))]
        st = run(segments, rng)
        assert st["issued"] == sum(segments) and st["ready"] == sum(segments)


def fails(drop, ring=R, tries=300):
    rng = random.Random(7)
    for _ in range(tries):
        segments = [rng.randint(1, 12) for _ in range(rng.randint(2, 6))]
        try:
            run(segments, rng, drop, ring)
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("drop", ["inv_free", "op_empty", "acc_empty"])
def test_each_reuse_wait_is_needed(drop):
    """Without one of the waits that guard a buffer's reuse, some schedule
    reads overwritten data or overtakes a barrier phase."""
    assert fails(drop), f"no schedule noticed the missing {drop} wait"


def test_scale_slot_wait_is_implied_by_a_deep_ring():
    """A converter writes scale slot g % R only after the MMA of pair g - OS
    has completed, which needed the epilogue to free the accumulator buffer of
    pair g - OS - ACC after reading that pair's scales; so with R >= OS + ACC
    slots the slot's last reader is done already and the kernel's scale-slot
    wait never holds anything up (it stays, at the cost of one non-blocking
    test).  With one slot fewer the wait is needed."""
    assert R >= OS + ACC
    assert not fails("sc_empty", ring=R, tries=100)
    assert not fails("sc_empty", ring=OS + ACC, tries=100)
    rng = random.Random(1)
    for _ in range(10):  # the protocol itself is sound with a shallower ring
        run([rng.randint(1, 12) for _ in range(rng.randint(1, 5))], rng, ring=OS + ACC - 1)
    assert fails("sc_empty", ring=OS + ACC - 1)
