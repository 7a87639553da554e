"""CPU replay of the prefill top-k kernel's filter against brute force.

The kernel keeps, per (token, head) row, the pins (the first n_sink and the
last n_window visible blocks) and the highest-scoring free blocks, ties to
the lower block id, blocks whose page was out of range (-inf) left out.  It
seeds its running list with the pins, then passes the row's blocks 512 at a
time (lane l holds blocks g0 + 32 i + l) through a bound on 32-bit coarse
keys: the KMAX-th largest lane maximum until the list is full, the list's
last key after.  Only blocks at or above the bound are merged.  This replays
those steps (restated from the kernel) on rows built to stress them (ties,
-0, -inf, sorted rows that overflow the candidate space, short rows) and
checks every row against a brute-force sort of all its keys.
"""

import numpy as np
import pytest

GROUP, LANES, PER_LANE = 512, 32, 16
NEG_INF = np.float32(-np.inf)


def order_bits(x):
    """32-bit key that orders floats (-0 taken as +0)."""
    u = int((np.float32(x) + np.float32(0.0)).view(np.uint32))
    return (~u & 0xFFFFFFFF) if u & 0x80000000 else (u | 0x80000000)


def pack(score, j, pinned):
    s = np.float32(score)
    s = np.float32(0.0) if s == 0 else s
    rid = 0x7FFFFFFF - j
    if pinned:
        return (1 << 63) | (rid << 32) | int(s.view(np.uint32))
    return (order_bits(s) << 31) | rid


def coarse(key):
    if key == 0:
        return 0
    return 0xFFFFFFFF if key >> 63 else (key >> 31) & 0xFFFFFFFF


def top(keys, width):
    out = sorted((x for x in set(keys) if x), reverse=True)[:width]
    return out + [0] * (width - len(out))


def kernel_row(scores, nb, k, n_sink, n_window, kmax):
    """The kernel's steps for one row; returns its descending key list (k)."""
    ns = min(n_sink, nb)
    w0 = max(ns, nb - n_window)
    npin = ns + (nb - w0)
    pins = []
    for lane in range(npin):
        j = lane if lane < ns else w0 + (lane - ns)
        pins.append(0 if scores[j] == NEG_INF else pack(scores[j], j, True))
    run = top(pins, kmax)  # in id order already, or compacted by a merge
    cap = kmax * PER_LANE
    floor = order_bits(NEG_INF) + 1
    for g0 in range(0, nb, GROUP):
        js = np.arange(g0, g0 + GROUP)
        vals = [scores[j] if j < nb else NEG_INF for j in js]
        ck = [order_bits(v) for v in vals]
        tail = run[kmax - 1]
        lane_bound = 0
        if tail == 0:
            lane_max = [max(ck[LANES * i + lane] for i in range(PER_LANE)) for lane in range(LANES)]
            lane_bound = sorted(lane_max, reverse=True)[kmax - 1]
        bound = max(lane_bound, coarse(tail), floor)
        cand = [(int(j), v) for j, v, c in zip(js, vals, ck) if c >= bound]
        if len(cand) <= cap:
            keys = [0 if (j < ns or j >= w0) else pack(v, j, False) for j, v in cand]
        else:  # ties overflow the candidate space: every free block of the group
            keys = [pack(v, int(j), False) for j, v in zip(js, vals)
                    if j < nb and ns <= j < w0 and v != NEG_INF]
        run = top(run + keys, kmax)
    return run[:k]


def brute_row(scores, nb, k, n_sink, n_window):
    keys = []
    for j in range(nb):
        if scores[j] == NEG_INF:
            continue
        keys.append(pack(scores[j], j, j < n_sink or j >= nb - n_window))
    return top(keys, k)


def random_row(rng, kind, nb):
    if kind == "normal":
        s = rng.standard_normal(nb).astype(np.float32)
    elif kind == "ties":
        s = rng.integers(-3, 4, nb).astype(np.float32)
    elif kind == "ascending":  # the best blocks last: candidates pile up group after group
        s = np.arange(nb, dtype=np.float32)
    elif kind == "descending":
        s = -np.arange(nb, dtype=np.float32)
    else:  # "const": every block ties
        s = np.full(nb, 1.5, dtype=np.float32)
    zeros = rng.random(nb) < 0.05
    s[zeros] = np.where(rng.random(zeros.sum()) < 0.5, np.float32(0.0), np.float32(-0.0))
    s[rng.random(nb) < 0.03] = NEG_INF
    return s


@pytest.mark.parametrize("kmax", [16, 32])
@pytest.mark.parametrize("kind", ["normal", "ties", "ascending", "descending", "const"])
def test_filter_matches_brute_force(kmax, kind):
    rng = np.random.default_rng(hash((kmax, kind)) % 2**32)
    for _ in range(12):
        nb = int(rng.choice([0, 1, 3, 17, 200, 511, 512, 513, 1024, 1040, 1700]))
        k = int(rng.integers(1, kmax + 1))
        n_sink = int(rng.integers(0, k + 1))
        n_window = int(rng.integers(0, k - n_sink + 1))
        s = random_row(rng, kind, nb)
        got = kernel_row(s, nb, k, n_sink, n_window, kmax)
        assert got == brute_row(s, nb, k, n_sink, n_window), (kind, nb, k, n_sink, n_window)


def test_bound_prunes_on_long_rows():
    """On a long row of random scores the bound keeps the merges small."""
    rng = np.random.default_rng(5)
    nb, kmax = 1024, 16
    s = rng.standard_normal(nb).astype(np.float32)
    ns, w0 = 1, nb - 2
    run = top([pack(s[0], 0, True), pack(s[nb - 2], nb - 2, True), pack(s[nb - 1], nb - 1, True)], kmax)
    sizes = []
    for g0 in range(0, nb, GROUP):
        ck = [order_bits(s[j]) for j in range(g0, g0 + GROUP)]
        tail = run[kmax - 1]
        lane_bound = 0
        if tail == 0:
            lane_max = [max(ck[LANES * i + lane] for i in range(PER_LANE)) for lane in range(LANES)]
            lane_bound = sorted(lane_max, reverse=True)[kmax - 1]
        bound = max(lane_bound, coarse(tail))
        cand = [g0 + i for i, c in enumerate(ck) if c >= bound]
        sizes.append(len(cand))
        run = top(run + [pack(s[j], j, False) for j in cand if ns <= j < w0], kmax)
    assert sizes[0] <= 64 and sizes[1] <= 32, sizes
