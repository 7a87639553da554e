"""CPU replay of the prefill top-k kernel's filter against brute force.

The kernel keeps, per (token, head) row, the pins (the first n_sink and the
last n_window visible blocks) and the highest-scoring free blocks, ties to
the lower block id, blocks whose page was out of range (-inf) left out.  It
seeds its running list with the pins, then reads the row's blocks 1024 at a
time (lane l holds blocks g0 + 128 i + 4 l + e, i < 8, e < 4) and keeps only
those whose fp32 score is at or above one bound: the KMAX-th largest lane
maximum while the list is not full, the score of the list's last key after
(+inf when that key is a pin), and never -inf.  Up to 64 candidates are
merged; a group with more (ties) merges all its free blocks.  This replays
those steps (restated from the kernel) on rows built to stress them (ties,
-0, -inf, sorted rows, short rows, pins that fill the list) and checks every
row against a brute-force sort of all its keys.
"""

import numpy as np
import pytest

GROUP, LANES, PER_LANE, CAP = 1024, 32, 32, 64
NEG_INF = np.float32(-np.inf)
FLT_LOWEST = np.float32(-3.402823466e38)


def lane_of(j_in_group):
    """Lane holding block g0 + j of a group (16-byte loads: 4 blocks a lane, 128 a row of lanes)."""
    return (j_in_group % 128) // 4


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


def tail_bound(key):
    if key == 0:
        return NEG_INF
    if key >> 63:
        return np.float32(np.inf)
    o = (key >> 31) & 0xFFFFFFFF
    u = (o & 0x7FFFFFFF) if o & 0x80000000 else (~o & 0xFFFFFFFF)
    return np.uint32(u).view(np.float32)


def group_bound(vals, kmax):
    """kmax 16: the 16th largest lane maximum; 32: the 32nd largest of the lane
    maxima and second maxima."""
    per_lane = [[] for _ in range(LANES)]
    for off, v in enumerate(vals):
        per_lane[lane_of(off)].append(v)
    take = 1 if kmax == 16 else 2
    pool = [x for lane in per_lane for x in sorted(lane, reverse=True)[:take]]
    return sorted(pool, reverse=True)[kmax - 1]


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
    for g0 in range(0, nb, GROUP):
        js = np.arange(g0, g0 + GROUP)
        vals = np.array([scores[j] if j < nb else NEG_INF for j in js], dtype=np.float32)
        tail = run[kmax - 1]
        if tail == 0:
            bound = group_bound(vals, kmax)
        else:
            bound = tail_bound(tail)
        bound = max(np.float32(bound), FLT_LOWEST)
        cand = [(int(j), v) for j, v in zip(js, vals) if v >= bound]
        if len(cand) <= CAP:
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


def test_pins_that_fill_the_list_admit_no_free_block():
    s = np.random.default_rng(9).standard_normal(300).astype(np.float32)
    got = kernel_row(s, 300, 16, 8, 8, 16)
    assert got == brute_row(s, 300, 16, 8, 8)
    assert all(key >> 63 for key in got)


def test_bound_prunes_on_long_rows():
    """On a row of random scores the bound leaves a few dozen candidates."""
    rng = np.random.default_rng(5)
    sizes = []
    for kmax in (16, 32):
        for _ in range(20):
            s = rng.standard_normal(GROUP).astype(np.float32)
            bound = group_bound(s, kmax)
            sizes.append(int((s >= bound).sum()))
            assert sizes[-1] >= kmax
    assert max(sizes) <= CAP, sizes
