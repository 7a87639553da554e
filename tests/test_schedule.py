"""The score kernel's work split, restated on the CPU and checked for bounds.

The CUDA kernels cannot be run under a memory checker on this pool, so their
index arithmetic is replayed here: the request prefix sums, the partition of
the batch's pages into chunks (a static home chunk per CTA plus pool chunks
claimed through a counter, in a random interleaving of the CTAs), the
(chunk, request) segments, the stage each page lands in, the candidate slot
each segment writes and the slots the merge kernel reads.  For random batches
it checks that every page of every request is visited exactly once, that each
stage's barrier phases are used in order by their single owner warp, that
every slot index is unique and inside the workspace, and that the chunks the
merge reads for a request are exactly those that wrote its lists.
"""

import random

import pytest

MAX_GRID = 1024
MAX_LEVELS = 6
MIN_POOL_HOME = 64


def ceil_div(a, b):
    return -(-a // b)


class Partition:
    """Mirror of msa::Partition (csrc/layout.cuh)."""

    def __init__(self, total, grid, split_blocks):
        self.grid, self.total = grid, total
        self.lo = [0] * (MAX_LEVELS + 2)
        if split_blocks > 0:
            self.forced, self.unit, self.levels = True, split_blocks, 0
            self.chunks = ceil_div(total, split_blocks) if total > 0 else 0
            self.pool = max(0, self.chunks - grid)
            return
        self.forced = False
        H = ceil_div(total, grid) if total > 0 else 1
        self.unit = H
        T, pool_pages = 0, 0
        while H >= MIN_POOL_HOME and T < MAX_LEVELS and (H >> (T + 3)) > 0:
            pool_pages += H >> (T + 3)
            T += 1
        self.levels = T
        self.lo[1] = H - pool_pages
        for t in range(T):
            self.lo[t + 2] = self.lo[t + 1] + (H >> (t + 3))
        self.chunks = self.chunk_of(total - 1) + 1 if total > 0 else 0
        self.pool = grid * T

    def range(self, c):
        if self.forced:
            s, e = c * self.unit, c * self.unit + self.unit
        else:
            g, r = divmod(c, 1 + self.levels)
            s, e = g * self.unit + self.lo[r], g * self.unit + self.lo[r + 1]
        return min(s, self.total), min(e, self.total)

    def chunk_of(self, p):
        if self.forced:
            return p // self.unit
        g = p // self.unit
        off = p - g * self.unit
        r = 0
        while r < self.levels and self.lo[r + 1] <= off:
            r += 1
        return g * (1 + self.levels) + r

    def first_chunk(self, g):
        c = g if self.forced else g * (1 + self.levels)
        return c if c < self.chunks else -1

    def pool_chunk(self, i):
        if i < 0 or i >= self.pool:
            return -1
        c = self.grid + i if self.forced else (i % self.grid) * (1 + self.levels) + 1 + i // self.grid
        return c if c < self.chunks else -2


def chunk_capacity(grid, max_pages, split_blocks):
    return ceil_div(max_pages, split_blocks) if split_blocks > 0 else grid * (1 + MAX_LEVELS)


# (consumer warps, stages per consumer warp, stages per page) of each format;
# the replay also covers pages split over several stages
FORMATS = {"bf16": (2, 3, 1), "fp8": (4, 3, 1), "fp8_mq": (4, 2, 1), "bf16_wide4": (4, 1, 1)}


def stage_of(it, h=0, fmt=FORMATS["bf16"]):
    C, spc, units = fmt
    local = (it // C) * units + h
    return it % C + C * (local % spc)


def use_of(it, h=0, fmt=FORMATS["bf16"]):
    C, spc, units = fmt
    return ((it // C) * units + h) // spc


def find_row(prefix, batch, p):
    lo, hi = 0, batch - 1
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if prefix[mid] <= p:
            lo = mid
        else:
            hi = mid - 1
    return lo


def score_grid(sms, batch, max_blocks, split_blocks):
    work = batch * max_blocks
    units = ceil_div(work, split_blocks) if split_blocks else work
    return max(1, min(sms, MAX_GRID, units))


def replay(seq, max_model_len, bt_stride, split_blocks, sms, rng, fmt=FORMATS["bf16"]):
    B = len(seq)
    max_blocks = ceil_div(max_model_len, 128)
    grid = score_grid(sms, B, max_blocks, split_blocks)
    limit = min(max_model_len, bt_stride * 128)
    nb = [ceil_div(L, 128) if 0 <= L <= limit else 0 for L in seq]
    prefix = [0]
    for n in nb:
        prefix.append(prefix[-1] + n)
    total = prefix[-1]
    part = Partition(total, grid, split_blocks)
    capacity = chunk_capacity(grid, B * max_blocks, split_blocks) + B
    assert part.chunks + B <= capacity
    # every chunk inside the batch is non-empty and they tile [0, total)
    pos = 0
    for c in range(part.chunks):
        a, b = part.range(c)
        assert a == pos and b > a, (c, a, b, pos)
        pos = b
        assert part.chunk_of(a) == c and part.chunk_of(b - 1) == c
    assert pos == total

    # each CTA: its static chunk, then pool tickets in a random interleaving
    seqs = [[] for _ in range(grid)]
    for g in range(grid):
        c = part.first_chunk(g)
        if c >= 0:
            seqs[g].append(c)
    tickets = list(range(part.pool + grid))  # extra tickets past the end come back -1
    for i in tickets:
        g = rng.randrange(grid)
        c = part.pool_chunk(i)
        if c >= 0:
            seqs[g].append(c)
    done = sorted(c for s in seqs for c in s)
    assert done == list(range(part.chunks)), "every chunk exactly once"

    seen, written = set(), {}
    for g in range(grid):
        it, uses = 0, {}
        for c in seqs[g]:
            p0, p1 = part.range(c)
            pg = p0
            while pg < p1:
                b = find_row(prefix, B, pg)
                assert prefix[b] <= pg < prefix[b + 1]
                seg_end = min(p1, prefix[b + 1])
                for x in range(pg, seg_end):
                    my = it + (x - pg)
                    j = x - prefix[b]
                    assert 0 <= j < nb[b] <= bt_stride
                    assert (b, j) not in seen
                    seen.add((b, j))
                    for h in range(fmt[2]):
                        s = stage_of(my, h, fmt)
                        assert s % fmt[0] == my % fmt[0]  # owned by the page's consumer warp
                        assert 0 <= s < fmt[0] * fmt[1]
                        assert uses.get(s, -1) == use_of(my, h, fmt) - 1  # phases in order
                        uses[s] = use_of(my, h, fmt)
                it += seg_end - pg
                slot = c + b
                assert slot < capacity and slot not in written
                written[slot] = (c, b)
                pg = seg_end
        # the producer's drain waits on the last C * spc units: each used
        # stage's latest use is among them, exactly once
        n_units = it * fmt[2]
        last = [stage_of(u // fmt[2], u % fmt[2], fmt) for u in range(max(0, n_units - fmt[0] * fmt[1]), n_units)]
        assert len(last) == len(set(last))
        assert set(last) == set(uses)
        for u in range(max(0, n_units - fmt[0] * fmt[1]), n_units):
            q, h = divmod(u, fmt[2])
            assert use_of(q, h, fmt) == uses[stage_of(q, h, fmt)]
    assert len(seen) == total
    segments = [0] * B
    for (c, b) in written.values():
        segments[b] += 1
    for b in range(B):
        if prefix[b + 1] > prefix[b]:
            first, last = part.chunk_of(prefix[b]), part.chunk_of(prefix[b + 1] - 1)
            for c in range(first, last + 1):
                assert written[c + b] == (c, b)
            # one list per (chunk, request) segment: the merge reads exactly these
            assert segments[b] == last - first + 1
        else:
            assert segments[b] == 0
    return grid, part


def test_headline_geometry():
    rng = random.Random(1)
    grid, part = replay([131072] * 32, 131072, 1024, 0, 152, rng)
    assert grid == 152 and part.unit == 216 and part.levels == 5
    assert part.lo[:7] == [0, 166, 193, 206, 212, 215, 216]
    grid, part = replay([8700] * 16, 8704, 68, 0, 152, rng)
    assert part.unit == 8 and part.levels == 0


@pytest.mark.parametrize("W", [0, 1, 2, 3, 8, 64, 1024])
def test_named_workloads(W):
    rng = random.Random(W)
    for sms in (152, 7, 1000):
        replay([131072, 0, 129] + [1024] * 13, 131072, 1024, W, sms, rng)
        replay([8700] * 16, 8704, 68, W, sms, rng)
        replay([1000, 700], 1024, 8, W, sms, rng)
        replay([32768] * 32, 32768, 256, W, sms, rng)


def test_random_batches():
    rng = random.Random(0)
    for _ in range(400):
        B = rng.randint(1, 40)
        mml = rng.choice([128, 1000, 4096, 16384, 70000])
        bts = ceil_div(mml, 128) + rng.randint(0, 3)
        seq = [rng.choice([0, 1, 127, 128, 129, rng.randint(0, mml), -3, mml + 500])
               for _ in range(B)]
        W = rng.choice([0, 0, 0, 1, 2, 5, 17, 64])
        for sms in (152, 7):
            replay(seq, mml, bts, W, sms, rng)


@pytest.mark.parametrize("fmt", sorted(FORMATS) + ["split_pages"])
def test_stage_rings_of_every_format(fmt):
    rng = random.Random(7)
    for _ in range(60):
        B = rng.randint(1, 40)
        seq = [rng.choice([0, 1, 127, 128, 129, rng.randint(1, 20000)]) for _ in range(B)]
        shape = FORMATS[fmt] if fmt in FORMATS else (4, 6, 2)
        replay(seq, 20480, 160, rng.choice([0, 0, 1, 3, 64]), rng.choice([1, 7, 152]), rng, shape)
