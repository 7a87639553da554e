"""CPU replay of the prefill kernels' work split.

The tensor-core prefill kernel cuts the batch's (tile of 64 new tokens, page)
units into one equal range per CTA, using a closed form for the pages that
tiles [0, t) of a request see, locates the range's first and last units, and
walks the range's tiles last one first (pages within a tile in order), so
that the CTAs scoring one request's tiles read its pages nearly together.
This replays that arithmetic (restated from the kernel) and checks that the
ranges of any grid cover every unit exactly once, and that on a long chunked
prefill the pages in flight form at most two compact fronts per request.
The bf16 kernel runs on pairs of CTAs (one range per pair) and multiplies a
segment's pages two at a time: pair g of a segment [j, je) is pages j + 2 g
(the even CTA's) and j + 2 g + 1 (the odd CTA's, absent past je); that
grouping is replayed too, with the pair kernel's ranges: on a batch of at
least 2 G * 512 units pair g of G walks ranges g and then g + G of a 2G-way
split, else range g of G.
"""

import numpy as np
import pytest

TILE, PAGE = 64, 128


def tiles_of(n):
    return (n + TILE - 1) // TILE


def tile_pages(n, L, t):
    last = min(n, TILE * (t + 1)) - 1
    return (L - n + last) // PAGE + 1


def pages_before(n, L, t, tile=None):
    """Closed form by residue: tile t' = R m + r (R = PAGE / tile) sees
    m + floor((c + tile r) / PAGE) + 1 pages."""
    tile = TILE if tile is None else tile
    R = PAGE // tile
    c = L - n + tile - 1
    total = t
    for r in range(R):
        n_r = (t - r + R - 1) // R if t > r else 0
        total += n_r * ((c + tile * r) // PAGE) + n_r * (n_r - 1) // 2
    return total


def req_units(n, L, ok=True):
    if not ok or n == 0:
        return 0
    T = tiles_of(n)
    return pages_before(n, L, T - 1) + tile_pages(n, L, T - 1)


def locate(reqs, units, u):
    """(b, t, j) of unit u of the batch's units in order."""
    cum = 0
    for b, v in enumerate(units):
        if cum + v > u:
            n, L, _ = reqs[b]
            rel = u - cum
            lo, hi = 0, tiles_of(n) - 1
            while lo < hi:
                mid = (lo + hi + 1) >> 1
                if pages_before(n, L, mid) <= rel:
                    lo = mid
                else:
                    hi = mid - 1
            return b, lo, rel - pages_before(n, L, lo)
        cum += v
    raise AssertionError("unit past the last one")


def plan(reqs, G, g):
    """(first (b, t, j), last (b, t, j + 1), units) for CTA g, as the kernel's
    planning warp computes them."""
    units = [req_units(n, L, ok) for n, L, ok in reqs]
    W = sum(units)
    u0, u1 = W * g // G, W * (g + 1) // G
    if u1 <= u0:
        return None
    b1, t1, j1 = locate(reqs, units, u1 - 1)
    return locate(reqs, units, u0), (b1, t1, j1 + 1), u1 - u0


def walk(reqs, start):
    """The kernel cursor's order: segments from the range's last tile back to
    its first, each segment's pages in order."""
    (fb, ft, fj), (b, t, je), left = start
    j = fj if (b, t) == (fb, ft) else 0
    out = []
    while left > 0:
        out.extend((b, t, x) for x in range(j, je))
        left -= je - j
        if left > 0:
            assert (b, t) != (fb, ft), "walked past the range"
            if t > 0:
                t -= 1
            else:
                b -= 1
                while b > fb and (not reqs[b][2] or reqs[b][0] == 0):
                    b -= 1
                t = tiles_of(reqs[b][0]) - 1
            n, L, _ = reqs[b]
            je = tile_pages(n, L, t)
            j = fj if (b, t) == (fb, ft) else 0
    assert left == 0 and (b, t) == (fb, ft)
    return out


def all_units(reqs):
    return [(b, t, j) for b, (n, L, ok) in enumerate(reqs) if ok
            for t in range(tiles_of(n)) for j in range(tile_pages(n, L, t))]


@pytest.mark.parametrize("tile", [16, 32, 64, 128])
def test_closed_form_matches_brute_force(tile):
    rng = np.random.default_rng(tile)
    for _ in range(1500):
        L = int(rng.integers(1, 300000))
        n = int(rng.integers(1, min(L, 5000) + 1))
        T = (n + tile - 1) // tile
        acc = 0
        for t in range(T):
            assert pages_before(n, L, t, tile) == acc, (n, L, t, tile)
            last = min(n, tile * (t + 1)) - 1
            acc += (L - n + last) // PAGE + 1


def _random_batch(rng):
    B = int(rng.integers(1, 40))
    reqs = []
    for _ in range(B):
        kind = rng.integers(0, 5)
        L = int(rng.integers(0, 20000)) if kind else int(rng.integers(0, 300))
        n = int(rng.integers(0, min(L, 3000) + 1)) if L else 0
        ok = bool(rng.random() > 0.1)
        reqs.append((n, L, ok))
    return reqs


@pytest.mark.parametrize("seed", range(6))
def test_ranges_cover_every_unit_once(seed):
    rng = np.random.default_rng(100 + seed)
    for _ in range(60):
        reqs = _random_batch(rng)
        expect = all_units(reqs)
        for G in (1, 2, 7, 76, 148, 152, 1000):
            got = []
            for g in range(G):
                start = plan(reqs, G, g)
                if start is not None:
                    got.extend(walk(reqs, start))
            assert sorted(got) == expect, (reqs, G)


def test_named_prefill_shapes():
    for pairs in ([(8192, 8192)], [(2048, 131072)] * 4, [(1, 1), (3, 3), (0, 50), (129, 4000)]):
        reqs = [(n, L, True) for n, L in pairs]
        got = []
        for g in range(148):
            s = plan(reqs, 148, g)
            if s is not None:
                got.extend(walk(reqs, s))
        assert sorted(got) == all_units(reqs)


def test_long_prefill_reads_pages_on_two_fronts():
    """4 requests x 2048 new tokens at 128K on 152 CTAs, each CTA taking one
    unit per step: at every step at least 90 % of the pages of one request
    being read lie in two windows of 32 pages (a page leaves DRAM about twice,
    not once per tile as with a first-tile-first walk; the few CTAs whose
    range straddles two requests read a third, small window)."""
    reqs = [(2048, 131072, True)] * 4
    G = 152
    walks = [walk(reqs, plan(reqs, G, g)) for g in range(G)]
    assert sorted(u for w in walks for u in w) == all_units(reqs)

    def windows(pages):
        """sizes of the groups of pages no more than 32 apart, largest first"""
        pages = sorted(pages)
        sizes = [1]
        for a, b in zip(pages, pages[1:]):
            if b - a > 32:
                sizes.append(1)
            else:
                sizes[-1] += 1
        return sorted(sizes, reverse=True)

    def fronts(pages):
        return len(windows(pages))

    worst = 1.0
    for step in range(max(len(w) for w in walks)):
        by_req = {}
        for w in walks:
            if step < len(w):
                b, _, page = w[step]
                by_req.setdefault(b, []).append(page)
        for v in by_req.values():
            if len(v) >= 8:
                worst = min(worst, sum(windows(v)[:2]) / len(v))
    assert worst >= 0.9, worst

    # first tile first, the same ranges: pages scattered over the whole context
    fwd = []
    for g in range(G):
        (b, t, j), _, left = plan(reqs, G, g)
        seq = []
        while left > 0:
            n, L, _ = reqs[b]
            je = min(tile_pages(n, L, t), j + left)
            seq.extend((b, x) for x in range(j, je))
            left -= je - j
            t, j = t + 1, 0
            if t >= tiles_of(n):
                b, t = b + 1, 0
        fwd.append(seq)
    spread = max(fronts([w[0][1] for w in fwd if w[0][0] == b]) for b in range(4))
    assert spread > 8


def pairs_of(j, je):
    return (je - j + 1) // 2


def pair_walk(reqs, start):
    """The pair kernel's order: the cursor's segments, each cut into pairs of
    pages; per pair (even CTA's page, odd CTA's page or None)."""
    seq = walk(reqs, start)
    segs = []
    for b, t, x in seq:
        if segs and segs[-1][0] == (b, t) and segs[-1][1][-1] == x - 1:
            segs[-1][1].append(x)
        else:
            segs.append(((b, t), [x]))
    out = []
    for (b, t), pages in segs:
        j, je = pages[0], pages[-1] + 1
        for g in range(pairs_of(j, je)):
            first = j + 2 * g
            second = first + 1 if first + 1 < je else None
            out.append((b, t, first, second))
    return out


@pytest.mark.parametrize("seed", range(4))
def test_pairs_cover_every_page_once(seed):
    """Every unit of a pair's range is the even or the odd CTA's page of
    exactly one pair; only a segment's last pair can lack its second page;
    stage (pair mod 6) and accumulator buffer (pair mod 2) follow the pairs."""
    rng = np.random.default_rng(500 + seed)
    for _ in range(40):
        reqs = _random_batch(rng)
        expect = all_units(reqs)
        for G in (1, 3, 76):
            got = []
            for g in range(G):
                start = plan(reqs, G, g)
                if start is None:
                    continue
                pairs = pair_walk(reqs, start)
                units = start[2]
                segments = len({(b, t) for b, t, _, _ in pairs})
                assert (units + 1) // 2 <= len(pairs) <= (units + segments) // 2 + segments
                for i, (b, t, first, second) in enumerate(pairs):
                    got.append((b, t, first))
                    if second is not None:
                        got.append((b, t, second))
                    else:  # a missing second page ends its segment
                        assert i + 1 == len(pairs) or pairs[i + 1][:2] != (b, t)
            assert sorted(got) == expect, (reqs, G)


def test_pair_counts_on_the_chunked_prefill():
    """4 x 2048 new tokens at 128K on 76 pairs: ~878 pairs of pages per pair
    of CTAs, at most a few half-empty ones."""
    reqs = [(2048, 131072, True)] * 4
    counts, halves = [], 0
    for g in range(76):
        pairs = pair_walk(reqs, plan(reqs, 76, g))
        counts.append(len(pairs))
        halves += sum(1 for p in pairs if p[3] is None)
    assert max(counts) - min(counts) <= 2
    assert halves <= 2 * 76


SPLIT_UNITS = 512


def pair_ranges(reqs, G, g):
    """The pair kernel's ranges for pair g of G, in walking order."""
    W = sum(req_units(n, L, ok) for n, L, ok in reqs)
    if W >= 2 * G * SPLIT_UNITS:
        return [plan(reqs, 2 * G, g), plan(reqs, 2 * G, g + G)]
    return [plan(reqs, G, g)]


@pytest.mark.parametrize("seed", range(3))
def test_pair_ranges_cover_every_unit_once(seed):
    rng = np.random.default_rng(700 + seed)
    batches = [_random_batch(rng) for _ in range(30)]
    batches.append([(2048, 131072, True)] * 4)  # the chunked prefill: two ranges a pair
    batches.append([(16, 8192, True)] * 256)    # short requests: one range a pair
    for reqs in batches:
        expect = all_units(reqs)
        for G in (1, 5, 76):
            got = []
            for g in range(G):
                for start in pair_ranges(reqs, G, g):
                    if start is not None:
                        got.extend(walk(reqs, start))
            assert sorted(got) == expect, (reqs, G)
    W = sum(req_units(n, L, ok) for n, L, ok in batches[-2])
    assert W >= 2 * 76 * SPLIT_UNITS
    W = sum(req_units(n, L, ok) for n, L, ok in batches[-1])
    assert W < 2 * 76 * SPLIT_UNITS


def test_two_ranges_keep_the_pages_of_a_request_together():
    """Chunked prefill on 76 pairs, one unit a pair per step, an LRU cache of
    1000 pages (31 MiB): with ranges g and g + 76 of 152 every page is missed
    once; one range of twice the length per pair misses ~9 times as often."""
    import collections
    reqs = [(2048, 131072, True)] * 4

    def misses(walks, cap=1000):
        lru, miss, pos = collections.OrderedDict(), 0, [0] * len(walks)
        while any(p < len(w) for p, w in zip(pos, walks)):
            for i, w in enumerate(walks):
                if pos[i] < len(w):
                    b, _, j = w[pos[i]]
                    pos[i] += 1
                    if (b, j) in lru:
                        lru.move_to_end((b, j))
                    else:
                        miss += 1
                        lru[(b, j)] = 1
                        if len(lru) > cap:
                            lru.popitem(last=False)
        return miss

    two = [sum((walk(reqs, r) for r in pair_ranges(reqs, 76, g)), []) for g in range(76)]
    one = [walk(reqs, plan(reqs, 76, g)) for g in range(76)]
    pages = 4 * 1024
    assert misses(two) == pages
    assert misses(one) > 5 * pages
