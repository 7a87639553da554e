"""CPU replay of the prefill kernel's work split.

The tensor-core prefill kernel cuts the batch's (tile of 64 new tokens, page)
units into one equal range per CTA, using a closed form for the pages that
tiles [0, t) of a request see, then walks tiles in order from its start.
This replays that arithmetic (restated from the kernel) and checks that the
ranges of any grid cover every unit exactly once.
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


def plan(reqs, G, g):
    """(b, t, j, units) for CTA g, as the kernel's planning warp computes them."""
    units = [req_units(n, L, ok) for n, L, ok in reqs]
    W = sum(units)
    u0, u1 = W * g // G, W * (g + 1) // G
    if u1 <= u0:
        return None
    cum = 0
    for b, v in enumerate(units):
        if cum + v > u0:
            n, L, _ = reqs[b]
            rel = u0 - cum
            lo, hi = 0, tiles_of(n) - 1
            while lo < hi:
                mid = (lo + hi + 1) >> 1
                if pages_before(n, L, mid) <= rel:
                    lo = mid
                else:
                    hi = mid - 1
            return b, lo, rel - pages_before(n, L, lo), u1 - u0
        cum += v
    raise AssertionError("range start past the last unit")


def walk(reqs, start):
    b, t, j, left = start
    out = []
    while left > 0:
        n, L, _ = reqs[b]
        nb = tile_pages(n, L, t)
        je = min(nb, j + left)
        out.extend((b, t, x) for x in range(j, je))
        left -= je - j
        if left > 0:
            t, j = t + 1, 0
            if t >= tiles_of(n):
                t = 0
                b += 1
                while b < len(reqs) and (not reqs[b][2] or reqs[b][0] == 0):
                    b += 1
                assert b < len(reqs), "walked past the batch"
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
        for G in (1, 2, 7, 148, 152, 1000):
            got = []
            for g in range(G):
                start = plan(reqs, G, g)
                if start is not None:
                    got.extend(walk(reqs, start))
            assert got == expect, (reqs, G)


def test_named_prefill_shapes():
    for pairs in ([(8192, 8192)], [(2048, 131072)] * 4, [(1, 1), (3, 3), (0, 50), (129, 4000)]):
        reqs = [(n, L, True) for n, L in pairs]
        got = []
        for g in range(148):
            s = plan(reqs, 148, g)
            if s is not None:
                got.extend(walk(reqs, s))
        assert got == all_units(reqs)
