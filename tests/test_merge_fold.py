"""The merge kernel's list fold, restated on the CPU.

merge_kernel (csrc/msa_indexer.cu) combines a request's chunk lists in three
stages: per staged tile of lists, each group of KMAX lanes merges the lists
grp, grp + G, grp + 2G, ... of the tile pairwise (up to three levels, the
levels taken only as far as the tile's list count per group needs) and folds
the result into its running list; then the two groups of a warp meet by a
shuffle (KMAX = 16); then a tree over the groups through shared memory.  The
control flow decides which lists meet where, and every branch is uniform over
the CTA, so a list that no branch reaches would be lost without any fault.
This replays that flow with exact top-KMAX merges and checks, for every list
count a request can have in one or several tiles, that the result is the
top-KMAX of all the lists.
"""

import random

import pytest

THREADS = 256
TILE_KEYS = 2048


def top(keys, kmax):
    """A descending top-kmax list, padded with the empty key 0."""
    out = sorted((k for k in keys if k), reverse=True)[:kmax]
    return out + [0] * (kmax - len(out))


def merge(a, b, kmax):
    return top(a + b, kmax)


def fold(lists, kmax, drop_third_level=False):
    """The kernel's fold of `lists` (each a descending list of kmax keys).
    drop_third_level plants a mistake (lists 4-7 of a group never merged)
    for the check of the checker."""
    groups = THREADS // kmax
    tile_lists = TILE_KEYS // kmax
    assert tile_lists == groups * 8
    n_lists = len(lists)
    empty = [0] * kmax
    run = [empty[:] for _ in range(groups)]
    for t0 in range(0, n_lists, tile_lists):
        nt = min(tile_lists, n_lists - t0)
        per = (nt + groups - 1) // groups  # uniform over the CTA
        for grp in range(groups):
            def lst(m):
                li = grp + groups * m
                return lists[t0 + li] if li < nt else empty
            a0 = lst(0)
            if per > 1:
                a0 = merge(a0, lst(1), kmax)
                if per > 2:
                    a2 = merge(lst(2), lst(3), kmax)
                    if per > 4 and not drop_third_level:
                        a4 = merge(lst(4), lst(5), kmax)
                        a6 = merge(lst(6), lst(7), kmax)
                        a4 = merge(a4, a6, kmax)
                    a0 = merge(a0, a2, kmax)
                    if per > 4 and not drop_third_level:
                        a0 = merge(a0, a4, kmax)
            run[grp] = a0 if t0 == 0 else merge(run[grp], a0, kmax)
    used = min(n_lists, groups)
    first_step = 1
    if kmax == 16:
        if used > 1:  # both halves of each warp take the union of the pair
            run = [merge(run[g], run[g ^ 1], kmax) for g in range(groups)]
        first_step = 2
    step = first_step
    while step < groups:
        if step >= used:
            break
        nxt = []
        for g in range(groups):
            active = g % (2 * step) == 0 and g + step < groups
            nxt.append(merge(run[g], run[g + step] if active else empty, kmax))
        run = nxt
        step <<= 1
    return run[0]


def random_lists(rng, n, kmax, sparse):
    keys = rng.sample(range(1, 1 << 40), n * kmax)
    lists = []
    for i in range(n):
        ks = keys[i * kmax:(i + 1) * kmax]
        if sparse and rng.random() < 0.3:
            ks = ks[:rng.randint(0, kmax)]  # a chunk with fewer free blocks
        lists.append(top(ks, kmax))
    return lists


@pytest.mark.parametrize("kmax", [16, 32])
def test_fold_equals_the_top_of_all_lists(kmax):
    """Every list count of one tile and of up to three tiles, sparse lists too."""
    rng = random.Random(kmax)
    tile_lists = TILE_KEYS // kmax
    for n in list(range(0, tile_lists + 2)) + [2 * tile_lists - 1, 2 * tile_lists + 5,
                                                3 * tile_lists]:
        for sparse in (False, True):
            lists = random_lists(rng, n, kmax, sparse)
            want = top([k for l in lists for k in l], kmax)
            assert fold(lists, kmax) == want, (n, sparse)


def test_fold_checker_catches_a_lost_level():
    """The replay itself: with lists 4-7 of each group never merged, a tile of
    five or more lists a group loses the winners planted in list 4 of group 0."""
    kmax, groups = 16, THREADS // 16
    lists = random_lists(random.Random(3), groups * 6, kmax, False)
    lists[4 * groups] = top([(1 << 41) + i for i in range(kmax)], kmax)
    want = top([k for l in lists for k in l], kmax)
    assert fold(lists, kmax) == want
    assert fold(lists, kmax, drop_third_level=True) != want
