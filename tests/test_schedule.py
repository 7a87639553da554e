"""The score kernel's work split, restated on the CPU and checked for bounds.

The CUDA kernels cannot be run under a memory checker on this pool, so their
index arithmetic is replayed here: the request prefix sums, the chunking of
the batch's pages over the CTAs, the (chunk, request) segments, the stage each
page lands in, the candidate slot each segment writes, and the slots the
merge kernel reads.  For random batches it checks that every page of every
request is visited exactly once, that each stage's barrier phases are used in
order by their single owner warp, and that every slot index is unique and
inside the workspace that msa_indexer_workspace_bytes() sizes.
"""

import random

import pytest

CONSUMERS, STAGES_PER_CONSUMER = 2, 3  # must match score_kernel's pipeline shape
STAGES = CONSUMERS * STAGES_PER_CONSUMER
MAX_GRID = 1024


def stage_of(it):
    return it % CONSUMERS + CONSUMERS * ((it // CONSUMERS) % STAGES_PER_CONSUMER)


def ceil_div(a, b):
    return -(-a // b)


def workspace_slots(max_batch, max_model_len, split):
    chunks = MAX_GRID if split == 0 else ceil_div(max_batch * ceil_div(max_model_len, 128), split)
    return chunks + max_batch


def find_row(prefix, batch, p):
    lo, hi = 0, batch - 1
    while lo < hi:
        mid = (lo + hi + 1) >> 1
        if prefix[mid] <= p:
            lo = mid
        else:
            hi = mid - 1
    return lo


def replay(seq, max_model_len, bt_stride, split_blocks, sms):
    B = len(seq)
    max_blocks = ceil_div(max_model_len, 128)
    work = B * max_blocks
    units = ceil_div(work, split_blocks) if split_blocks else work
    grid = max(1, min(sms, MAX_GRID, units))
    limit = min(max_model_len, bt_stride * 128)
    nb = [ceil_div(L, 128) if 0 <= L <= limit else 0 for L in seq]
    prefix = [0]
    for n in nb:
        prefix.append(prefix[-1] + n)
    total = prefix[-1]
    split = split_blocks if split_blocks else max(1, ceil_div(total, grid))
    chunks = ceil_div(total, split) if total else 0
    host_need = (grid if split_blocks == 0 else ceil_div(B * max_blocks, split_blocks)) + B
    capacity = workspace_slots(B, max_model_len, split_blocks)
    assert host_need <= capacity
    seen, written = set(), {}
    for cta in range(grid):
        it, uses = 0, {}
        for c in range(cta, chunks, grid):
            p0, p1 = c * split, min(total, c * split + split)
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
                    s = stage_of(my)
                    assert s % CONSUMERS == my % CONSUMERS  # owned by the page's consumer warp
                    assert uses.get(s, -1) == my // STAGES - 1  # phases in order
                    uses[s] = my // STAGES
                it += seg_end - pg
                slot = c + b
                assert slot < capacity and slot not in written
                written[slot] = (c, b)
                pg = seg_end
    assert len(seen) == total
    for b in range(B):
        if prefix[b + 1] > prefix[b]:
            first = prefix[b] // split
            n_lists = (prefix[b + 1] - 1) // split - first + 1
            for i in range(n_lists):
                assert written[first + i + b] == (first + i, b)
    return grid, split, chunks


def test_headline_geometry():
    assert replay([131072] * 32, 131072, 1024, 0, 152) == (152, 216, 152)
    assert replay([8700] * 16, 8704, 68, 0, 152) == (152, 8, 136)


@pytest.mark.parametrize("W", [0, 1, 2, 3, 8, 64, 1024])
def test_named_workloads(W):
    for sms in (152, 7, 1000):
        replay([131072, 0, 129] + [1024] * 13, 131072, 1024, W, sms)
        replay([8700] * 16, 8704, 68, W, sms)
        replay([1000, 700], 1024, 8, W, sms)


def test_random_batches():
    rng = random.Random(0)
    for _ in range(300):
        B = rng.randint(1, 40)
        mml = rng.choice([128, 1000, 4096, 16384, 70000])
        bts = ceil_div(mml, 128) + rng.randint(0, 3)
        seq = [rng.choice([0, 1, 127, 128, 129, rng.randint(0, mml), -3, mml + 500])
               for _ in range(B)]
        W = rng.choice([0, 0, 1, 2, 5, 17, 64])
        for sms in (152, 7):
            replay(seq, mml, bts, W, sms)
