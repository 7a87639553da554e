"""CPU replay of the E4M3 prefill kernel's warp roles and row mappings.

Restated from the kernel: 23 warps; warp 0 producer, warp 2 MMA issue,
warps 1 and 3-5 convert one key row per thread, warps 6-21 are the
epilogue and warp 22 waits on the barriers for the issuing thread.  Epilogue warp e (warp 6 + e) may read only the TMEM lanes of its
quarter (warp % 4); it owns M tile e / 8 and the 16 rows 32 q + 16 ((e / 4)
% 2) of that quarter.  Per page it reads those 16 rows in the mma-fragment
layout (lane (g, c) holds rows g and g + 8, columns 8 i + 2 c + {0, 1}) and
lanes with c < 2 write one row each; for the query conversion two lanes share
a row, one half of its 128 dimensions each.
"""

from collections import Counter

TILE_TOKENS, HEADS, M_ROWS, M_TILES, PAGE = 64, 4, 128, 2, 128
FIRST_EPI, EPI_WARPS, WAITER, WARPS = 6, 16, 22, 23
CONVERTERS = (1, 3, 4, 5)


def roles():
    out = {}
    for w in range(WARPS):
        if w == 0:
            out[w] = "producer"
        elif w == 2:
            out[w] = "mma"
        elif w < FIRST_EPI:
            out[w] = "converter"
        elif w == WAITER:
            out[w] = "waiter"
        else:
            out[w] = "epilogue"
    return out


def epilogue_warp(w):
    e = w - FIRST_EPI
    quarter = w & 3
    mt = e >> 3
    hh = (e >> 2) & 1
    return quarter, mt, 32 * quarter + 16 * hh


def test_roles_and_register_budget():
    r = roles()
    assert [w for w in r if r[w] == "converter"] == list(CONVERTERS)
    assert sum(v == "epilogue" for v in r.values()) == EPI_WARPS
    assert [w for w in r if r[w] == "waiter"] == [WAITER] and WAITER == FIRST_EPI + EPI_WARPS
    # the MMA warp's SM sub-partition (warp % 4) holds no converter warp
    assert all(w % 4 != 2 % 4 for w in CONVERTERS)
    per_sub = Counter(w % 4 for w in range(WARPS))
    regs = (16384 // (32 * max(per_sub.values()))) & ~7
    assert regs == 80
    assert WARPS * 32 * regs <= 65536


def test_converters_cover_every_key_row_once():
    rows = Counter()
    for w in CONVERTERS:
        for lane in range(32):
            rows[32 * (0 if w == 1 else w - 2) + lane] += 1
    assert sorted(rows) == list(range(PAGE)) and set(rows.values()) == {1}


def test_epilogue_reads_its_quarter_and_writes_each_row_once():
    written = Counter()
    converted = Counter()
    for w in range(FIRST_EPI, FIRST_EPI + EPI_WARPS):
        quarter, mt, row0 = epilogue_warp(w)
        # the 16 TMEM lanes read per load lie in the warp's quarter
        assert 32 * quarter <= row0 and row0 + 16 <= 32 * quarter + 32
        for lane in range(32):
            g, c = lane >> 2, lane & 3
            held = {row0 + g, row0 + g + 8}
            assert all(32 * quarter <= r < 32 * quarter + 32 for r in held)
            if c < 2:
                mine = row0 + g + 8 * (c & 1)
                assert mine in held
                written[mt * M_ROWS + mine] += 1
            converted[(mt * M_ROWS + row0 + (lane & 15), lane >> 4)] += 1
    assert sorted(written) == list(range(M_TILES * M_ROWS))
    assert set(written.values()) == {1}
    assert len(converted) == M_TILES * M_ROWS * 2 and set(converted.values()) == {1}


def test_row_positions():
    """Rows g and g + 8 of a warp's 16 are the tokens pos_q and pos_q + 2,
    pos_q = the warp's first token + g / 4 (4 heads per token)."""
    for w in range(FIRST_EPI, FIRST_EPI + EPI_WARPS):
        _, mt, row0 = epilogue_warp(w)
        first = (mt * M_ROWS + row0) // HEADS
        for g in range(8):
            pos_q = first + (g >> 2)
            assert (mt * M_ROWS + row0 + g) // HEADS == pos_q
            assert (mt * M_ROWS + row0 + g + 8) // HEADS == pos_q + 2
        # the warp's smallest token bounds every row's visibility from below
        assert all((mt * M_ROWS + row0 + r) // HEADS >= first for r in range(16))
