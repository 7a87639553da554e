"""CPU replay of the E4M3 prefill kernel's warp roles and row mappings.

Restated from the kernel (tc_prefill_fp8_kernel, pairs of CTAs): 23 warps a
CTA; warp 0 producer, warp 1 the issuing thread (even CTA) or forwarder (odd
CTA), warp 2 the waiter, warps 3-6 converters (query row and key row 32 w' +
lane, w' = warp - 3) and warps 7-22 the epilogue.  Epilogue warp e (warp 7 +
e) may read only the TMEM lanes of its quarter (warp % 4); it owns page
(e / 4) % 2 of the pair and the 16 rows 32 q + 16 (e / 8) of that quarter.
Per pair it reads those 16 rows x 128 columns in the mma-fragment layout
(lane (g, c) holds rows g and g + 8, columns 8 i + 2 c + {0, 1}) and lanes
with c < 2 write one row each.  The CTA's 128 rows are rows 128 rank ..
128 rank + 127 of the tile's 256 (64 tokens x 4 heads).
"""

from collections import Counter

TILE_TOKENS, HEADS, M_ROWS, PAGE = 64, 4, 128, 128
FIRST_CONV, CONV_WARPS, FIRST_EPI, EPI_WARPS, WAITER, WARPS = 3, 4, 7, 16, 2, 23


def roles():
    out = {}
    for w in range(WARPS):
        if w == 0:
            out[w] = "producer"
        elif w == 1:
            out[w] = "mma"
        elif w == WAITER:
            out[w] = "waiter"
        elif w < FIRST_EPI:
            out[w] = "converter"
        else:
            out[w] = "epilogue"
    return out


def epilogue_warp(w):
    e = w - FIRST_EPI
    quarter = w & 3
    idx = e >> 2
    return quarter, idx & 1, 32 * quarter + 16 * (idx >> 1)  # quarter, page of the pair, row0


def test_roles_and_register_budget():
    r = roles()
    assert [w for w in r if r[w] == "converter"] == list(range(FIRST_CONV, FIRST_CONV + CONV_WARPS))
    assert sum(v == "epilogue" for v in r.values()) == EPI_WARPS
    assert FIRST_EPI + EPI_WARPS == WARPS
    per_sub = Counter(w % 4 for w in range(WARPS))
    regs = (16384 // (32 * max(per_sub.values()))) & ~7
    assert regs == 80
    assert WARPS * 32 * regs <= 65536


def test_converters_cover_every_row_once():
    """A query row and a key row a lane: the CTA's 128 of each, once."""
    rows = Counter()
    for w in range(FIRST_CONV, FIRST_CONV + CONV_WARPS):
        for lane in range(32):
            rows[32 * (w - FIRST_CONV) + lane] += 1
    assert sorted(rows) == list(range(M_ROWS)) and set(rows.values()) == {1}
    assert M_ROWS == PAGE


def test_epilogue_reads_its_quarter_and_writes_each_row_of_each_page_once():
    for rank in (0, 1):
        written = Counter()
        for w in range(FIRST_EPI, FIRST_EPI + EPI_WARPS):
            quarter, h, row0 = epilogue_warp(w)
            # the 16 TMEM lanes read per load lie in the warp's quarter
            assert 32 * quarter <= row0 and row0 + 16 <= 32 * quarter + 32
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                held = {row0 + g, row0 + g + 8}
                assert all(32 * quarter <= r < 32 * quarter + 32 for r in held)
                if c < 2:
                    mine = row0 + g + 8 * (c & 1)
                    assert mine in held
                    written[(h, M_ROWS * rank + mine)] += 1
        assert sorted(written) == [(h, M_ROWS * rank + r) for h in (0, 1) for r in range(M_ROWS)]
        assert set(written.values()) == {1}


def test_row_positions():
    """Rows g and g + 8 of a warp's 16 are the tokens pos_q and pos_q + 2,
    pos_q = the warp's first token + g / 4 (4 heads per token)."""
    for rank in (0, 1):
        for w in range(FIRST_EPI, FIRST_EPI + EPI_WARPS):
            _, _, row0 = epilogue_warp(w)
            first = (M_ROWS * rank + row0) // HEADS
            for g in range(8):
                pos_q = first + (g >> 2)
                assert (M_ROWS * rank + row0 + g) // HEADS == pos_q
                assert (M_ROWS * rank + row0 + g + 8) // HEADS == pos_q + 2
            # the warp's smallest token bounds every row's visibility from below
            assert all((M_ROWS * rank + row0 + r) // HEADS >= first for r in range(16))
            assert first < TILE_TOKENS
