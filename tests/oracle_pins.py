"""Checks that pin the CPU oracle to facts other than itself.

Each check takes an ``oracle.Oracle`` and raises AssertionError on failure:

* ``check_golden``: hand-derived closed-form fixtures under tests/golden/;
* ``check_scores_vs_numpy``: block scores against an independent numpy
  matmul + max over the valid tokens (a library routine, not the oracle's loop);
* ``check_select_vs_rank_count``: the sort-based selection against a
  brute-force rank counter on tie-heavy integer scores;
* ``check_invariants``: fewer-than-k returns everything, pins are present,
  split-merge equals unsplit for every split width, empty rows return nothing,
  permuting the page pool changes nothing, scaling q by 2 keeps the ids.

The mutation tests run the same checks against deliberately broken copies of
the oracle and require at least one check to fail for each.
"""

from __future__ import annotations

import glob
import json
import os

import numpy as np

import workloads as wl

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
HEADS, DIM, PAGE = wl.HEADS, wl.DIM, wl.PAGE


# ----------------------------------------------------------------------------
# planted closed-form cases
# ----------------------------------------------------------------------------

def build_planted(fx: dict):
    """Inputs of a golden fixture: see tests/golden/README.md for the rule."""
    seq = np.asarray(fx["seq_lens"], dtype=np.int32)
    B = seq.shape[0]
    nb = [(int(L) + PAGE - 1) // PAGE for L in seq]
    stride = max(1, max(nb))
    num_pages = max(1, sum(nb))
    dim, m = int(fx["dim"]), int(fx["m"])
    pool = np.zeros((num_pages, PAGE, DIM), dtype=np.float32)
    bt = np.full((B, stride), -1, dtype=np.int32)
    page = 0
    for b in range(B):
        for j in range(nb[b]):
            bt[b, j] = page
            t = np.arange(PAGE)
            pool[page, :, dim] = float(fx["c"][b][j]) - (t % m)
            page += 1
    q = np.zeros((B, HEADS, DIM), dtype=np.float32)
    for b in range(B):
        q[b, :, dim] = np.asarray(fx["alpha"], dtype=np.float32)
    pool_bits = wl.f32_to_bf16_bits(pool)
    q_bits = wl.f32_to_bf16_bits(q)
    wl.poison_tails(pool_bits, bt, seq)
    return q_bits, pool_bits, bt, seq


def load_golden():
    out = []
    for path in sorted(glob.glob(os.path.join(GOLDEN_DIR, "planted_*.json"))):
        with open(path) as f:
            out.append(json.load(f))
    return out


def check_expand_golden(orc) -> None:
    with open(os.path.join(GOLDEN_DIR, "expand_pages.json")) as f:
        fx = json.load(f)
    seq = np.asarray(fx["seq_lens"], dtype=np.int32)
    B, stride = seq.shape[0], int(fx["kv_stride"])
    kvb = np.array([[1000 * b + 100 + p for p in range(stride)] for b in range(B)], dtype=np.int32)
    ids = np.asarray(fx["ids"], dtype=np.int32)
    pages, num = orc.expand_pages(ids, seq, kvb, int(fx["page_tokens"]))
    np.testing.assert_array_equal(num, np.asarray(fx["expected_num"], dtype=np.int32))
    for b in range(B):
        for h in range(HEADS):
            exp = fx["expected_pages_prefix"][b][h]
            assert list(pages[b, h, :len(exp)]) == exp, (b, h)
            assert np.all(pages[b, h, len(exp):] == -1)


def check_expand_invariants(orc) -> None:
    """Brute-force set view: the pages listed are exactly those of the selected blocks."""
    rng = np.random.default_rng(17)
    for page_tokens in (16, 32, 64, 128, 8):
        per = 128 // page_tokens
        for _ in range(20):
            B, k = int(rng.integers(1, 4)), int(rng.integers(1, 17))
            seq = rng.integers(0, 2000, size=B).astype(np.int32)
            stride = int(-(-2000 // page_tokens)) + 1
            kvb = rng.permutation(B * stride).astype(np.int32).reshape(B, stride)
            ids = np.full((B, HEADS, k), -1, dtype=np.int32)
            for b in range(B):
                nb = -(-int(seq[b]) // 128)
                for h in range(HEADS):
                    m = min(k, nb)
                    if m:
                        ids[b, h, :m] = rng.choice(nb, size=m, replace=False)
            pages, num = orc.expand_pages(ids, seq, kvb, page_tokens)
            for b in range(B):
                small = -(-int(seq[b]) // page_tokens)
                for h in range(HEADS):
                    want = [int(kvb[b, j * per + s]) for j in sorted(x for x in ids[b, h] if x >= 0)
                            for s in range(per) if j * per + s < small]
                    assert int(num[b, h]) == len(want)
                    assert list(pages[b, h, :len(want)]) == want
                    assert np.all(pages[b, h, len(want):] == -1)


def check_golden(orc) -> None:
    fixtures = load_golden()
    assert len(fixtures) >= 4, "golden fixtures missing"
    for fx in fixtures:
        q, pool, bt, seq = build_planted(fx)
        k = int(fx["k"])
        s = orc.block_scores(q, pool, bt, seq)
        ids, sc = orc.select(s, seq, k, int(fx["n_sink"]), int(fx["n_window"]))
        exp_ids = np.asarray(fx["expected_ids"], dtype=np.int32)
        assert ids.shape == exp_ids.shape, fx["name"]
        np.testing.assert_array_equal(ids, exp_ids, err_msg=fx["name"])
        for b in range(seq.shape[0]):
            for h in range(HEADS):
                row = list(fx["expected_scores"][b][h])
                exp = np.full(k, -np.inf)
                exp[:len(row)] = row
                np.testing.assert_array_equal(sc[b, h], exp, err_msg=f"{fx['name']} b={b} h={h}")


# ----------------------------------------------------------------------------
# block scores against numpy
# ----------------------------------------------------------------------------

def numpy_block_scores(q_bits, pool_bits, bt, seq) -> np.ndarray:
    qf = wl.bf16_bits_to_f32(q_bits).astype(np.float64)
    B, stride = bt.shape
    out = np.full((B, HEADS, stride), -np.inf)
    for b in range(B):
        L = int(seq[b])
        for j in range((L + PAGE - 1) // PAGE):
            valid = min(PAGE, L - j * PAGE)
            kf = wl.bf16_bits_to_f32(pool_bits[int(bt[b, j]), :valid]).astype(np.float64)
            out[b, :, j] = (qf[b] @ kf.T).max(axis=1)
    return out


def mixed_workload(seed: int = 11):
    """Small, mixed lengths: empty, single-token, partial and full blocks."""
    return wl.random_workload([0, 1, 127, 128, 129, 700, 1000, 2048, 1999], num_pages=96,
                              seed=seed, q_scale=1.0 / np.sqrt(DIM), max_model_len=2048)


def check_scores_vs_numpy(orc) -> None:
    for seed in (11, 12):
        w = mixed_workload(seed)
        s = orc.block_scores(w.q, w.pool, w.block_table, w.seq_lens)
        ref = numpy_block_scores(w.q, w.pool, w.block_table, w.seq_lens)
        finite = np.isfinite(ref)
        np.testing.assert_array_equal(np.isfinite(s), finite)
        np.testing.assert_allclose(s[finite], ref[finite], rtol=1e-12, atol=1e-12)
        assert np.all(s[~finite] == -np.inf)


# ----------------------------------------------------------------------------
# selection against a brute-force rank counter
# ----------------------------------------------------------------------------

def rank_count_select(s_row, nb, k, n_sink, n_window):
    """Block j is chosen iff pinned, or fewer than (k - #pinned) free blocks beat it.

    A free block i beats j when its score is higher, or equal with a lower id.
    Output: pinned ids ascending, then chosen free ids by how many beat them.
    """
    pinned = [j for j in range(nb) if j < n_sink or j >= nb - n_window]
    free = [j for j in range(nb) if j not in pinned]
    slots = k - len(pinned)
    ranked = []
    for j in free:
        beaten = 0
        for i in free:
            if s_row[i] > s_row[j] or (s_row[i] == s_row[j] and i < j):
                beaten += 1
        if beaten < slots:
            ranked.append((beaten, j))
    ranked.sort()
    ids = pinned + [j for _, j in ranked]
    scores = [float(s_row[j]) for j in ids]
    ids += [-1] * (k - len(ids))
    scores += [-np.inf] * (k - len(scores))
    return ids, scores


def check_select_vs_rank_count(orc, cases: int = 150, seed: int = 5) -> None:
    rng = np.random.default_rng(seed)
    for _ in range(cases):
        B = int(rng.integers(1, 4))
        stride = int(rng.integers(1, 13))
        k = int(rng.integers(1, 17))
        n_sink = int(rng.integers(0, k + 1))
        n_window = int(rng.integers(0, k - n_sink + 1))
        seq = rng.integers(0, stride * PAGE + 1, size=B).astype(np.int32)
        s = rng.integers(-3, 4, size=(B, HEADS, stride)).astype(np.float64)
        ids, sc = orc.select(s, seq, k, n_sink, n_window)
        for b in range(B):
            nb = (int(seq[b]) + PAGE - 1) // PAGE
            for h in range(HEADS):
                e_ids, e_sc = rank_count_select(s[b, h], nb, k, n_sink, n_window)
                assert list(ids[b, h]) == e_ids, (b, h, nb, k, n_sink, n_window, list(ids[b, h]), e_ids)
                np.testing.assert_array_equal(sc[b, h], np.asarray(e_sc))


# ----------------------------------------------------------------------------
# invariants
# ----------------------------------------------------------------------------

def check_invariants(orc) -> None:
    w = mixed_workload(21)
    s = orc.block_scores(w.q, w.pool, w.block_table, w.seq_lens)
    nb = w.num_blocks
    for (k, n_sink, n_window) in [(16, 1, 2), (4, 1, 1), (3, 0, 1), (8, 2, 0), (1, 0, 0)]:
        ids, sc = orc.select(s, w.seq_lens, k, n_sink, n_window)
        for b in range(w.batch):
            for h in range(HEADS):
                got = [int(x) for x in ids[b, h] if x >= 0]
                assert len(set(got)) == len(got)
                # fewer than k blocks: every block; else exactly k
                assert len(got) == min(k, int(nb[b]))
                # empty row: nothing
                if nb[b] == 0:
                    assert all(x == -1 for x in ids[b, h])
                    assert np.all(sc[b, h] == -np.inf)
                # pins present, first, increasing
                pins = [j for j in range(int(nb[b])) if j < n_sink or j >= nb[b] - n_window]
                assert got[:len(pins)] == pins
                # scores reported are the block scores
                for r, j in enumerate(got):
                    assert sc[b, h, r] == s[b, h, j]
        # split-merge equals unsplit, every split width
        for W in list(range(1, 18)) + [31, 64, 1000]:
            sids, ssc = orc.select_split(s, w.seq_lens, k, n_sink, n_window, W)
            np.testing.assert_array_equal(sids, ids, err_msg=f"split width {W}")
            np.testing.assert_array_equal(ssc, sc)

    # permuting where the pages live changes nothing
    rng = np.random.default_rng(3)
    perm = rng.permutation(w.num_pages)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.shape[0])
    pool2 = w.pool[perm]
    bt2 = np.where(w.block_table >= 0, inv[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    s2 = orc.block_scores(w.q, pool2, bt2, w.seq_lens)
    np.testing.assert_array_equal(s2, s)

    # scaling q by 2 (exact in bf16) keeps the selection and doubles the scores
    q2 = wl.f32_to_bf16_bits(wl.bf16_bits_to_f32(w.q) * 2.0)
    s3 = orc.block_scores(q2, w.pool, w.block_table, w.seq_lens)
    fin = np.isfinite(s)
    np.testing.assert_array_equal(s3[fin], 2.0 * s[fin])
    ids_a, _ = orc.select(s, w.seq_lens, 16, 1, 2)
    ids_b, _ = orc.select(s3, w.seq_lens, 16, 1, 2)
    np.testing.assert_array_equal(ids_a, ids_b)


# ----------------------------------------------------------------------------
# fp8 E4M3 cache
# ----------------------------------------------------------------------------

def check_e4m3_codes(orc) -> None:
    """Every E4M3 code against torch's float8_e4m3fn decoding, plus closed forms."""
    import torch
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([orc.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    np.testing.assert_array_equal(got[fin], ref[fin])
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9
    assert got[0x08] == 2.0 ** -6 and got[0x07] == 7 * 2.0 ** -9 and got[0xC0] == -2.0


def check_fp8_golden(orc) -> None:
    with open(os.path.join(GOLDEN_DIR, "fp8_per_token_scale.json")) as f:
        fx = json.load(f)
    L = int(fx["seq_len"])
    codes = np.zeros((2, PAGE, DIM), dtype=np.uint8)
    scale = np.ones((2, PAGE), dtype=np.float32)
    codes[:, :, 0] = fx["code_dim0"]
    t = np.arange(PAGE)
    scale[0] = (t % 5) + 1
    scale[1] = 0.5 * ((t % 3) + 1)
    rem = L - PAGE
    codes[1, rem::2, :] = 0x7F
    codes[1, rem + 1::2, :] = 0x7E
    scale[1, rem:] = 1e4
    q = np.zeros((1, HEADS, DIM), dtype=np.float32)
    q[0, :, 0] = fx["alpha"]
    bt = np.array([[0, 1]], dtype=np.int32)
    seq = np.array([L], dtype=np.int32)
    s = orc.block_scores_fp8(wl.f32_to_bf16_bits(q), codes, scale, bt, seq)
    ids, sc = orc.select(s, seq, int(fx["k"]), int(fx["n_sink"]), int(fx["n_window"]))
    np.testing.assert_array_equal(ids, np.asarray(fx["expected_ids"], dtype=np.int32))
    np.testing.assert_array_equal(sc, np.asarray(fx["expected_scores"], dtype=np.float64))


def check_fp8_vs_numpy(orc) -> None:
    import torch
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    w = wl.to_fp8(mixed_workload(13))
    s = orc.block_scores_fp8(w.q, w.pool8, w.kscale, w.block_table, w.seq_lens)
    qf = wl.bf16_bits_to_f32(w.q).astype(np.float64)
    for b in range(w.batch):
        L = int(w.seq_lens[b])
        for j in range((L + PAGE - 1) // PAGE):
            valid = min(PAGE, L - j * PAGE)
            page = int(w.block_table[b, j])
            kf = table[w.pool8[page, :valid]] * w.kscale[page, :valid, None].astype(np.float64)
            ref = (qf[b] @ kf.T).max(axis=1)
            np.testing.assert_allclose(s[b, :, j], ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------
# several query positions per request
# ----------------------------------------------------------------------------

def check_multi_query_golden(orc) -> None:
    with open(os.path.join(GOLDEN_DIR, "multi_query_causal.json")) as f:
        fx = json.load(f)
    L, Q = int(fx["seq_len"]), int(fx["q_len"])
    pool = np.zeros((2, PAGE, DIM), dtype=np.float32)
    for tok, v in fx["planted_dim0"].items():
        t = int(tok)
        pool[t // PAGE, t % PAGE, 0] = v
    q = np.zeros((1, Q, HEADS, DIM), dtype=np.float32)
    q[0, :, :, 0] = np.asarray(fx["alpha"], dtype=np.float32)[None, :]
    s, ids, sel, lens = orc.run_multi(wl.f32_to_bf16_bits(q), wl.f32_to_bf16_bits(pool),
                                      np.array([[0, 1]], dtype=np.int32),
                                      np.array([L], dtype=np.int32), int(fx["k"]),
                                      int(fx["n_sink"]), int(fx["n_window"]))
    assert list(lens[0]) == [127, 128, 129, 130]
    np.testing.assert_array_equal(ids, np.asarray(fx["expected_ids"], dtype=np.int32))
    for i in range(Q):
        for h in range(HEADS):
            row = fx["expected_scores"][0][i][h]
            exp = np.full(int(fx["k"]), -np.inf)
            exp[:len(row)] = row
            np.testing.assert_array_equal(sel[0, i, h], exp, err_msg=f"position {i} head {h}")


def check_multi_query_one_position_is_decode(orc) -> None:
    w = mixed_workload(14)
    s1, ids1, sel1 = orc.run(w)
    s, ids, sel, _ = orc.run_multi(w.q[:, None], w.pool, w.block_table, w.seq_lens, w.k,
                                   w.n_sink, w.n_window)
    np.testing.assert_array_equal(ids[:, 0], ids1)
    np.testing.assert_array_equal(s[:, 0], s1)


def check_multi_query_fp8_golden(orc) -> None:
    """The multi-position fixture on an E4M3 cache: each planted key is coded
    by hand at twice its value (2, 8, 4, 16 -> E4M3 0x40, 0x50, 0x48, 0x58:
    sign 0, biased exponent 8, 10, 9, 11, mantissa 0) with every token scale
    0.5, so the dequantised keys are the fixture's and so are ids and scores."""
    with open(os.path.join(GOLDEN_DIR, "multi_query_causal.json")) as f:
        fx = json.load(f)
    L, Q = int(fx["seq_len"]), int(fx["q_len"])
    code_of_double = {1.0: 0x40, 4.0: 0x50, 2.0: 0x48, 8.0: 0x58}
    codes = np.zeros((2, PAGE, DIM), dtype=np.uint8)
    for tok, v in fx["planted_dim0"].items():
        t = int(tok)
        codes[t // PAGE, t % PAGE, 0] = code_of_double[float(v)]
    scale = np.full((2, PAGE), 0.5, dtype=np.float32)
    q = np.zeros((1, Q, HEADS, DIM), dtype=np.float32)
    q[0, :, :, 0] = np.asarray(fx["alpha"], dtype=np.float32)[None, :]
    s, ids, sel, lens = orc.run_multi(wl.f32_to_bf16_bits(q), None,
                                      np.array([[0, 1]], dtype=np.int32),
                                      np.array([L], dtype=np.int32), int(fx["k"]),
                                      int(fx["n_sink"]), int(fx["n_window"]), pool8=codes,
                                      kscale=scale)
    assert list(lens[0]) == [127, 128, 129, 130]
    np.testing.assert_array_equal(ids, np.asarray(fx["expected_ids"], dtype=np.int32))
    for i in range(Q):
        for h in range(HEADS):
            row = fx["expected_scores"][0][i][h]
            exp = np.full(int(fx["k"]), -np.inf)
            exp[:len(row)] = row
            np.testing.assert_array_equal(sel[0, i, h], exp, err_msg=f"position {i} head {h}")


def check_prefill_matches_multi_query_fixture(orc) -> None:
    """Four new tokens at the end of a 130-token request are the four draft
    positions of the multi-position fixture: the same ids and scores."""
    with open(os.path.join(GOLDEN_DIR, "multi_query_causal.json")) as f:
        fx = json.load(f)
    L, Q = int(fx["seq_len"]), int(fx["q_len"])
    pool = np.zeros((2, PAGE, DIM), dtype=np.float32)
    for tok, v in fx["planted_dim0"].items():
        pool[int(tok) // PAGE, int(tok) % PAGE, 0] = v
    q = np.zeros((Q, HEADS, DIM), dtype=np.float32)
    q[:, :, 0] = np.asarray(fx["alpha"], dtype=np.float32)[None, :]
    s, ids, sel, lens = orc.run_prefill(wl.f32_to_bf16_bits(q), np.array([0, Q]),
                                        wl.f32_to_bf16_bits(pool), np.array([[0, 1]], dtype=np.int32),
                                        np.array([L], dtype=np.int32), int(fx["k"]),
                                        int(fx["n_sink"]), int(fx["n_window"]))
    assert list(lens) == [127, 128, 129, 130]
    np.testing.assert_array_equal(ids, np.asarray(fx["expected_ids"], dtype=np.int32)[0])


def check_prefill_fp8_matches_fixture(orc) -> None:
    """The E4M3 causal fixture through the prefill route: the request's last
    four tokens as new tokens give the fixture's ids and scores."""
    with open(os.path.join(GOLDEN_DIR, "multi_query_causal.json")) as f:
        fx = json.load(f)
    L, Q, k = int(fx["seq_len"]), int(fx["q_len"]), int(fx["k"])
    code_of_double = {1.0: 0x40, 4.0: 0x50, 2.0: 0x48, 8.0: 0x58}
    codes = np.zeros((2, PAGE, DIM), dtype=np.uint8)
    for tok, v in fx["planted_dim0"].items():
        codes[int(tok) // PAGE, int(tok) % PAGE, 0] = code_of_double[float(v)]
    scale = np.full((2, PAGE), 0.5, dtype=np.float32)
    q = np.zeros((Q, HEADS, DIM), dtype=np.float32)
    q[:, :, 0] = np.asarray(fx["alpha"], dtype=np.float32)[None, :]
    s, ids, sel, lens = orc.run_prefill(wl.f32_to_bf16_bits(q), np.array([0, Q]), None,
                                        np.array([[0, 1]], dtype=np.int32),
                                        np.array([L], dtype=np.int32), k, int(fx["n_sink"]),
                                        int(fx["n_window"]), pool8=codes, kscale=scale)
    assert list(lens) == [127, 128, 129, 130]
    np.testing.assert_array_equal(ids, np.asarray(fx["expected_ids"], dtype=np.int32)[0])
    for i in range(Q):
        for h in range(HEADS):
            row = fx["expected_scores"][0][i][h]
            exp = np.full(k, -np.inf)
            exp[:len(row)] = row
            np.testing.assert_array_equal(sel[i, h], exp, err_msg=f"token {i} head {h}")


ALL_CHECKS = (check_golden, check_scores_vs_numpy, check_select_vs_rank_count, check_invariants,
              check_expand_golden, check_expand_invariants, check_e4m3_codes, check_fp8_golden,
              check_fp8_vs_numpy, check_multi_query_golden, check_multi_query_one_position_is_decode,
              check_prefill_matches_multi_query_fixture, check_multi_query_fp8_golden,
              check_prefill_fp8_matches_fixture)
