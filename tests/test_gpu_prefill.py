"""Prefill scoring (every new token over its own causal prefix) against the oracle.

Request b appends n_b new tokens to a cache of seq_len_b tokens that already
holds them; new token t sees the first seq_len_b - n_b + t + 1 tokens (the
prefill branch of vLLM PR #57832 scores the prefill query rows with
cu_seqlens_q).  Each row is checked like a decode query of that length.
"""

import numpy as np
import pytest

import parity
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    import sparse_attention_decode_gb300 as m
    m.load()
    return m


def prefill_case(pairs, seed, *, ternary=False, max_model_len=None, num_pages=None):
    """(n_new, seq_len) per request -> (workload, q bits [total_q,4,128], cu_seqlens_q)."""
    lens = [L for _, L in pairs]
    w = wl.random_workload(lens, seed=seed, q_scale=1 / np.sqrt(128),
                           max_model_len=max_model_len, num_pages=num_pages, poison=not ternary)
    rng = np.random.default_rng(seed + 991)
    total = sum(n for n, _ in pairs)
    if ternary:
        q = wl._ternary_bits(rng, (total, 4, 128))
        w.pool = wl._ternary_pool(rng, w.num_pages)
        wl.poison_tails(w.pool, w.block_table, w.seq_lens)
    else:
        q = wl.f32_to_bf16_bits(rng.standard_normal((total, 4, 128), dtype=np.float32)
                                / np.float32(np.sqrt(128)))
    cu = np.zeros(len(pairs) + 1, dtype=np.int32)
    cu[1:] = np.cumsum([n for n, _ in pairs])
    return w, q, cu


def run_prefill(msa, w, q_bits, cu, k=16, n_sink=1, n_window=2, block_scores=True, ws_pad=0,
                ws=None):
    import torch
    total = q_bits.shape[0]
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    pool = torch.from_numpy(w.pool.view(np.int16)).view(torch.bfloat16).cuda()
    bt = torch.from_numpy(w.block_table).cuda()
    seq = torch.from_numpy(w.seq_lens).cuda()
    d_cu = torch.from_numpy(cu).cuda()
    ids = torch.full((total, 4, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((total, 4, k), 7.0, dtype=torch.float32, device="cuda")
    stride = (w.max_model_len + 127) // 128
    blk = None
    if block_scores:
        blk = torch.full((total, 4, stride), float("nan"), dtype=torch.float32, device="cuda")
    if ws is None:
        n = msa.msa_indexer_prefill_workspace_bytes(total, w.max_model_len)
        ws = torch.zeros(n + ws_pad, dtype=torch.uint8, device="cuda")
    msa.msa_indexer_prefill(q, d_cu, pool, bt, seq, k, n_sink, n_window, ids, sc, ws,
                            max_model_len=w.max_model_len, out_block_scores=blk)
    fault = msa.msa_indexer_get_error(ws)
    return (ids.cpu().numpy(), sc.cpu().numpy(), None if blk is None else blk.cpu().numpy(),
            fault, ws)


def check_prefill(orc, w, q_bits, cu, got, k=16, n_sink=1, n_window=2, exact=False):
    s, o_ids, _, lens = orc.run_prefill(q_bits, cu, w.pool, w.block_table, w.seq_lens, k,
                                        n_sink, n_window)
    rows_bt = np.repeat(w.block_table, np.diff(cu), axis=0)
    rows = wl.Workload(name=f"{w.name}_prefill", q=q_bits, pool=w.pool, block_table=rows_bt,
                       seq_lens=lens, k=k, n_sink=n_sink, n_window=n_window,
                       max_model_len=w.max_model_len)
    g_ids, g_sc, g_blk = got[:3]
    stride = rows.bt_stride
    return parity.check(rows, s[:, :, :stride], o_ids, g_ids, g_sc,
                        None if g_blk is None else g_blk[:, :, :stride], k=k, n_sink=n_sink,
                        n_window=n_window, exact=exact)


MIXED = [(1, 1), (3, 3), (32, 300), (33, 129), (100, 300), (0, 50), (1, 5000), (64, 256),
         (31, 31), (128, 128), (129, 4000)]


def test_prefill_mixed_batch(msa, orc):
    """Whole prompts, chunked prefill tails and single tokens in one batch; tiles cut mid-request."""
    w, q, cu = prefill_case(MIXED, seed=200, max_model_len=8192)
    got = run_prefill(msa, w, q, cu)
    assert got[3] == 0
    check_prefill(orc, w, q, cu, got)


@pytest.mark.parametrize("pairs", [[(700, 8000)], [(1000, 1000), (257, 16384)],
                                   [(17, 16384)] * 6])
def test_prefill_long(msa, orc, pairs):
    w, q, cu = prefill_case(pairs, seed=210 + len(pairs), max_model_len=16384)
    got = run_prefill(msa, w, q, cu)
    assert got[3] == 0
    check_prefill(orc, w, q, cu, got)


def test_prefill_exact_integers(msa, orc):
    """Ternary q and keys: integer scores with many ties; ids, order and scores bit-exact."""
    pairs = [(96, 3000), (40, 40), (1, 129), (65, 2049)]
    w, q, cu = prefill_case(pairs, seed=220, ternary=True, max_model_len=4096)
    got = run_prefill(msa, w, q, cu, k=32, n_sink=2, n_window=3)
    assert got[3] == 0
    check_prefill(orc, w, q, cu, got, k=32, n_sink=2, n_window=3, exact=True)


@pytest.mark.parametrize("k,n_sink,n_window", [(1, 0, 0), (1, 1, 0), (16, 16, 0), (16, 0, 16),
                                               (17, 1, 2), (32, 4, 8)])
def test_prefill_k_and_pins(msa, orc, k, n_sink, n_window):
    w, q, cu = prefill_case(MIXED, seed=230 + k, max_model_len=8192)
    got = run_prefill(msa, w, q, cu, k=k, n_sink=n_sink, n_window=n_window, block_scores=False)
    assert got[3] == 0
    check_prefill(orc, w, q, cu, got, k=k, n_sink=n_sink, n_window=n_window)


def test_prefill_workspace_scores_equal_caller_buffer(msa):
    """Block scores kept in the workspace give the same selection as a caller buffer."""
    w, q, cu = prefill_case(MIXED, seed=240, max_model_len=8192)
    a = run_prefill(msa, w, q, cu)
    b = run_prefill(msa, w, q, cu, block_scores=False)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_prefill_last_token_matches_decode(msa):
    """The last new token of each request is the decode query at that length."""
    pairs = [(50, 3000), (1, 700), (200, 200), (33, 8191)]
    w, q, cu = prefill_case(pairs, seed=250, max_model_len=8192)
    p_ids, p_sc, p_blk, fault, _ = run_prefill(msa, w, q, cu)
    assert fault == 0
    last = cu[1:] - 1
    dec = wl.Workload(name="last", q=q[last], pool=w.pool, block_table=w.block_table,
                      seq_lens=w.seq_lens, k=16, n_sink=1, n_window=2,
                      max_model_len=w.max_model_len)
    d_ids, d_sc, d_blk, dfault = parity.run_gpu(dec)
    assert dfault == 0
    parity.check(dec, d_blk.astype(np.float64), d_ids, p_ids[last], p_sc[last], p_blk[last])


def test_prefill_bad_page_and_bad_rows(msa, orc):
    """A bad page is skipped and reported; a request with more new tokens than tokens is emptied."""
    pairs = [(40, 1000), (10, 600), (5, 300)]
    w, q, cu = prefill_case(pairs, seed=260, max_model_len=2048, num_pages=40)
    good_page = int(w.block_table[0, 3])
    w.block_table[0, 3] = w.num_pages + 5
    ids, sc, blk, fault, _ = run_prefill(msa, w, q, cu)
    assert fault & msa.MSA_FAULT_PAGE_ID
    r0 = np.arange(cu[0], cu[1])
    assert np.isneginf(blk[r0][:, :, 3]).all()
    assert not (ids[r0] == 3).any()
    # the other requests (pages are not shared) match the oracle on the clean table
    w.block_table[0, 3] = good_page
    s, o_ids, _, lens = orc.run_prefill(q, cu, w.pool, w.block_table, w.seq_lens, 16, 1, 2)
    rows = np.arange(cu[1], cu[3])
    sub = wl.Workload(name="rows_1_2", q=q[rows], pool=w.pool,
                      block_table=np.repeat(w.block_table[1:], np.diff(cu)[1:], axis=0),
                      seq_lens=lens[rows], max_model_len=w.max_model_len)
    st = sub.bt_stride
    parity.check(sub, s[rows][:, :, :st], o_ids[rows], ids[rows], sc[rows], blk[rows][:, :, :st])
    # n_new > seq_len: the request is refused
    w2, q2, cu2 = prefill_case([(8, 100), (4, 200)], seed=261, max_model_len=1024)
    w2.seq_lens[1] = 3
    ids2, sc2, _, fault2, _ = run_prefill(msa, w2, q2, cu2)
    assert fault2 & msa.MSA_FAULT_SEQ_LEN
    assert (ids2[8:] == -1).all() and np.isneginf(sc2[8:]).all()
    assert (ids2[:8, :, 0] >= 0).all()


def test_prefill_waits_that_run_out_empty_every_row(msa, orc):
    """The bounded-wait hook on the prefill path, made without any fault: while
    it is set the bf16 scoring kernel loads no query row and no page (no copy
    is ever in flight), so its first waits run out after the short poll limit.
    The call must return and report MSA_FAULT_TIMEOUT, and its top-k must write
    every row empty although some block scores were never written.  The same
    workspace then matches the oracle twice (the pass count and the finish
    counter in its header were left consistent); the E4M3 prefill is refused
    while the hook is set."""
    import torch
    w, q, cu = prefill_case(MIXED, seed=262, max_model_len=8192)
    total = q.shape[0]
    ws = torch.zeros(msa.msa_indexer_prefill_workspace_bytes(total, w.max_model_len),
                     dtype=torch.uint8, device="cuda")
    msa.msa_indexer_test_withhold_pages(True)
    try:
        ids, sc, _, fault, _ = run_prefill(msa, w, q, cu, ws=ws)
        codes = torch.zeros((w.num_pages, 128, 128), dtype=torch.uint8, device="cuda")
        scales = torch.ones((w.num_pages, 128), dtype=torch.float32, device="cuda")
        d = [torch.from_numpy(x).cuda() for x in (w.block_table, w.seq_lens, cu)]
        qd = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).cuda()
        out_i = torch.empty((total, 4, 16), dtype=torch.int32, device="cuda")
        out_s = torch.empty((total, 4, 16), dtype=torch.float32, device="cuda")
        with pytest.raises(msa.MsaError) as e:
            msa.msa_indexer_prefill_fp8(qd, d[2], codes, scales, d[0], d[1], 16, 1, 2, out_i, out_s,
                                        ws, max_model_len=w.max_model_len)
        assert e.value.status == msa.MSA_ERR_UNSUPPORTED
    finally:
        msa.msa_indexer_test_withhold_pages(False)
    assert fault & msa.MSA_FAULT_TIMEOUT
    assert (ids == -1).all() and np.isneginf(sc).all()
    for _ in range(2):
        got = run_prefill(msa, w, q, cu, ws=ws)
        assert got[3] == 0
        check_prefill(orc, w, q, cu, got)


def test_prefill_outputs_do_not_spill(msa):
    import torch
    w, q, cu = prefill_case(MIXED, seed=270, max_model_len=8192)
    total, k, pad = q.shape[0], 16, 4096
    d = parity.to_device(w)
    ids = torch.full((total * 4 * k + pad,), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((total * 4 * k + pad,), 7.0, dtype=torch.float32, device="cuda")
    n = msa.msa_indexer_prefill_workspace_bytes(total, w.max_model_len)
    ws = torch.zeros(n + pad, dtype=torch.uint8, device="cuda")
    ws[n:] = 0xA5
    qd = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).cuda()
    msa.msa_indexer_prefill(qd, torch.from_numpy(cu).cuda(), d[1], d[2], d[3], k, 1, 2,
                            ids[:total * 4 * k], sc[:total * 4 * k], ws[:n],
                            max_model_len=w.max_model_len)
    torch.cuda.synchronize()
    assert (ids[total * 4 * k:] == -7).all() and (sc[total * 4 * k:] == 7.0).all()
    assert (ws[n:] == 0xA5).all()


def test_prefill_score_only_entry_matches(msa):
    """msa_indexer_prefill_score writes the same block scores as msa_indexer_prefill."""
    import torch
    w, q, cu = prefill_case(MIXED, seed=280, max_model_len=8192)
    ids, sc, blk, fault, _ = run_prefill(msa, w, q, cu)
    assert fault == 0
    total = q.shape[0]
    d = parity.to_device(w)
    out = torch.full((total, 4, (w.max_model_len + 127) // 128), float("nan"), dtype=torch.float32,
                     device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    msa.msa_indexer_prefill_score(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).cuda(),
                                  torch.from_numpy(cu).cuda(), d[1], d[2], d[3], out, ws,
                                  max_model_len=w.max_model_len)
    assert msa.msa_indexer_get_error(ws) == 0
    np.testing.assert_array_equal(out.cpu().numpy(), blk)


def test_prefill_graph_replay_with_changed_batches(msa, orc):
    """Captured once; replayed after new lengths, row splits, tables and queries (same total_q)."""
    import torch
    total, max_len, k = 300, 16384, 16
    first = [(100, 9000), (200, 4000)]
    w, q, cu = prefill_case(first, seed=300, max_model_len=max_len, num_pages=400)
    d_q = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).cuda()
    d_pool = torch.from_numpy(w.pool.view(np.int16)).view(torch.bfloat16).cuda()
    d_bt = torch.zeros((3, w.bt_stride), dtype=torch.int32, device="cuda")
    d_bt[:2].copy_(torch.from_numpy(w.block_table))
    d_seq = torch.zeros(3, dtype=torch.int32, device="cuda")
    d_seq[:2].copy_(torch.from_numpy(w.seq_lens))
    d_cu = torch.tensor([0, 100, 300, 300], dtype=torch.int32, device="cuda")
    ids = torch.empty((total, 4, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((total, 4, k), dtype=torch.float32, device="cuda")
    ws = torch.zeros(msa.msa_indexer_prefill_workspace_bytes(total, max_len), dtype=torch.uint8,
                     device="cuda")

    def call():
        msa.msa_indexer_prefill(d_q, d_cu, d_pool, d_bt, d_seq, k, 1, 2, ids, sc, ws,
                                max_model_len=max_len)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for seed, pairs in ((301, [(1, 1), (64, 16384), (235, 700)]), (302, [(300, 12000), (0, 5), (0, 0)])):
        w2, q2, cu2 = prefill_case(pairs, seed=seed, max_model_len=max_len, num_pages=400)
        assert q2.shape[0] == total
        d_q.copy_(torch.from_numpy(q2.view(np.int16)).view(torch.bfloat16))
        d_pool.copy_(torch.from_numpy(w2.pool.view(np.int16)).view(torch.bfloat16))
        d_bt.copy_(torch.from_numpy(w2.block_table))
        d_seq.copy_(torch.from_numpy(w2.seq_lens))
        d_cu.copy_(torch.from_numpy(cu2))
        g.replay()
        torch.cuda.synchronize()
        check_prefill(orc, w2, q2, cu2, (ids.cpu().numpy(), sc.cpu().numpy(), None))
    assert msa.msa_indexer_get_error(ws) == 0


def test_prefill_without_rows(msa):
    """total_q = 0: the call succeeds and writes nothing."""
    import torch
    w, q, cu = prefill_case([(4, 300)], seed=310, max_model_len=1024)
    d = parity.to_device(w)
    q0 = torch.empty((0, 4, 128), dtype=torch.bfloat16, device="cuda")
    cu0 = torch.zeros(2, dtype=torch.int32, device="cuda")
    ids = torch.full((4,), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((4,), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    msa.msa_indexer_prefill(q0, cu0, d[1], d[2], d[3], 16, 1, 2, ids, sc, ws,
                            max_model_len=w.max_model_len)
    torch.cuda.synchronize()
    assert (ids == -7).all() and (sc == 7.0).all()
    assert msa.msa_indexer_get_error(ws) == 0


@pytest.mark.slow
def test_prefill_bench_workload_sampled_rows(msa, orc):
    """The benchmarked prefill (4 x 2048 new tokens at 128K, the launch bench.py
    times) on the GPU; sampled rows checked one by one against the oracle."""
    import bench
    w, q, cu = bench.prefill_workload()
    got = run_prefill(msa, w, q, cu)
    assert got[3] == 0
    total = q.shape[0]
    rng = np.random.default_rng(400)
    firsts, lasts = cu[:-1], cu[1:] - 1
    rows = np.unique(np.concatenate([firsts, lasts, rng.choice(total, 16, replace=False)]))
    req = np.searchsorted(cu, rows, side="right") - 1
    lens = (w.seq_lens[req] - np.diff(cu)[req] + (rows - cu[req]) + 1).astype(np.int32)
    bt_rows = w.block_table[req]
    s = orc.block_scores(q[rows], w.pool, bt_rows, lens)
    o_ids, _ = orc.select(s, lens, w.k, w.n_sink, w.n_window)
    sub = wl.Workload(name="bench_prefill_rows", q=q[rows], pool=w.pool, block_table=bt_rows,
                      seq_lens=lens, k=w.k, n_sink=w.n_sink, n_window=w.n_window,
                      max_model_len=w.max_model_len)
    st = sub.bt_stride
    parity.check(sub, s[:, :, :st], o_ids, got[0][rows], got[1][rows], got[2][rows][:, :, :st])


def _many_pairs(seed, count=200, max_new=24, max_len=2000):
    rng = np.random.default_rng(seed)
    pairs = []
    for _ in range(count):
        n = int(rng.integers(0, max_new + 1))
        pairs.append((n, int(rng.integers(max(n, 1), max_len + 1))))
    return pairs


def test_prefill_many_requests(msa, orc):
    """200 short ragged requests (some with no new tokens): most CTA ranges
    cross request boundaries, walked last tile first."""
    w, q, cu = prefill_case(_many_pairs(500), seed=501, max_model_len=2048)
    got = run_prefill(msa, w, q, cu)
    assert got[3] == 0
    check_prefill(orc, w, q, cu, got)


@pytest.mark.parametrize("max_len", [139264, 139392])
def test_prefill_rows_just_past_one_group(msa, orc, max_len):
    """Rows just past one group of 1024 blocks (a 128K context with a few
    thousand new tokens): a second group of 1 to 64 blocks; rows of exactly
    1024 and 1088 blocks sit on either side.  A row stride of 1089 blocks
    takes the plain-load path."""
    pairs = [(32, 133000), (8, 139264), (2, 131073)]
    w, q, cu = prefill_case(pairs, seed=310 + max_len % 11, max_model_len=max_len)
    got = run_prefill(msa, w, q, cu)
    assert got[3] == 0
    check_prefill(orc, w, q, cu, got)


@pytest.mark.parametrize("max_len,k", [(300032, 16), (300160, 16), (300032, 32)])
def test_prefill_rows_longer_than_one_group(msa, orc, max_len, k):
    """Rows of more than 1024 blocks (contexts past 128K tokens): the per-row
    top-k takes them 1024 at a time, the first group copied ahead into shared
    memory and later ones loaded in place.  A row stride of 2345 blocks (not a
    multiple of four) takes the plain-load path instead of 16-byte copies."""
    pairs = [(24, 300000), (8, 140001), (4, 1000)]
    w, q, cu = prefill_case(pairs, seed=290 + k + max_len % 7, max_model_len=max_len)
    got = run_prefill(msa, w, q, cu, k=k)
    assert got[3] == 0
    check_prefill(orc, w, q, cu, got, k=k)
