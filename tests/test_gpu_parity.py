"""CUDA path vs the CPU oracle on identical seeded inputs (through the C ABI)."""

import numpy as np
import pytest

import parity
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import sparse_attention_decode_gb300 as msa
    msa.load()
    return msa


def _compare(orc, w, **kw):
    o_scores, o_ids, _ = orc.run(w, k=kw.get("k"), n_sink=kw.get("n_sink"), n_window=kw.get("n_window"))
    g_ids, g_sc, g_blk, fault = parity.run_gpu(w, **kw)
    assert fault == 0, f"fault word {fault:#x}"
    return parity.check(w, o_scores, o_ids, g_ids, g_sc, g_blk, k=kw.get("k"),
                        n_sink=kw.get("n_sink"), n_window=kw.get("n_window"))


@pytest.mark.parametrize("name", ["tiny", "decode_point", "ragged"])
def test_config_parity(lib, orc, name):
    _compare(orc, wl.make(name))


def test_ragged_permuted_rows(lib, orc):
    _compare(orc, wl.ragged(permute_rows=True))


@pytest.mark.parametrize("split", [64, 0])
def test_adversarial_exact(lib, orc, split):
    """Integer scores: ids, order and scores bit-exact; all winners in one split at W=64."""
    w = wl.adversarial()
    _compare(orc, w, split_blocks=split)


@pytest.mark.slow
def test_long_context_full(lib, orc):
    """B=32 x 128K: the launch configuration the benchmark times (automatic split)."""
    w = wl.long_context()
    _compare(orc, w)


@pytest.mark.parametrize("k,n_sink,n_window", [(1, 0, 0), (1, 1, 0), (2, 0, 1), (3, 1, 1),
                                               (16, 0, 0), (16, 16, 0), (16, 0, 16), (17, 1, 2),
                                               (32, 1, 2), (32, 4, 8)])
def test_k_and_pins(lib, orc, k, n_sink, n_window):
    w = wl.random_workload([1, 127, 128, 129, 2000, 5000, 8700, 0], num_pages=200, seed=31,
                           q_scale=1 / np.sqrt(128), max_model_len=8704)
    _compare(orc, w, k=k, n_sink=n_sink, n_window=n_window)


def _grid_lengths():
    return [1, 127, 128, 129, 256, 1000, 4096, 8699, 8700, 8701, 16384]


@pytest.mark.parametrize("B", [1, 2, 4, 8, 15, 16, 32])
def test_batch_by_length_grid(lib, orc, B):
    """Batch {1..32} x kv_len {1..16384} incl. consecutive decode lengths."""
    lens = _grid_lengths()
    for i, L in enumerate(lens):
        seq = [L] * B if i % 2 == 0 else [lens[(i + r) % len(lens)] for r in range(B)]
        w = wl.random_workload(seq, seed=100 + B * 31 + i, q_scale=1 / np.sqrt(128),
                               max_model_len=16384)
        _compare(orc, w)


def test_split_width_is_bitwise_invariant(lib):
    """Block scores and ids do not depend on how the pages are split over CTAs."""
    for w in (wl.decode_point(), wl.ragged()):
        ref_ids, ref_sc, ref_blk, f0 = parity.run_gpu(w, split_blocks=0)
        assert f0 == 0
        for W in (1, 2, 3, 8, 64, 1024):
            ids, sc, blk, f = parity.run_gpu(w, split_blocks=W)
            assert f == 0
            np.testing.assert_array_equal(blk, ref_blk, err_msg=f"{w.name} W={W}")
            np.testing.assert_array_equal(ids, ref_ids, err_msg=f"{w.name} W={W}")
            np.testing.assert_array_equal(sc, ref_sc, err_msg=f"{w.name} W={W}")


def test_shape_bound_is_bitwise_invariant(lib):
    """Sizing for an 8x larger batch and context bound changes nothing."""
    w = wl.decode_point()
    a = parity.run_gpu(w)
    b = parity.run_gpu(w, max_batch=8 * w.batch, max_model_len=8 * w.max_model_len)
    for x, y in zip(a[:3], b[:3]):
        np.testing.assert_array_equal(x, y)
    assert a[3] == 0 and b[3] == 0


def test_four_and_two_consumer_formats_agree(lib, orc):
    """A one-position bf16 pass of one to 64 pages per SM (decode_point: 16 x 68
    blocks against 152 SMs) runs four consumer warps with one stage each;
    sized for a 16x longer context (16 x 1088 blocks) the same call runs two
    warps with three stages.  Block scores, ids and scores are bit-identical,
    and both match the oracle."""
    w = wl.decode_point()
    a = parity.run_gpu(w)
    b = parity.run_gpu(w, max_model_len=16 * w.max_model_len)
    for x, y in zip(a[:3], b[:3]):
        np.testing.assert_array_equal(x, y)
    assert a[3] == 0 and b[3] == 0
    o_scores, o_ids, _ = orc.run(w)
    parity.check(w, o_scores, o_ids, a[0], a[1], a[2])


def test_graph_replay_with_changed_lengths(lib, orc):
    """Capture once at one set of lengths; replay after changing lengths and tables."""
    import torch
    import sparse_attention_decode_gb300 as msa
    max_len, B, k = 16384, 8, 16
    first = wl.random_workload([4096] * B, num_pages=1024, seed=41, q_scale=1 / np.sqrt(128),
                               max_model_len=max_len)
    q, pool, bt, seq = parity.to_device(first)
    ids = torch.empty((B, 4, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((B, 4, k), dtype=torch.float32, device="cuda")
    ws = msa.new_workspace(B, max_len, k)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        msa.msa_indexer_decode(q, pool, bt, seq, k, 1, 2, ids, sc, ws, max_model_len=max_len)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        msa.msa_indexer_decode(q, pool, bt, seq, k, 1, 2, ids, sc, ws, max_model_len=max_len)
    for seed, lens in ((42, [1, 0, 129, 16384, 700, 8700, 128, 3000]), (43, [16000] * 8)):
        w = wl.random_workload(lens, num_pages=1024, seed=seed, q_scale=1 / np.sqrt(128),
                               max_model_len=max_len)
        q2, pool2, bt2, seq2 = parity.to_device(w)
        q.copy_(q2)
        pool.copy_(pool2)
        bt.copy_(bt2)
        seq.copy_(seq2)
        g.replay()
        torch.cuda.synchronize()
        o_scores, o_ids, _ = orc.run(w)
        parity.check(w, o_scores, o_ids, ids.cpu().numpy(), sc.cpu().numpy())
    assert msa.msa_indexer_get_error(ws) == 0


@pytest.mark.parametrize("page_tokens", [16, 8, 32, 64, 128])
def test_expand_pages_matches_oracle(lib, orc, page_tokens):
    """Selected blocks -> small KV page ids, bit-exact against the oracle's expansion."""
    import torch
    for w in (wl.ragged(), wl.decode_point()):
        ids, sc, blk, fault = parity.run_gpu(w)
        assert fault == 0
        per = 128 // page_tokens
        stride = int(w.num_blocks.max()) * per + 3
        rng = np.random.default_rng(page_tokens)
        kvb = rng.permutation(w.batch * stride).astype(np.int32).reshape(w.batch, stride)
        d_ids = torch.from_numpy(ids).cuda()
        d_seq = torch.from_numpy(w.seq_lens).cuda()
        d_kvb = torch.from_numpy(kvb).cuda()
        pages = torch.full((w.batch, 4, w.k * per), -7, dtype=torch.int32, device="cuda")
        num = torch.full((w.batch, 4), -7, dtype=torch.int32, device="cuda")
        lib.msa_indexer_expand_pages(d_ids, d_seq, d_kvb, pages, num, page_tokens=page_tokens)
        torch.cuda.synchronize()
        e_pages, e_num = orc.expand_pages(ids, w.seq_lens, kvb, page_tokens)
        np.testing.assert_array_equal(num.cpu().numpy(), e_num)
        np.testing.assert_array_equal(pages.cpu().numpy(), e_pages)


@pytest.mark.parametrize("page_tokens", [16, 64])
def test_decode_pages_fused_matches_separate(lib, orc, page_tokens):
    """The page expansion fused into the merge equals decode + msa_indexer_expand_pages."""
    import torch
    for w in (wl.ragged(), wl.decode_point(), wl.tiny()):
        q, pool, bt, seq = parity.to_device(w)
        per = 128 // page_tokens
        stride = int(w.num_blocks.max()) * per + 5
        rng = np.random.default_rng(page_tokens + 1)
        kvb = torch.from_numpy(rng.permutation(w.batch * stride).astype(np.int32)
                               .reshape(w.batch, stride)).cuda()
        B, k = w.batch, w.k
        outs = []
        for fused in (False, True):
            ids = torch.full((B, 4, k), -7, dtype=torch.int32, device="cuda")
            sc = torch.full((B, 4, k), 7.0, dtype=torch.float32, device="cuda")
            pages = torch.full((B, 4, k * per), -7, dtype=torch.int32, device="cuda")
            num = torch.full((B, 4), -7, dtype=torch.int32, device="cuda")
            ws = lib.new_workspace(B, w.max_model_len, k)
            if fused:
                lib.msa_indexer_decode_pages(q, pool, bt, seq, k, w.n_sink, w.n_window, ids, sc, ws,
                                             kvb, pages, num, max_model_len=w.max_model_len,
                                             page_tokens=page_tokens)
            else:
                lib.msa_indexer_decode(q, pool, bt, seq, k, w.n_sink, w.n_window, ids, sc, ws,
                                       max_model_len=w.max_model_len)
                lib.msa_indexer_expand_pages(ids, seq, kvb, pages, num, page_tokens=page_tokens)
            torch.cuda.synchronize()
            assert lib.msa_indexer_get_error(ws) == 0
            outs.append([t.cpu().numpy() for t in (ids, sc, pages, num)])
        for a, b in zip(*outs):
            np.testing.assert_array_equal(a, b)
        e_pages, e_num = orc.expand_pages(outs[1][0], w.seq_lens, kvb.cpu().numpy(), page_tokens)
        np.testing.assert_array_equal(outs[1][2], e_pages)
        np.testing.assert_array_equal(outs[1][3], e_num)


def test_max_batch(lib, orc):
    """The largest batch the library accepts (MSA_MAX_BATCH = 4096 requests),
    short ragged lengths with empty requests: the per-request prefix in shared
    memory, chunks spanning many requests and the merge grid at their limits."""
    rng = np.random.default_rng(4096)
    seq = rng.integers(0, 400, 4096)
    seq[rng.random(4096) < 0.05] = 0
    w = wl.random_workload(seq, seed=4096, q_scale=1 / np.sqrt(128), max_model_len=512,
                           name="max_batch")
    _compare(orc, w)


@pytest.mark.parametrize("case", ["decode_point", "ragged", "k32", "split1", "b256", "b200_split3",
                                  "b257", "max_batch"])
def test_decode_equals_its_two_stages(lib, case):
    """msa_indexer_decode and msa_indexer_score followed by msa_indexer_merge
    must give bitwise-identical ids, scores and block scores, alternating on
    one workspace (split 1 gives the long request up to 1024 lists).  Up to
    256 requests the decode call's merge derives each request's page range and
    the pass's chunking from the lengths itself, while the separate merge
    reads what the score pass left in the workspace: b256 and b200_split3
    (a forced split) take the first way over several warps of lengths, b257
    and max_batch the second."""
    import torch
    k, split = 16, 0
    if case in ("decode_point", "ragged"):
        w = wl.make(case)
    elif case == "k32":
        w, k = wl.decode_point(), 32
    elif case == "split1":
        w, split = wl.ragged(), 1  # up to 1024 lists for the long request
    elif case in ("b256", "b200_split3", "b257"):
        B = {"b256": 256, "b200_split3": 200, "b257": 257}[case]
        rng = np.random.default_rng(B)
        seq = rng.integers(0, 5000, B)
        seq[rng.random(B) < 0.05] = 0
        w = wl.random_workload(seq, seed=B, q_scale=1 / np.sqrt(128), max_model_len=8192)
        split = 3 if case == "b200_split3" else 0
    else:
        rng = np.random.default_rng(7)
        seq = rng.integers(0, 3000, 1500)
        seq[rng.random(1500) < 0.05] = 0
        w = wl.random_workload(seq, seed=7, q_scale=1 / np.sqrt(128), max_model_len=4096)
    q, pool, bt, seq = parity.to_device(w)
    B, S = w.batch, w.bt_stride
    ws = lib.new_workspace(B, w.max_model_len, k, split)
    outs = []
    for fused in (True, False, True):
        ids = torch.full((B, 4, k), -7, dtype=torch.int32, device="cuda")
        sc = torch.full((B, 4, k), 7.0, dtype=torch.float32, device="cuda")
        blk = torch.full((B, 4, S), float("nan"), dtype=torch.float32, device="cuda")
        if fused:
            lib.msa_indexer_decode(q, pool, bt, seq, k, 1, 2, ids, sc, ws,
                                   max_model_len=w.max_model_len, out_block_scores=blk,
                                   split_blocks=split)
        else:
            lib.msa_indexer_score(q, pool, bt, seq, k, 1, 2, ws, max_model_len=w.max_model_len,
                                  out_block_scores=blk, split_blocks=split)
            lib.msa_indexer_merge(B, k, ids, sc, ws)
        outs.append([t.cpu().numpy() for t in (ids, sc, blk)])
    assert lib.msa_indexer_get_error(ws) == 0
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            np.testing.assert_array_equal(a, b)


def test_one_workspace_across_changing_batches(lib):
    """A serving loop calls the indexer with a different batch every step on
    one workspace sized for the largest.  The state one call leaves for the
    next (ticket and arrival counters) must not depend on where the batch-sized
    regions of the workspace fall, so each call equals the same call on a fresh
    workspace, bit for bit."""
    max_batch, max_len, k = 300, 4096, 16
    ws = lib.new_workspace(max_batch, max_len, k)
    rng = np.random.default_rng(11)
    for step, B in enumerate([16, 3, 300, 1, 77, 300, 16]):
        seq = rng.integers(0, max_len + 1, B)
        w = wl.random_workload(seq, seed=500 + step, q_scale=1 / np.sqrt(128), max_model_len=max_len)
        shared = parity.run_gpu(w, ws=ws, max_batch=max_batch)
        fresh = parity.run_gpu(w, max_batch=max_batch)
        assert shared[3] == 0 and fresh[3] == 0
        for a, b in zip(shared[:3], fresh[:3]):
            np.testing.assert_array_equal(a, b, err_msg=f"step {step} B={B}")


def test_million_token_request(lib, orc):
    """One request of 2^20 tokens beside short and empty ones: its 8192 pages
    spread over every CTA, so the merge folds more lists than one staged tile
    holds."""
    w = wl.random_workload([1 << 20, 3000, 0, 129], seed=77, q_scale=1 / np.sqrt(128),
                           max_model_len=1 << 20)
    _compare(orc, w)
