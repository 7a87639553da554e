"""Several query positions per request (speculative verify) against the oracle."""

import json
import os

import numpy as np
import pytest

import parity
import workloads as wl

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def msa():
    import sparse_attention_decode_gb300 as m
    m.load()
    return m


def multi_workload(seq_lens, q_len, seed, **kw):
    w = wl.random_workload(seq_lens, seed=seed, q_scale=1 / np.sqrt(128), **kw)
    rng = np.random.default_rng(seed + 77)
    q = rng.standard_normal((w.batch, q_len, 4, 128), dtype=np.float32) / np.float32(np.sqrt(128))
    return w, wl.f32_to_bf16_bits(q)


def run_mq(msa, w, q_bits, q_len, k=16, n_sink=1, n_window=2, split_blocks=0):
    import torch
    B = w.batch
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    pool = torch.from_numpy(w.pool.view(np.int16)).view(torch.bfloat16).cuda()
    bt = torch.from_numpy(w.block_table).cuda()
    seq = torch.from_numpy(w.seq_lens).cuda()
    ids = torch.full((B, q_len, 4, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((B, q_len, 4, k), 7.0, dtype=torch.float32, device="cuda")
    blk = torch.full((B, q_len, 4, w.bt_stride), float("nan"), dtype=torch.float32, device="cuda")
    ws = msa.new_workspace(B, w.max_model_len, k, split_blocks, q_len=q_len)
    msa.msa_indexer_decode_mq(q, pool, bt, seq, k, n_sink, n_window, ids, sc, ws,
                              max_model_len=w.max_model_len, out_block_scores=blk,
                              split_blocks=split_blocks)
    assert msa.msa_indexer_get_error(ws) == 0
    return ids.cpu().numpy(), sc.cpu().numpy(), blk.cpu().numpy()


def check_rows(orc, w, q_bits, q_len, got, k=16, n_sink=1, n_window=2):
    s, o_ids, _, lens = orc.run_multi(q_bits, w.pool, w.block_table, w.seq_lens, k, n_sink,
                                      n_window)
    B = w.batch
    rows = wl.Workload(name=f"{w.name}_q{q_len}", q=q_bits.reshape(B * q_len, 4, 128),
                       pool=w.pool, block_table=np.repeat(w.block_table, q_len, axis=0),
                       seq_lens=lens.reshape(-1), k=k, n_sink=n_sink, n_window=n_window,
                       max_model_len=w.max_model_len)
    g_ids, g_sc, g_blk = got
    stride = w.bt_stride
    parity.check(rows, s.reshape(B * q_len, 4, stride), o_ids.reshape(B * q_len, 4, k),
                 g_ids.reshape(B * q_len, 4, k), g_sc.reshape(B * q_len, 4, k),
                 g_blk.reshape(B * q_len, 4, stride))


@pytest.mark.parametrize("q_len", [1, 2, 4])
def test_multi_query_parity(msa, orc, q_len):
    lens = [1, 2, 3, 4, 5, 127, 128, 129, 130, 131, 255, 256, 257, 3000, 8700, 0]
    w, q = multi_workload(lens, q_len, seed=60 + q_len, num_pages=300, max_model_len=8704)
    check_rows(orc, w, q, q_len, run_mq(msa, w, q, q_len))


@pytest.mark.parametrize("q_len", [2, 4])
def test_multi_query_long_rows(msa, orc, q_len):
    w, q = multi_workload([131072, 70000, 129, 1024], q_len, seed=70 + q_len, num_pages=1700,
                          max_model_len=131072)
    check_rows(orc, w, q, q_len, run_mq(msa, w, q, q_len))


def test_multi_query_split_invariance(msa):
    w, q = multi_workload([8700] * 8 + [1000] * 8, 4, seed=80, num_pages=700, max_model_len=8704)
    ref = run_mq(msa, w, q, 4)
    for W in (1, 5, 64):
        got = run_mq(msa, w, q, 4, split_blocks=W)
        for x, y in zip(ref, got):
            np.testing.assert_array_equal(x, y)


def test_one_position_equals_decode(msa):
    w = wl.decode_point()
    ids, sc, blk, _ = parity.run_gpu(w)
    got = run_mq(msa, w, w.q[:, None], 1)
    np.testing.assert_array_equal(got[0][:, 0], ids)
    np.testing.assert_array_equal(got[1][:, 0], sc)


def test_multi_query_golden_on_gpu(msa):
    """The hand-derived causal fixture, exact (all scores are exact products)."""
    with open(os.path.join(GOLDEN, "multi_query_causal.json")) as f:
        fx = json.load(f)
    L, Q, k = int(fx["seq_len"]), int(fx["q_len"]), int(fx["k"])
    pool = np.zeros((2, 128, 128), dtype=np.float32)
    for tok, v in fx["planted_dim0"].items():
        pool[int(tok) // 128, int(tok) % 128, 0] = v
    q = np.zeros((1, Q, 4, 128), dtype=np.float32)
    q[0, :, :, 0] = np.asarray(fx["alpha"], dtype=np.float32)[None, :]
    w = wl.Workload(name="golden_mq", q=wl.f32_to_bf16_bits(q[:, 0]), pool=wl.f32_to_bf16_bits(pool),
                    block_table=np.array([[0, 1]], dtype=np.int32),
                    seq_lens=np.array([L], dtype=np.int32), k=k, n_sink=0, n_window=0,
                    max_model_len=256)
    ids, sc, _ = run_mq(msa, w, wl.f32_to_bf16_bits(q), Q, k=k, n_sink=0, n_window=0)
    np.testing.assert_array_equal(ids, np.asarray(fx["expected_ids"], dtype=np.int32))
    for i in range(Q):
        for h in range(4):
            row = fx["expected_scores"][0][i][h]
            exp = np.full(k, -np.inf)
            exp[:len(row)] = row
            np.testing.assert_array_equal(sc[0, i, h].astype(np.float64), exp)


def run_mq_fp8(msa, w8, q_bits, q_len, k=16, n_sink=1, n_window=2, split_blocks=0):
    import torch
    B = w8.batch
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    pool8 = torch.from_numpy(w8.pool8).cuda()
    ks = torch.from_numpy(w8.kscale).cuda()
    bt = torch.from_numpy(w8.block_table).cuda()
    seq = torch.from_numpy(w8.seq_lens).cuda()
    ids = torch.full((B, q_len, 4, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((B, q_len, 4, k), 7.0, dtype=torch.float32, device="cuda")
    blk = torch.full((B, q_len, 4, w8.bt_stride), float("nan"), dtype=torch.float32, device="cuda")
    ws = msa.new_workspace(B, w8.max_model_len, k, split_blocks, q_len=q_len)
    msa.msa_indexer_decode_mq_fp8(q, pool8, ks, bt, seq, k, n_sink, n_window, ids, sc, ws,
                                  max_model_len=w8.max_model_len, out_block_scores=blk,
                                  split_blocks=split_blocks)
    assert msa.msa_indexer_get_error(ws) == 0
    return ids.cpu().numpy(), sc.cpu().numpy(), blk.cpu().numpy()


def check_rows_fp8(orc, w8, q_bits, q_len, got, k=16, n_sink=1, n_window=2):
    s, o_ids, _, lens = orc.run_multi(q_bits, None, w8.block_table, w8.seq_lens, k, n_sink,
                                      n_window, pool8=w8.pool8, kscale=w8.kscale)
    B = w8.batch
    rows = wl.Workload(name=f"{w8.name}_q{q_len}", q=q_bits.reshape(B * q_len, 4, 128),
                       pool=None, block_table=np.repeat(w8.block_table, q_len, axis=0),
                       seq_lens=lens.reshape(-1), k=k, n_sink=n_sink, n_window=n_window,
                       max_model_len=w8.max_model_len)
    g_ids, g_sc, g_blk = got
    stride = w8.bt_stride
    parity.check(rows, s.reshape(B * q_len, 4, stride), o_ids.reshape(B * q_len, 4, k),
                 g_ids.reshape(B * q_len, 4, k), g_sc.reshape(B * q_len, 4, k),
                 g_blk.reshape(B * q_len, 4, stride))


@pytest.mark.parametrize("q_len", [1, 2, 4])
def test_multi_query_fp8_parity(msa, orc, q_len):
    lens = [1, 2, 3, 4, 5, 127, 128, 129, 130, 131, 255, 256, 257, 3000, 8700, 0]
    w, q = multi_workload(lens, q_len, seed=90 + q_len, num_pages=300, max_model_len=8704)
    w8 = wl.to_fp8(w)
    check_rows_fp8(orc, w8, q, q_len, run_mq_fp8(msa, w8, q, q_len))


@pytest.mark.parametrize("k", [16, 32])
def test_multi_query_fp8_long_rows(msa, orc, k):
    w, q = multi_workload([131072, 70000, 129, 1024], 4, seed=95, num_pages=1700,
                          max_model_len=131072)
    w8 = wl.to_fp8(w)
    check_rows_fp8(orc, w8, q, 4, run_mq_fp8(msa, w8, q, 4, k=k, n_sink=2, n_window=3), k=k,
                   n_sink=2, n_window=3)


def test_multi_query_fp8_one_position_equals_decode_fp8(msa):
    import torch
    w8 = wl.to_fp8(wl.decode_point())
    ids1, sc1, blk1, f = parity.run_gpu(w8)
    assert f == 0
    got = run_mq_fp8(msa, w8, w8.q[:, None], 1)
    np.testing.assert_array_equal(got[0][:, 0], ids1)
    np.testing.assert_array_equal(got[1][:, 0], sc1)
    np.testing.assert_array_equal(got[2][:, 0], blk1)


def test_multi_query_fp8_golden_on_gpu(msa):
    """The hand-coded E4M3 version of the causal fixture, exact."""
    with open(os.path.join(GOLDEN, "multi_query_causal.json")) as f:
        fx = json.load(f)
    L, Q, k = int(fx["seq_len"]), int(fx["q_len"]), int(fx["k"])
    code_of_double = {1.0: 0x40, 4.0: 0x50, 2.0: 0x48, 8.0: 0x58}
    codes = np.zeros((2, 128, 128), dtype=np.uint8)
    for tok, v in fx["planted_dim0"].items():
        codes[int(tok) // 128, int(tok) % 128, 0] = code_of_double[float(v)]
    q = np.zeros((1, Q, 4, 128), dtype=np.float32)
    q[0, :, :, 0] = np.asarray(fx["alpha"], dtype=np.float32)[None, :]
    w8 = wl.Workload(name="golden_mq_fp8", q=wl.f32_to_bf16_bits(q[:, 0]), pool=None,
                     block_table=np.array([[0, 1]], dtype=np.int32),
                     seq_lens=np.array([L], dtype=np.int32), k=k, n_sink=0, n_window=0,
                     max_model_len=256, pool8=codes,
                     kscale=np.full((2, 128), 0.5, dtype=np.float32))
    ids, sc, _ = run_mq_fp8(msa, w8, wl.f32_to_bf16_bits(q), Q, k=k, n_sink=0, n_window=0)
    np.testing.assert_array_equal(ids, np.asarray(fx["expected_ids"], dtype=np.int32))
    for i in range(Q):
        for h in range(4):
            row = fx["expected_scores"][0][i][h]
            exp = np.full(k, -np.inf)
            exp[:len(row)] = row
            np.testing.assert_array_equal(sc[0, i, h].astype(np.float64), exp)


def test_multi_query_fp8_bad_page_is_reported(msa):
    w, q = multi_workload([3000, 3000], 4, seed=97, num_pages=60, max_model_len=4096)
    w8 = wl.to_fp8(w)
    w8.block_table[1, 4] = w8.pool8.shape[0] + 3
    import torch
    B, k = w8.batch, 16
    qd = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).cuda()
    ids = torch.empty((B, 4, 4, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((B, 4, 4, k), dtype=torch.float32, device="cuda")
    ws = msa.new_workspace(B, w8.max_model_len, k, q_len=4)
    msa.msa_indexer_decode_mq_fp8(qd, torch.from_numpy(w8.pool8).cuda(),
                                  torch.from_numpy(w8.kscale).cuda(),
                                  torch.from_numpy(w8.block_table).cuda(),
                                  torch.from_numpy(w8.seq_lens).cuda(), k, 1, 2, ids, sc, ws,
                                  max_model_len=w8.max_model_len)
    assert msa.msa_indexer_get_error(ws) & msa.MSA_FAULT_PAGE_ID
    assert not (ids[1].cpu().numpy() == 4).any()


def _max_batch_lens(seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 400, 4096)
    lens[rng.random(4096) < 0.05] = 0
    return lens


def test_multi_query_max_batch(msa, orc):
    """q_len 4 at the largest accepted batch (4096 short ragged requests)."""
    w, q = multi_workload(_max_batch_lens(4098), 4, seed=4098, max_model_len=512)
    check_rows(orc, w, q, 4, run_mq(msa, w, q, 4))


def test_multi_query_fp8_max_batch(msa, orc):
    """q_len 4 on the E4M3 cache at the largest accepted batch."""
    w, q = multi_workload(_max_batch_lens(4099), 4, seed=4099, max_model_len=512)
    w8 = wl.to_fp8(w)
    check_rows_fp8(orc, w8, q, 4, run_mq_fp8(msa, w8, q, 4))
