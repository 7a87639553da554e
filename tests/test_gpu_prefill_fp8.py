"""Prefill scoring on the E4M3 index-K cache against the oracle.

The same rows as the bf16 prefill (each new token over its own causal
prefix); keys dequantise as e4m3(code) x per-token scale.
"""

import json
import os

import numpy as np
import pytest

import parity
import workloads as wl
from test_gpu_prefill import MIXED, check_prefill, prefill_case

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module")
def msa():
    import sparse_attention_decode_gb300 as m
    m.load()
    return m


def run_prefill_fp8(msa, w8, q_bits, cu, k=16, n_sink=1, n_window=2, block_scores=True):
    import torch
    total = q_bits.shape[0]
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    pool8 = torch.from_numpy(w8.pool8).cuda()
    ks = torch.from_numpy(w8.kscale).cuda()
    bt = torch.from_numpy(w8.block_table).cuda()
    seq = torch.from_numpy(w8.seq_lens).cuda()
    d_cu = torch.from_numpy(cu).cuda()
    ids = torch.full((total, 4, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((total, 4, k), 7.0, dtype=torch.float32, device="cuda")
    stride = (w8.max_model_len + 127) // 128
    blk = None
    if block_scores:
        blk = torch.full((total, 4, stride), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(msa.msa_indexer_prefill_workspace_bytes(total, w8.max_model_len),
                     dtype=torch.uint8, device="cuda")
    msa.msa_indexer_prefill_fp8(q, d_cu, pool8, ks, bt, seq, k, n_sink, n_window, ids, sc, ws,
                                max_model_len=w8.max_model_len, out_block_scores=blk)
    fault = msa.msa_indexer_get_error(ws)
    return (ids.cpu().numpy(), sc.cpu().numpy(), None if blk is None else blk.cpu().numpy(), fault)


def check_fp8(orc, w8, q, cu, got, k=16, n_sink=1, n_window=2, exact=False):
    s, o_ids, _, lens = orc.run_prefill(q, cu, None, w8.block_table, w8.seq_lens, k, n_sink,
                                        n_window, pool8=w8.pool8, kscale=w8.kscale)
    rows_bt = np.repeat(w8.block_table, np.diff(cu), axis=0)
    rows = wl.Workload(name=f"{w8.name}_prefill_fp8", q=q, pool=None, block_table=rows_bt,
                       seq_lens=lens, k=k, n_sink=n_sink, n_window=n_window,
                       max_model_len=w8.max_model_len)
    st = rows.bt_stride
    g_ids, g_sc, g_blk = got[:3]
    return parity.check(rows, s[:, :, :st], o_ids, g_ids, g_sc,
                        None if g_blk is None else g_blk[:, :, :st], k=k, n_sink=n_sink,
                        n_window=n_window, exact=exact)


def test_prefill_fp8_mixed_batch(msa, orc):
    w, q, cu = prefill_case(MIXED, seed=600, max_model_len=8192)
    w8 = wl.to_fp8(w)
    got = run_prefill_fp8(msa, w8, q, cu)
    assert got[3] == 0
    check_fp8(orc, w8, q, cu, got)


@pytest.mark.parametrize("pairs", [[(700, 8000)], [(1000, 1000), (257, 16384)]])
def test_prefill_fp8_long(msa, orc, pairs):
    w, q, cu = prefill_case(pairs, seed=610 + len(pairs), max_model_len=16384)
    w8 = wl.to_fp8(w)
    got = run_prefill_fp8(msa, w8, q, cu)
    assert got[3] == 0
    check_fp8(orc, w8, q, cu, got)


@pytest.mark.parametrize("k,n_sink,n_window", [(1, 0, 0), (16, 0, 16), (17, 1, 2), (32, 4, 8)])
def test_prefill_fp8_k_and_pins(msa, orc, k, n_sink, n_window):
    w, q, cu = prefill_case(MIXED, seed=620 + k, max_model_len=8192)
    w8 = wl.to_fp8(w)
    got = run_prefill_fp8(msa, w8, q, cu, k=k, n_sink=n_sink, n_window=n_window)
    assert got[3] == 0
    check_fp8(orc, w8, q, cu, got, k=k, n_sink=n_sink, n_window=n_window)


def test_prefill_fp8_wide_q_range(msa, orc):
    """Query rows spanning many binades (the per-row f16 scaling)."""
    w, q, cu = prefill_case([(64, 3000), (33, 700)], seed=630, max_model_len=4096)
    rng = np.random.default_rng(631)
    qf = wl.bf16_bits_to_f32(q) * np.exp2(rng.integers(-30, 30, size=(q.shape[0], 4, 1))).astype(np.float32)
    q2 = wl.f32_to_bf16_bits(qf.astype(np.float32))
    w8 = wl.to_fp8(w)
    got = run_prefill_fp8(msa, w8, q2, cu)
    assert got[3] == 0
    check_fp8(orc, w8, q2, cu, got)


def test_prefill_fp8_fixture_exact(msa):
    """The hand-coded E4M3 causal fixture: the request's last four tokens, exact."""
    with open(os.path.join(GOLDEN, "multi_query_causal.json")) as f:
        fx = json.load(f)
    L, Q, k = int(fx["seq_len"]), int(fx["q_len"]), int(fx["k"])
    code_of_double = {1.0: 0x40, 4.0: 0x50, 2.0: 0x48, 8.0: 0x58}
    codes = np.zeros((2, 128, 128), dtype=np.uint8)
    for tok, v in fx["planted_dim0"].items():
        codes[int(tok) // 128, int(tok) % 128, 0] = code_of_double[float(v)]
    q = np.zeros((Q, 4, 128), dtype=np.float32)
    q[:, :, 0] = np.asarray(fx["alpha"], dtype=np.float32)[None, :]
    w8 = wl.Workload(name="golden_prefill_fp8", q=wl.f32_to_bf16_bits(q[:1]), pool=None,
                     block_table=np.array([[0, 1]], dtype=np.int32),
                     seq_lens=np.array([L], dtype=np.int32), k=k, n_sink=0, n_window=0,
                     max_model_len=256, pool8=codes, kscale=np.full((2, 128), 0.5, dtype=np.float32))
    ids, sc, _, fault = run_prefill_fp8(msa, w8, wl.f32_to_bf16_bits(q), np.array([0, Q], dtype=np.int32),
                                        k=k, n_sink=0, n_window=0)
    assert fault == 0
    np.testing.assert_array_equal(ids, np.asarray(fx["expected_ids"], dtype=np.int32)[0])
    for i in range(Q):
        for h in range(4):
            row = fx["expected_scores"][0][i][h]
            exp = np.full(k, -np.inf)
            exp[:len(row)] = row
            np.testing.assert_array_equal(sc[i, h].astype(np.float64), exp)


def test_prefill_fp8_matches_bf16_when_codes_are_exact(msa):
    """Keys exactly representable in E4M3 with scale 1: the fp8 prefill equals the bf16 one."""
    import torch
    w, q, cu = prefill_case([(100, 3000), (40, 900)], seed=640, max_model_len=4096)
    rng = np.random.default_rng(641)
    codes = rng.integers(0, 256, size=w.pool.shape, dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0  # no NaN codes
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    w.pool = wl.f32_to_bf16_bits(table[codes].astype(np.float32))
    wl.poison_tails(w.pool, w.block_table, w.seq_lens)
    w8 = wl.Workload(name="exact_codes", q=w.q, pool=w.pool, block_table=w.block_table,
                     seq_lens=w.seq_lens, k=16, n_sink=1, n_window=2,
                     max_model_len=w.max_model_len, pool8=codes,
                     kscale=np.ones(codes.shape[:2], dtype=np.float32))
    from test_gpu_prefill import run_prefill
    a = run_prefill(msa, w, q, cu)
    b = run_prefill_fp8(msa, w8, q, cu)
    assert a[3] == 0 and b[3] == 0
    for r in range(q.shape[0]):
        req = np.searchsorted(cu, r, side="right") - 1
        nb = (int(w.seq_lens[req]) - int(np.diff(cu)[req]) + (r - cu[req]) + 1 + 127) // 128
        np.testing.assert_allclose(b[2][r, :, :nb], a[2][r, :, :nb], rtol=2e-3, atol=1e-3)


def test_prefill_fp8_bad_page_is_reported(msa):
    w, q, cu = prefill_case([(40, 1000), (10, 600)], seed=650, max_model_len=2048, num_pages=30)
    w8 = wl.to_fp8(w)
    w8.block_table[0, 3] = w8.pool8.shape[0] + 5
    ids, sc, blk, fault = run_prefill_fp8(msa, w8, q, cu)
    assert fault & msa.MSA_FAULT_PAGE_ID
    assert np.isneginf(blk[:40, :, 3]).all()
    assert not (ids[:40] == 3).any()


def test_prefill_score_fp8_entry_matches(msa):
    import torch
    w, q, cu = prefill_case(MIXED, seed=660, max_model_len=8192)
    w8 = wl.to_fp8(w)
    got = run_prefill_fp8(msa, w8, q, cu)
    assert got[3] == 0
    total = q.shape[0]
    out = torch.full((total, 4, 64), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    msa.msa_indexer_prefill_score_fp8(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).cuda(),
                                      torch.from_numpy(cu).cuda(), torch.from_numpy(w8.pool8).cuda(),
                                      torch.from_numpy(w8.kscale).cuda(),
                                      torch.from_numpy(w8.block_table).cuda(),
                                      torch.from_numpy(w8.seq_lens).cuda(), out, ws,
                                      max_model_len=w8.max_model_len)
    assert msa.msa_indexer_get_error(ws) == 0
    np.testing.assert_array_equal(out.cpu().numpy(), got[2])


def test_prefill_fp8_bench_workload_sampled_rows(msa, orc):
    """The benchmarked prefill on the E4M3 cache (4 x 2048 new tokens at 128K,
    the launch `bench.py --path prefill --cache fp8` times) on the GPU; sampled
    rows checked one by one against the oracle."""
    import bench
    w, q, cu = bench.prefill_workload()
    w8 = wl.to_fp8(w)
    got = run_prefill_fp8(msa, w8, q, cu)
    assert got[3] == 0
    total = q.shape[0]
    rng = np.random.default_rng(401)
    firsts, lasts = cu[:-1], cu[1:] - 1
    rows = np.unique(np.concatenate([firsts, lasts, rng.choice(total, 16, replace=False)]))
    req = np.searchsorted(cu, rows, side="right") - 1
    lens = (w8.seq_lens[req] - np.diff(cu)[req] + (rows - cu[req]) + 1).astype(np.int32)
    bt_rows = w8.block_table[req]
    s = orc.block_scores_fp8(q[rows], w8.pool8, w8.kscale, bt_rows, lens)
    o_ids, _ = orc.select(s, lens, w8.k, w8.n_sink, w8.n_window)
    sub = wl.Workload(name="bench_prefill_fp8_rows", q=q[rows], pool=None, block_table=bt_rows,
                      seq_lens=lens, k=w8.k, n_sink=w8.n_sink, n_window=w8.n_window,
                      max_model_len=w8.max_model_len)
    st = sub.bt_stride
    parity.check(sub, s[:, :, :st], o_ids, got[0][rows], got[1][rows], got[2][rows][:, :, :st])


def test_prefill_fp8_many_requests(msa, orc):
    """200 short ragged requests on the E4M3 cache."""
    from test_gpu_prefill import _many_pairs
    w, q, cu = prefill_case(_many_pairs(502), seed=503, max_model_len=2048)
    w8 = wl.to_fp8(w)
    got = run_prefill_fp8(msa, w8, q, cu)
    assert got[3] == 0
    check_fp8(orc, w8, q, cu, got)
