"""Comparison of the CUDA path with the oracle, and device helpers for the tests.

Tolerance (stated by the indexer's target): block scores agree within
|gpu - oracle| <= 1e-3 + 2e-3 * |oracle|.  Selected ids match exactly, except
that blocks whose oracle score lies within that tolerance of the k-th
selected free block's score (the "band") may be exchanged among themselves.
Where every score is an exact integer (the adversarial workload) there is no
rounding, so ids, order and scores must match exactly.
"""

from __future__ import annotations

import numpy as np

import workloads as wl

RTOL = 2e-3
ATOL = 1e-3


def within(g, o, rtol=RTOL, atol=ATOL):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    return np.abs(g - o) <= atol + rtol * np.abs(o)


def to_device(w, device="cuda"):
    """(q, pool, bt, seq) on the device; for an fp8 workload `pool` is (codes, scales)."""
    import torch
    q = torch.from_numpy(w.q.view(np.int16)).view(torch.bfloat16).to(device)
    if w.pool8 is not None:
        pool = (torch.from_numpy(w.pool8).to(device), torch.from_numpy(w.kscale).to(device))
    else:
        pool = torch.from_numpy(w.pool.view(np.int16)).view(torch.bfloat16).to(device)
    bt = torch.from_numpy(w.block_table).to(device)
    seq = torch.from_numpy(w.seq_lens).to(device)
    return q, pool, bt, seq


def run_gpu(w, *, k=None, n_sink=None, n_window=None, split_blocks=0, max_batch=None,
            max_model_len=None, device="cuda", tensors=None, block_scores=True, ws=None):
    """One decode call through the C ABI; returns numpy (ids, scores, block_scores, fault)."""
    import torch
    import sparse_attention_decode_gb300 as msa
    k = w.k if k is None else k
    n_sink = w.n_sink if n_sink is None else n_sink
    n_window = w.n_window if n_window is None else n_window
    max_batch = w.batch if max_batch is None else max_batch
    max_model_len = w.max_model_len if max_model_len is None else max_model_len
    q, pool, bt, seq = tensors if tensors is not None else to_device(w, device)
    B = w.batch
    ids = torch.full((B, 4, k), -7, dtype=torch.int32, device=device)
    sc = torch.full((B, 4, k), 7.0, dtype=torch.float32, device=device)
    blk = None
    if block_scores:
        blk = torch.full((B, 4, w.bt_stride), float("nan"), dtype=torch.float32, device=device)
    if ws is None:
        ws = msa.new_workspace(max_batch, max_model_len, k, split_blocks, device=device)
    if isinstance(pool, tuple):
        msa.msa_indexer_decode_fp8(q, pool[0], pool[1], bt, seq, k, n_sink, n_window, ids, sc, ws,
                                   max_batch=max_batch, max_model_len=max_model_len,
                                   out_block_scores=blk, split_blocks=split_blocks)
    else:
        msa.msa_indexer_decode(q, pool, bt, seq, k, n_sink, n_window, ids, sc, ws,
                               max_batch=max_batch, max_model_len=max_model_len,
                               out_block_scores=blk, split_blocks=split_blocks)
    fault = msa.msa_indexer_get_error(ws)
    return (ids.cpu().numpy(), sc.cpu().numpy(),
            None if blk is None else blk.cpu().numpy(), fault)


def check(w, o_scores, o_ids, g_ids, g_sc, g_blk=None, *, k=None, n_sink=None, n_window=None,
          exact=None):
    """Raises AssertionError on any disagreement; returns the number of band exchanges."""
    k = w.k if k is None else k
    n_sink = w.n_sink if n_sink is None else n_sink
    n_window = w.n_window if n_window is None else n_window
    exact = w.exact_integers if exact is None else exact
    nbs = w.num_blocks
    swaps = 0
    for b in range(w.batch):
        nb = int(nbs[b])
        for h in range(wl.HEADS):
            tag = f"{w.name} b={b} h={h} nb={nb}"
            o_row = o_scores[b, h, :nb]
            if g_blk is not None:
                gb = g_blk[b, h, :nb].astype(np.float64)
                if exact:
                    assert np.array_equal(gb, o_row), f"{tag}: block scores differ"
                else:
                    bad = ~within(gb, o_row)
                    assert not bad.any(), f"{tag}: block score off at {np.nonzero(bad)[0][:5]}"
            ids = [int(x) for x in g_ids[b, h]]
            n_sel = min(k, nb)
            assert all(x >= 0 for x in ids[:n_sel]), f"{tag}: missing ids {ids}"
            assert all(x == -1 for x in ids[n_sel:]), f"{tag}: padding ids {ids}"
            assert np.all(np.isneginf(g_sc[b, h, n_sel:])), f"{tag}: padding scores"
            sel = ids[:n_sel]
            assert len(set(sel)) == n_sel and all(0 <= x < nb for x in sel), f"{tag}: {sel}"
            pins = [j for j in range(nb) if j < n_sink or j >= nb - n_window]
            assert sel[:len(pins)] == pins, f"{tag}: pins {sel[:len(pins)]} != {pins}"
            # reported scores are the block scores (fp32) of the selected ids
            gs = g_sc[b, h, :n_sel].astype(np.float64)
            if exact:
                assert list(o_ids[b, h]) == ids, f"{tag}: ids {ids} != {list(o_ids[b, h])}"
                assert np.array_equal(gs, o_scores[b, h, sel]), f"{tag}: scores"
                continue
            assert within(gs, o_scores[b, h, sel]).all(), f"{tag}: selected scores off"
            if g_blk is not None:
                assert np.array_equal(gs, g_blk[b, h, sel].astype(np.float64)), f"{tag}: score copy"
            free_g = sel[len(pins):]
            free_o = [int(x) for x in o_ids[b, h, len(pins):n_sel]]
            # GPU order: fp32 score descending, ties by increasing id
            fs = gs[len(pins):]
            for r in range(len(free_g) - 1):
                assert fs[r] > fs[r + 1] or (fs[r] == fs[r + 1] and free_g[r] < free_g[r + 1]), \
                    f"{tag}: order at {r}"
            if nb <= k:
                assert sorted(free_g) == sorted(free_o), f"{tag}: all blocks expected"
                continue
            if not free_o:
                assert not free_g
                continue
            o_k = o_scores[b, h, free_o[-1]]
            unpinned = np.array([j for j in range(nb) if j not in set(pins)])
            band = set(unpinned[within(o_row[unpinned], np.full(unpinned.shape, o_k))].tolist())
            sg, so = set(free_g), set(free_o)
            assert sg - band == so - band, f"{tag}: outside the band {sorted(sg - band)} vs {sorted(so - band)}"
            assert len(sg & band) == len(so & band), f"{tag}: band counts"
            swaps += len((sg & band) ^ (so & band)) // 2
    return swaps
