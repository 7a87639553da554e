"""The allocation-free decode entry point against the regular one.

msa_indexer_decode_noalloc serves callers that cannot allocate device memory
(a plugin whose host framework owns the GPU's memory, or a per-token path
that must not call cudaMalloc).  It keeps its scratch in a fixed array inside
the library, so consecutive calls reuse the same memory; these tests check
that two calls in a row (and a third after them) give what the regular entry
point, with its own caller-owned workspace, gives on the same inputs.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""

import numpy as np
import pytest

import parity
import workloads as wl

pytestmark = pytest.mark.gpu


def _noalloc(msa, tensors, w):
    import torch
    q, pool, bt, seq = tensors
    B, k = w.batch, w.k
    ids = torch.full((B, 4, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((B, 4, k), 7.0, dtype=torch.float32, device="cuda")
    blk = torch.full((B, 4, w.bt_stride), float("nan"), dtype=torch.float32, device="cuda")
    msa.msa_indexer_decode_noalloc(q, pool, bt, seq, k, w.n_sink, w.n_window, ids, sc,
                                   max_model_len=w.max_model_len, out_block_scores=blk)
    return ids, sc, blk


def _same(w, regular, got):
    r_ids, r_sc, r_blk, _ = regular
    ids, sc, blk = (t.cpu().numpy() for t in got)
    np.testing.assert_array_equal(ids, r_ids)
    finite = np.isfinite(r_sc)
    assert np.array_equal(np.isfinite(sc), finite)
    assert parity.within(sc[finite], r_sc[finite]).all()
    for b, nb in enumerate(w.num_blocks):
        assert parity.within(blk[b, :, :nb], r_blk[b, :, :nb]).all()


def test_noalloc_matches_decode_on_consecutive_calls():
    import torch
    import sparse_attention_decode_gb300 as msa
    msa.load()
    first, second = wl.decode_point(), wl.ragged()
    t_first, t_second = parity.to_device(first), parity.to_device(second)
    reg_first = parity.run_gpu(first, tensors=t_first)
    reg_second = parity.run_gpu(second, tensors=t_second)
    assert reg_first[3] == 0 and reg_second[3] == 0

    out1 = _noalloc(msa, t_first, first)
    out2 = _noalloc(msa, t_second, second)  # reuses the array right after call 1
    out3 = _noalloc(msa, t_first, first)    # and again after a different batch
    torch.cuda.synchronize()
    _same(first, reg_first, out1)
    _same(second, reg_second, out2)
    _same(first, reg_first, out3)


def test_noalloc_rejects_a_batch_beyond_its_scratch():
    import torch
    import sparse_attention_decode_gb300 as msa
    B = msa.MSA_MAX_BATCH
    q = torch.zeros((B, 4, 128), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((1, 128, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    seq = torch.zeros((B,), dtype=torch.int32, device="cuda")
    ids = torch.empty((B, 4, 32), dtype=torch.int32, device="cuda")
    sc = torch.empty((B, 4, 32), dtype=torch.float32, device="cuda")
    with pytest.raises(msa.MsaError) as e:
        msa.msa_indexer_decode_noalloc(q, pool, bt, seq, 32, 1, 2, ids, sc, max_model_len=128)
    assert e.value.status == msa.MSA_ERR_UNSUPPORTED
