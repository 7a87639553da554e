"""Host-made faults: bad device data and bad arguments.  No test faults the GPU.

Bad block-table entries and out-of-range lengths are plain data; the kernels
check them before any access, skip the work and report a fault bit.
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


def test_bad_page_id_is_skipped_and_reported(msa, orc):
    w = wl.random_workload([3000, 3000, 3000], num_pages=80, seed=51, q_scale=1 / np.sqrt(128),
                           max_model_len=4096)
    clean = wl.random_workload([3000, 3000, 3000], num_pages=80, seed=51,
                               q_scale=1 / np.sqrt(128), max_model_len=4096)
    w.block_table[1, 5] = w.num_pages + 7  # past the pool
    w.block_table[1, 9] = -3
    ids, sc, blk, fault = parity.run_gpu(w)
    assert fault & msa.MSA_FAULT_PAGE_ID
    assert np.isneginf(blk[1, :, 5]).all() and np.isneginf(blk[1, :, 9]).all()
    assert not (ids[1] == 5).any() and not (ids[1] == 9).any()
    # the other rows are untouched by the fault
    o_scores, o_ids, _ = orc.run(clean)
    sub = wl.Workload(name="rows0and2", q=clean.q[[0, 2]], pool=clean.pool,
                      block_table=clean.block_table[[0, 2]], seq_lens=clean.seq_lens[[0, 2]],
                      max_model_len=4096)
    parity.check(sub, o_scores[[0, 2]], o_ids[[0, 2]], ids[[0, 2]], sc[[0, 2]], blk[[0, 2]])
    # the fault word was cleared by the read
    ids2, _, _, fault2 = parity.run_gpu(clean)
    assert fault2 == 0


def test_bad_seq_len_empties_the_row(msa, orc):
    w = wl.random_workload([1000, 2000, 500], num_pages=40, seed=52, q_scale=1 / np.sqrt(128),
                           max_model_len=2048)
    w.seq_lens[1] = 99999  # above max_model_len
    ids, sc, blk, fault = parity.run_gpu(w)
    assert fault & msa.MSA_FAULT_SEQ_LEN
    assert (ids[1] == -1).all() and np.isneginf(sc[1]).all()
    w.seq_lens[1] = -5
    ids, sc, blk, fault = parity.run_gpu(w)
    assert fault & msa.MSA_FAULT_SEQ_LEN
    assert (ids[1] == -1).all()


def test_outputs_do_not_spill_past_their_end(msa):
    import torch
    w = wl.decode_point()
    q, pool, bt, seq = parity.to_device(w)
    B, k, pad = w.batch, 16, 4096
    ids = torch.full((B * 4 * k + pad,), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((B * 4 * k + pad,), 7.0, dtype=torch.float32, device="cuda")
    nbytes = msa.msa_indexer_workspace_bytes(B, w.max_model_len, k)
    ws = torch.zeros(nbytes + pad, dtype=torch.uint8, device="cuda")
    ws[nbytes:] = 0xA5
    msa.msa_indexer_decode(q, pool, bt, seq, k, 1, 2, ids[:B * 4 * k], sc[:B * 4 * k],
                           ws[:nbytes], max_model_len=w.max_model_len)
    torch.cuda.synchronize()
    assert (ids[B * 4 * k:] == -7).all() and (sc[B * 4 * k:] == 7.0).all()
    assert (ws[nbytes:] == 0xA5).all()


def test_argument_errors(msa):
    import torch
    w = wl.tiny()
    q, pool, bt, seq = parity.to_device(w)
    ids = torch.empty((2, 4, 16), dtype=torch.int32, device="cuda")
    sc = torch.empty((2, 4, 16), dtype=torch.float32, device="cuda")
    ws = msa.new_workspace(2, 1024, 16)
    with pytest.raises(msa.MsaError) as e:
        msa.msa_indexer_decode(q, pool, bt, seq, 16, 10, 10, ids, sc, ws, max_model_len=1024)
    assert e.value.status == msa.MSA_ERR_INVALID_ARG
    with pytest.raises(msa.MsaError) as e:
        msa.msa_indexer_decode(q, pool, bt, seq, 33, 1, 2, ids, sc, ws, max_model_len=1024)
    assert e.value.status == msa.MSA_ERR_UNSUPPORTED
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(msa.MsaError) as e:
        msa.msa_indexer_decode(q, pool, bt, seq, 16, 1, 2, ids, sc, small, max_model_len=1024)
    assert e.value.status == msa.MSA_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(msa.MsaError) as e:
        msa.msa_indexer_decode(q, pool, bt, seq, 16, 1, 2, ids, sc, ws, max_batch=1,
                               max_model_len=1024)
    assert e.value.status == msa.MSA_ERR_INVALID_ARG


@pytest.mark.parametrize("split", [0, 2])
def test_waits_that_run_out_end_the_call_and_leave_the_workspace_usable(msa, orc, split):
    """The bounded-wait path, made without any fault: with the test hook set,
    the producer loads no page and signals none (no copy is ever in flight),
    so every consumer's first page wait runs out after its short poll limit.
    The call must return, report MSA_FAULT_TIMEOUT and leave every row empty;
    the next call on the same workspace must match the oracle, which shows the
    ticket and arrival counters were returned to zero.  split=2 makes the
    producers claim pool chunks through the ticket counter."""
    w = wl.decode_point()
    tensors = parity.to_device(w)
    ws = msa.new_workspace(w.batch, w.max_model_len, w.k, split)
    msa.msa_indexer_test_withhold_pages(True)
    try:
        ids, sc, blk, fault = parity.run_gpu(w, tensors=tensors, ws=ws, split_blocks=split)
    finally:
        msa.msa_indexer_test_withhold_pages(False)
    assert fault & msa.MSA_FAULT_TIMEOUT
    assert (ids == -1).all() and np.isneginf(sc).all()
    o_scores, o_ids, _ = orc.run(w)
    for _ in range(2):
        ids, sc, blk, fault = parity.run_gpu(w, tensors=tensors, ws=ws, split_blocks=split)
        assert fault == 0
        parity.check(w, o_scores, o_ids, ids, sc, blk)
