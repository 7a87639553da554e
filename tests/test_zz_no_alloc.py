"""The allocation-free decode entry point against the regular one and the oracle.

msa_indexer_decode_noalloc serves callers that cannot allocate device memory
(a plugin whose host framework owns the GPU's memory, or a per-token path
that must not call cudaMalloc).  It keeps its scratch in a fixed array inside
the library, so consecutive calls reuse the same memory.  It runs the very
kernels of msa_indexer_decode on the same inputs, so its results must equal
the regular entry's bit for bit; they must also pass the oracle comparison.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""

import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import parity
import workloads as wl

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _noalloc(msa, tensors, w, k=None):
    import torch
    q, pool, bt, seq = tensors
    B, k = w.batch, (w.k if k is None else k)
    ids = torch.full((B, 4, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((B, 4, k), 7.0, dtype=torch.float32, device="cuda")
    blk = torch.full((B, 4, w.bt_stride), float("nan"), dtype=torch.float32, device="cuda")
    msa.msa_indexer_decode_noalloc(q, pool, bt, seq, k, w.n_sink, w.n_window, ids, sc,
                                   max_model_len=w.max_model_len, out_block_scores=blk)
    return [t.cpu().numpy() for t in (ids, sc, blk)]


def _bitwise(regular, got, what):
    for a, b, name in zip(regular[:3], got, ("ids", "scores", "block scores")):
        np.testing.assert_array_equal(b, a, err_msg=f"{what}: {name}")


def test_noalloc_matches_decode_on_consecutive_calls(orc):
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
    _bitwise(reg_first, out1, "call 1")
    _bitwise(reg_second, out2, "call 2")
    _bitwise(reg_first, out3, "call 3")
    for w, out in ((first, out1), (second, out2)):
        o_scores, o_ids, _ = orc.run(w)
        parity.check(w, o_scores, o_ids, out[0], out[1], out[2])


def test_noalloc_skips_a_bad_page_and_the_next_call_is_clean(orc):
    """Data faults are not reported by this entry (it has no workspace to read
    them from), but they are handled: a block whose table entry lies outside
    the pool is left out, the other rows are exact, and the next clean call
    equals the regular entry bit for bit."""
    import sparse_attention_decode_gb300 as msa
    msa.load()
    clean = wl.random_workload([3000, 3000, 3000], num_pages=80, seed=61,
                               q_scale=1 / np.sqrt(128), max_model_len=4096)
    bad = wl.random_workload([3000, 3000, 3000], num_pages=80, seed=61,
                             q_scale=1 / np.sqrt(128), max_model_len=4096)
    bad.block_table[1, 7] = bad.num_pages + 3
    ids, sc, blk = _noalloc(msa, parity.to_device(bad), bad)
    assert np.isneginf(blk[1, :, 7]).all()
    assert not (ids[1] == 7).any()
    o_scores, o_ids, _ = orc.run(clean)
    rows = [0, 2]
    sub = wl.Workload(name="rows0and2", q=clean.q[rows], pool=clean.pool,
                      block_table=clean.block_table[rows], seq_lens=clean.seq_lens[rows],
                      max_model_len=4096)
    parity.check(sub, o_scores[rows], o_ids[rows], ids[rows], sc[rows], blk[rows])
    t_clean = parity.to_device(clean)
    reg = parity.run_gpu(clean, tensors=t_clean)
    _bitwise(reg, _noalloc(msa, t_clean, clean), "clean call after a bad page")


def _largest_batch_that_fits(sms, k):
    """The documented scratch formula at max_model_len 128 (one block a request)."""
    kmax = 16 if k <= 16 else 32

    def need(B):
        ctas = min(sms, B)
        return 256 + -(-4 * (B + 1) // 256) * 256 + (7 * ctas + B) * 4 * kmax * 8

    B = 1
    while need(B + 1) <= 4 * 1024 * 1024:
        B += 1
    return B


def test_noalloc_size_limit_is_the_documented_one():
    """The largest batch whose scratch fits runs (and equals the regular
    entry); one request more is refused before anything is enqueued."""
    import torch
    import sparse_attention_decode_gb300 as msa
    msa.load()
    k = 32
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B = _largest_batch_that_fits(sms, k)
    assert 1024 <= B < msa.MSA_MAX_BATCH
    rng = np.random.default_rng(3)
    w = wl.random_workload(rng.integers(0, 129, B), seed=3, q_scale=1 / np.sqrt(128),
                           max_model_len=128, k=k)
    t = parity.to_device(w)
    reg = parity.run_gpu(w, tensors=t)
    assert reg[3] == 0
    _bitwise(reg, _noalloc(msa, t, w), f"batch {B}")
    q, pool, bt, seq = t
    q1 = torch.cat([q, q[:1]])
    bt1 = torch.cat([bt, bt[:1]])
    seq1 = torch.cat([seq, seq[:1]])
    ids = torch.empty((B + 1, 4, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((B + 1, 4, k), dtype=torch.float32, device="cuda")
    with pytest.raises(msa.MsaError) as e:
        msa.msa_indexer_decode_noalloc(q1, pool, bt1, seq1, k, 1, 2, ids, sc, max_model_len=128)
    assert e.value.status == msa.MSA_ERR_UNSUPPORTED


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


# A plugin inside a host framework often runs on a context of the framework's
# own rather than the primary one.  This child process (no torch) creates two
# driver contexts in turn and runs the allocation-free call and the regular
# one in each on the same inputs; each context holds its own copy of the
# library's scratch array, at its own address.
_CONTEXTS_SCRIPT = textwrap.dedent(r"""
    import ctypes, sys
    import numpy as np
    sys.path.insert(0, ROOT)
    import workloads as wl
    import sparse_attention_decode_gb300 as msa

    cu = ctypes.CDLL("libcuda.so.1")
    cu.cuMemcpyHtoD_v2.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t]
    cu.cuMemcpyDtoH_v2.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_size_t]
    cu.cuMemFree_v2.argtypes = [ctypes.c_uint64]
    def ok(r, what):
        if r != 0:
            raise RuntimeError(f"{what} failed: CUresult {r}")
    ok(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int(0)
    ok(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    lib = msa.load()
    w = wl.decode_point()
    B, k, S = w.batch, w.k, w.bt_stride
    host_in = {"q": w.q, "pool": w.pool, "bt": w.block_table, "seq": w.seq_lens}
    results, contexts = [], []
    for round_ in range(2):
        # both contexts stay alive to the end, so their handles differ
        ctx = ctypes.c_void_p()
        ok(cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, dev), "cuCtxCreate")  # now current
        contexts.append(ctx)
        ptrs = []
        def alloc(nbytes):
            p = ctypes.c_uint64()
            ok(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(nbytes)), "cuMemAlloc")
            ptrs.append(p)
            return p.value
        def upload(a):
            a = np.ascontiguousarray(a)
            p = alloc(a.nbytes)
            ok(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(p), a.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.c_size_t(a.nbytes)), "cuMemcpyHtoD")
            return p
        def download(p, shape, dtype):
            out = np.empty(shape, dtype=dtype)
            ok(cu.cuMemcpyDtoH_v2(out.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(p),
                                  ctypes.c_size_t(out.nbytes)), "cuMemcpyDtoH")
            return out
        d = {n: upload(a) for n, a in host_in.items()}
        nbytes = msa.msa_indexer_workspace_bytes(B, w.max_model_len, k)
        ws = upload(np.zeros(nbytes, dtype=np.uint8))
        outs = {}
        for name in ("noalloc", "noalloc again", "regular"):
            ids = alloc(B * 4 * k * 4)
            sc = alloc(B * 4 * k * 4)
            blk = upload(np.full((B, 4, S), np.nan, dtype=np.float32))
            args = [d["q"], d["pool"], w.num_pages, d["bt"], S, d["seq"], B]
            if name == "regular":
                st = lib.msa_indexer_decode(*args, B, w.max_model_len, k, w.n_sink, w.n_window,
                                            ids, sc, blk, ws, nbytes, 0, None)
            else:
                st = lib.msa_indexer_decode_noalloc(*args, w.max_model_len, k, w.n_sink,
                                                    w.n_window, ids, sc, blk, None)
            assert st == 0, (name, st)
            ok(cu.cuCtxSynchronize(), "cuCtxSynchronize")
            outs[name] = (download(ids, (B, 4, k), np.int32), download(sc, (B, 4, k), np.float32),
                          download(blk, (B, 4, S), np.float32))
        for name in ("noalloc", "noalloc again"):
            for a, b in zip(outs[name], outs["regular"]):
                assert np.array_equal(a, b, equal_nan=True), (round_, name)
        results.append(outs["regular"])
        for p in ptrs:
            ok(cu.cuMemFree_v2(p.value), "cuMemFree")
        popped = ctypes.c_void_p()
        ok(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "cuCtxPopCurrent")
    for ctx in contexts:
        ok(cu.cuCtxDestroy_v2(ctx), "cuCtxDestroy")
    for a, b in zip(results[0], results[1]):
        assert np.array_equal(a, b, equal_nan=True)
    print("contexts ok")
""")


def test_noalloc_in_two_driver_contexts():
    """Each context gets its own scratch address and a zeroed array: the
    allocation-free call equals the regular one in both, bit for bit."""
    import sparse_attention_decode_gb300 as msa
    msa.load()  # built by the session; the child only loads it
    script = f"ROOT = {ROOT!r}\n" + _CONTEXTS_SCRIPT
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "contexts ok" in r.stdout
