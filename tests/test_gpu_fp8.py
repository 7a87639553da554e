"""The fp8 E4M3 index-cache path against the oracle (same tolerance as bf16)."""

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
def test_fp8_config_parity(lib, orc, name):
    _compare(orc, wl.to_fp8(wl.make(name)))


@pytest.mark.slow
def test_fp8_long_context(lib, orc):
    _compare(orc, wl.to_fp8(wl.long_context()))


@pytest.mark.parametrize("k,n_sink,n_window", [(1, 0, 0), (16, 1, 2), (17, 1, 2), (32, 4, 8)])
def test_fp8_k_and_pins(lib, orc, k, n_sink, n_window):
    w = wl.to_fp8(wl.random_workload([1, 127, 128, 129, 2000, 5000, 8700, 0], num_pages=200,
                                     seed=33, q_scale=1 / np.sqrt(128), max_model_len=8704))
    _compare(orc, w, k=k, n_sink=n_sink, n_window=n_window)


def test_fp8_wide_q_range(lib, orc):
    """Heads whose q spans a wide range of magnitudes (tests the per-head power of two)."""
    w = wl.random_workload([3000, 4096, 777], num_pages=80, seed=34, max_model_len=4096)
    qf = wl.bf16_bits_to_f32(w.q).copy()
    qf[:, 0] *= 1e-3
    qf[:, 1] *= 300.0
    qf[:, 2, ::2] *= 1e-5
    w.q = wl.f32_to_bf16_bits(qf)
    _compare(orc, wl.to_fp8(w))


def test_fp8_split_width_is_bitwise_invariant(lib):
    w = wl.to_fp8(wl.ragged())
    ref = parity.run_gpu(w, split_blocks=0)
    for W in (1, 7, 64):
        got = parity.run_gpu(w, split_blocks=W)
        for x, y in zip(ref[:3], got[:3]):
            np.testing.assert_array_equal(x, y)


def test_fp8_matches_bf16_when_codes_are_exact(lib):
    """Keys that are exact E4M3 values with unit scales score the same on both caches."""
    w = wl.adversarial(batch=4)  # small integers: exact in E4M3 and bf16
    w8 = wl.to_fp8(w)
    w8.kscale[:] = 1.0
    import torch
    w8.pool8 = torch.from_numpy(wl.bf16_bits_to_f32(w.pool)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    a = parity.run_gpu(w)
    b = parity.run_gpu(w8)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_fp8_max_batch(lib, orc):
    """MSA_MAX_BATCH requests on the E4M3 cache, short ragged lengths with
    empty requests."""
    rng = np.random.default_rng(4097)
    seq = rng.integers(0, 400, 4096)
    seq[rng.random(4096) < 0.05] = 0
    w = wl.random_workload(seq, seed=4097, q_scale=1 / np.sqrt(128), max_model_len=512,
                           name="max_batch_fp8")
    _compare(orc, wl.to_fp8(w))
