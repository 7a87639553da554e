"""The C ABI library builds, loads and exports what include/msa_indexer.h declares.

No compute runs here: only host-side calls that return before touching the GPU.
"""

import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa_indexer.h")


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("no CUDA toolkit")
    from sparse_attention_decode_gb300 import build
    build.build()
    import sparse_attention_decode_gb300 as msa
    return msa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    import sparse_attention_decode_gb300 as msa
    assert declared_functions() == sorted(msa.EXPORTED)


def test_the_package_binds_every_declared_call():
    import sparse_attention_decode_gb300 as msa
    for name in declared_functions():
        if name != "msa_status_string":
            assert callable(getattr(msa, name, None)), name


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_workspace_bytes(lib):
    import sparse_attention_decode_gb300 as msa
    n = msa.msa_indexer_workspace_bytes(32, 131072, 16)
    # header 256 + prefix (33 ints -> 256) + (7 chunks x 1024 CTAs + 32) slots x 4 heads x 16 keys x 8 B
    fixed = 256 + 256
    assert n == fixed + (7 * 1024 + 32) * 4 * 16 * 8
    assert msa.msa_indexer_workspace_bytes(32, 131072, 16, 64) == fixed + (512 + 32) * 512
    assert msa.msa_indexer_workspace_bytes(32, 131072, 17) == fixed + (7 * 1024 + 32) * 4 * 32 * 8
    for bad in [(0, 1024, 16, 0), (32, 0, 16, 0), (32, 1024, 0, 0), (32, 1024, 33, 0),
                (32, 1024, 16, -1), (5000, 1024, 16, 0)]:
        assert msa.msa_indexer_workspace_bytes(*bad) == 0, bad


def test_status_strings(lib):
    import sparse_attention_decode_gb300 as msa
    assert msa.msa_status_string(0) == "ok"
    assert msa.msa_status_string(3) == "workspace too small"
    assert msa.msa_status_string(99) == "unknown status"


def test_null_pointers_are_rejected_before_any_gpu_work(lib):
    P = ctypes.c_void_p
    st = lib.msa_indexer_decode(None, None, 1, None, 1, None, 1, 1, 1024, 16, 1, 2, None, None,
                                None, None, 0, 0, None)
    assert st == 1
    st = lib.msa_indexer_merge(1, 16, None, None, None, 0, None)
    assert st == 1
    flags = ctypes.c_uint32(0)
    assert lib.msa_indexer_get_error(None, None, ctypes.byref(flags)) == 1


def test_bad_sizes_are_rejected_before_any_gpu_work(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only check: never hand placeholder pointers to a process with a GPU")
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    args = lambda **kw: [fake, fake, kw.get("pages", 10), fake, 8, fake, kw.get("B", 2),
                         kw.get("maxB", 2), 1024, kw.get("k", 16), kw.get("sink", 1),
                         kw.get("win", 2), fake, fake, None, ctypes.c_void_p(1 << 20), 1 << 20, 0,
                         None]
    assert lib.msa_indexer_decode(*args(sink=9, win=8)) == 1  # pins exceed k
    assert lib.msa_indexer_decode(*args(k=33)) == 2
    assert lib.msa_indexer_decode(*args(B=3)) == 1  # batch above max_batch
    assert lib.msa_indexer_decode(*args(pages=0)) == 1
    assert lib.msa_indexer_decode(*args(pages=1 << 25)) == 2
    assert lib.msa_indexer_decode(*args(maxB=5000, B=5000)) == 2


def test_prefill_workspace_and_argument_checks(lib):
    import sparse_attention_decode_gb300 as msa
    # header + total_q x 4 heads x blocks x fp32
    assert msa.msa_indexer_prefill_workspace_bytes(100, 8192) == 256 + 100 * 4 * 64 * 4
    assert msa.msa_indexer_prefill_workspace_bytes(0, 8192) == 256
    assert msa.msa_indexer_prefill_workspace_bytes(-1, 8192) == 0
    assert msa.msa_indexer_prefill_workspace_bytes(4, 0) == 0
    st = lib.msa_indexer_prefill(None, None, 4, None, 8, None, 8, None, 1, 1024, 16, 1, 2, None,
                                 None, None, None, 0, None)
    assert st == 1


def test_prefill_bad_sizes_are_rejected_before_any_gpu_work(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only check: never hand placeholder pointers to a process with a GPU")
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    args = lambda **kw: [fake, fake, kw.get("tq", 64), fake, kw.get("pages", 10), fake, 8, fake,
                         kw.get("B", 2), 1024, kw.get("k", 16), kw.get("sink", 1), kw.get("win", 2),
                         fake, fake, None, fake, kw.get("wsb", 1 << 20), None]
    assert lib.msa_indexer_prefill(*args(sink=9, win=8)) == 1  # pins exceed k
    assert lib.msa_indexer_prefill(*args(k=33)) == 2
    assert lib.msa_indexer_prefill(*args(B=0)) == 1
    assert lib.msa_indexer_prefill(*args(B=5000)) == 2
    assert lib.msa_indexer_prefill(*args(tq=-1)) == 1
    assert lib.msa_indexer_prefill(*args(pages=0)) == 1
    assert lib.msa_indexer_prefill(*args(wsb=256 + 64 * 4 * 8 * 4 - 4)) == 3
