"""Thin ctypes binding of libmsa_indexer.so (argument marshalling only).

Every function here has the name of the C entry point it calls and passes
device pointers of torch tensors straight through; all compute runs in the
CUDA kernels of the library.  If the library has not been built, importing
the package still works but every call raises: there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import build as _build

MSA_OK = 0
MSA_ERR_INVALID_ARG = 1
MSA_ERR_UNSUPPORTED = 2
MSA_ERR_WORKSPACE_TOO_SMALL = 3
MSA_ERR_CUDA = 4

MSA_FAULT_SEQ_LEN = 0x1
MSA_FAULT_PAGE_ID = 0x2
MSA_FAULT_TIMEOUT = 0x4
MSA_FAULT_SLOTS = 0x8

MSA_NUM_HEADS = 4
MSA_HEAD_DIM = 128
MSA_PAGE_TOKENS = 128
MSA_MAX_TOPK = 32
MSA_MAX_BATCH = 4096
MSA_NOALLOC_WORKSPACE_BYTES = 4 * 1024 * 1024

EXPORTED = (
    "msa_indexer_workspace_bytes",
    "msa_indexer_decode",
    "msa_indexer_score",
    "msa_indexer_merge",
    "msa_indexer_get_error",
    "msa_status_string",
    "msa_indexer_decode_noalloc",
    "msa_indexer_expand_pages",
    "msa_indexer_score_fp8",
    "msa_indexer_decode_fp8",
    "msa_indexer_decode_mq",
    "msa_indexer_workspace_bytes_mq",
    "msa_indexer_decode_mq_fp8",
    "msa_indexer_decode_pages",
    "msa_indexer_prefill",
    "msa_indexer_prefill_fp8",
    "msa_indexer_prefill_score",
    "msa_indexer_prefill_score_fp8",
    "msa_indexer_prefill_workspace_bytes",
    "msa_indexer_test_withhold_pages",
)

_lib = None


class MsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {msa_status_string(status)} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.LIBRARY


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """The compiled library; raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIBRARY
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library {p} is missing; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    c_i64, c_int, c_size, P = ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    lib.msa_indexer_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int]
    lib.msa_indexer_workspace_bytes.restype = c_size
    common = [P, P, c_i64, P, c_i64, P, c_int, c_int, c_int, c_int, c_int, c_int]
    lib.msa_indexer_decode.argtypes = common + [P, P, P, P, c_size, c_int, P]
    lib.msa_indexer_decode.restype = c_int
    lib.msa_indexer_score.argtypes = common + [P, P, c_size, c_int, P]
    lib.msa_indexer_score.restype = c_int
    lib.msa_indexer_merge.argtypes = [c_int, c_int, P, P, P, c_size, P]
    lib.msa_indexer_merge.restype = c_int
    lib.msa_indexer_get_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
    lib.msa_indexer_get_error.restype = c_int
    lib.msa_indexer_decode_noalloc.argtypes = common[:7] + common[8:] + [P, P, P, P]
    lib.msa_indexer_decode_noalloc.restype = c_int
    lib.msa_indexer_expand_pages.argtypes = [P, c_int, c_int, P, P, c_i64, c_int, P, P, P]
    lib.msa_indexer_expand_pages.restype = c_int
    common8 = [P, P, P, c_i64, P, c_i64, P, c_int, c_int, c_int, c_int, c_int, c_int]
    lib.msa_indexer_decode_fp8.argtypes = common8 + [P, P, P, P, c_size, c_int, P]
    lib.msa_indexer_decode_fp8.restype = c_int
    lib.msa_indexer_score_fp8.argtypes = common8 + [P, P, c_size, c_int, P]
    lib.msa_indexer_score_fp8.restype = c_int
    lib.msa_indexer_workspace_bytes_mq.argtypes = [c_int, c_int, c_int, c_int, c_int]
    lib.msa_indexer_workspace_bytes_mq.restype = c_size
    lib.msa_indexer_decode_mq.argtypes = [P, c_int] + common[1:] + [P, P, P, P, c_size, c_int, P]
    lib.msa_indexer_decode_mq.restype = c_int
    lib.msa_indexer_decode_mq_fp8.argtypes = [P, c_int] + common8[1:] + [P, P, P, P, c_size, c_int, P]
    lib.msa_indexer_decode_mq_fp8.restype = c_int
    lib.msa_indexer_prefill_workspace_bytes.argtypes = [c_int, c_int]
    lib.msa_indexer_prefill_workspace_bytes.restype = c_size
    lib.msa_indexer_prefill.argtypes = [P, P, c_int, P, c_i64, P, c_i64, P, c_int, c_int, c_int,
                                        c_int, c_int, P, P, P, P, c_size, P]
    lib.msa_indexer_prefill.restype = c_int
    lib.msa_indexer_decode_pages.argtypes = common + [P, P, P, P, c_size, c_int, P, c_i64, c_int,
                                                      P, P, P]
    lib.msa_indexer_decode_pages.restype = c_int
    lib.msa_indexer_prefill_score.argtypes = [P, P, c_int, P, c_i64, P, c_i64, P, c_int, c_int, P,
                                              P, c_size, P]
    lib.msa_indexer_prefill_score.restype = c_int
    lib.msa_indexer_prefill_fp8.argtypes = [P, P, c_int, P, P, c_i64, P, c_i64, P, c_int, c_int,
                                            c_int, c_int, c_int, P, P, P, P, c_size, P]
    lib.msa_indexer_prefill_fp8.restype = c_int
    lib.msa_indexer_prefill_score_fp8.argtypes = [P, P, c_int, P, P, c_i64, P, c_i64, P, c_int,
                                                  c_int, P, P, c_size, P]
    lib.msa_indexer_prefill_score_fp8.restype = c_int
    lib.msa_indexer_test_withhold_pages.argtypes = [c_int]
    lib.msa_indexer_test_withhold_pages.restype = None
    lib.msa_status_string.argtypes = [c_int]
    lib.msa_status_string.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return int(t.data_ptr())


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(status: int, what: str) -> None:
    if status != MSA_OK:
        raise MsaError(status, what)


def msa_status_string(status: int) -> str:
    return load().msa_status_string(int(status)).decode()


def msa_indexer_workspace_bytes(max_batch: int, max_model_len: int, k: int,
                                split_blocks: int = 0) -> int:
    return int(load().msa_indexer_workspace_bytes(max_batch, max_model_len, k, split_blocks))


def _shape_args(q, kcache_pool, block_table, seq_lens):
    import torch
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 3, "q: bf16 [B,4,128]"
    assert tuple(q.shape[1:]) == (MSA_NUM_HEADS, MSA_HEAD_DIM), "q: bf16 [B,4,128]"
    assert kcache_pool.dtype == torch.bfloat16 and kcache_pool.is_contiguous(), "kcache_pool: bf16"
    assert tuple(kcache_pool.shape[1:]) == (MSA_PAGE_TOKENS, MSA_HEAD_DIM), "kcache_pool: [P,128,128]"
    assert block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.stride(1) == 1
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    B = int(q.shape[0])
    assert block_table.shape[0] == B and seq_lens.shape[0] == B
    return B, int(kcache_pool.shape[0]), int(block_table.stride(0))


def msa_indexer_decode(q, kcache_pool, block_table, seq_lens, k: int, n_sink: int, n_window: int,
                       out_ids, out_scores, workspace, *, max_batch: Optional[int] = None,
                       max_model_len: int, out_block_scores=None, split_blocks: int = 0,
                       stream=None) -> None:
    """msa_indexer_decode() on torch CUDA tensors; raises MsaError on a bad status."""
    B, num_pages, bt_stride = _shape_args(q, kcache_pool, block_table, seq_lens)
    st = load().msa_indexer_decode(
        _ptr(q), _ptr(kcache_pool), num_pages, _ptr(block_table), bt_stride, _ptr(seq_lens), B,
        B if max_batch is None else max_batch, max_model_len, k, n_sink, n_window, _ptr(out_ids),
        _ptr(out_scores), _ptr(out_block_scores), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), split_blocks, _stream_ptr(stream))
    _check(st, "msa_indexer_decode")


def _fp8_args(q, kcache_fp8, kscale, block_table, seq_lens):
    import torch
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and tuple(q.shape[1:]) == (4, 128)
    assert kcache_fp8.element_size() == 1 and kcache_fp8.is_contiguous(), "kcache_fp8: 1-byte E4M3 codes"
    assert tuple(kcache_fp8.shape[1:]) == (MSA_PAGE_TOKENS, MSA_HEAD_DIM)
    assert kscale.dtype == torch.float32 and kscale.is_contiguous()
    assert tuple(kscale.shape) == tuple(kcache_fp8.shape[:2])
    assert block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.stride(1) == 1
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    B = int(q.shape[0])
    return B, int(kcache_fp8.shape[0]), int(block_table.stride(0))


def msa_indexer_decode_fp8(q, kcache_fp8, kscale, block_table, seq_lens, k: int, n_sink: int,
                           n_window: int, out_ids, out_scores, workspace, *,
                           max_batch: Optional[int] = None, max_model_len: int,
                           out_block_scores=None, split_blocks: int = 0, stream=None) -> None:
    """msa_indexer_decode_fp8(): the decode step on an E4M3 cache with per-token scales."""
    B, num_pages, bt_stride = _fp8_args(q, kcache_fp8, kscale, block_table, seq_lens)
    st = load().msa_indexer_decode_fp8(
        _ptr(q), _ptr(kcache_fp8), _ptr(kscale), num_pages, _ptr(block_table), bt_stride,
        _ptr(seq_lens), B, B if max_batch is None else max_batch, max_model_len, k, n_sink,
        n_window, _ptr(out_ids), _ptr(out_scores), _ptr(out_block_scores), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), split_blocks, _stream_ptr(stream))
    _check(st, "msa_indexer_decode_fp8")


def msa_indexer_score_fp8(q, kcache_fp8, kscale, block_table, seq_lens, k: int, n_sink: int,
                          n_window: int, workspace, *, max_batch: Optional[int] = None,
                          max_model_len: int, out_block_scores=None, split_blocks: int = 0,
                          stream=None) -> None:
    B, num_pages, bt_stride = _fp8_args(q, kcache_fp8, kscale, block_table, seq_lens)
    st = load().msa_indexer_score_fp8(
        _ptr(q), _ptr(kcache_fp8), _ptr(kscale), num_pages, _ptr(block_table), bt_stride,
        _ptr(seq_lens), B, B if max_batch is None else max_batch, max_model_len, k, n_sink,
        n_window, _ptr(out_block_scores), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), split_blocks, _stream_ptr(stream))
    _check(st, "msa_indexer_score_fp8")


def msa_indexer_score(q, kcache_pool, block_table, seq_lens, k: int, n_sink: int, n_window: int,
                      workspace, *, max_batch: Optional[int] = None, max_model_len: int,
                      out_block_scores=None, split_blocks: int = 0, stream=None) -> None:
    B, num_pages, bt_stride = _shape_args(q, kcache_pool, block_table, seq_lens)
    st = load().msa_indexer_score(
        _ptr(q), _ptr(kcache_pool), num_pages, _ptr(block_table), bt_stride, _ptr(seq_lens), B,
        B if max_batch is None else max_batch, max_model_len, k, n_sink, n_window,
        _ptr(out_block_scores), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), split_blocks, _stream_ptr(stream))
    _check(st, "msa_indexer_score")


def msa_indexer_merge(batch: int, k: int, out_ids, out_scores, workspace, *, stream=None) -> None:
    st = load().msa_indexer_merge(batch, k, _ptr(out_ids), _ptr(out_scores), _ptr(workspace),
                                  int(workspace.numel() * workspace.element_size()),
                                  _stream_ptr(stream))
    _check(st, "msa_indexer_merge")


def msa_indexer_decode_noalloc(q, kcache_pool, block_table, seq_lens, k: int, n_sink: int,
                               n_window: int, out_ids, out_scores, *, max_model_len: int,
                               out_block_scores=None, stream=None) -> None:
    """msa_indexer_decode_noalloc(): the decode step for callers that cannot allocate.

    No workspace argument: the library uses a fixed scratch array of its own
    (see the C header).  Calls that overlap on the GPU share that array and
    race, so serialise them.
    """
    B, num_pages, bt_stride = _shape_args(q, kcache_pool, block_table, seq_lens)
    st = load().msa_indexer_decode_noalloc(
        _ptr(q), _ptr(kcache_pool), num_pages, _ptr(block_table), bt_stride, _ptr(seq_lens), B,
        max_model_len, k, n_sink, n_window, _ptr(out_ids), _ptr(out_scores),
        _ptr(out_block_scores), _stream_ptr(stream))
    _check(st, "msa_indexer_decode_noalloc")


def msa_indexer_expand_pages(ids, seq_lens, kv_block_table, out_pages, out_num_pages, *,
                             page_tokens: int = 16, stream=None) -> None:
    """msa_indexer_expand_pages(): selected blocks -> small KV page ids."""
    import torch
    assert ids.dtype == torch.int32 and ids.is_contiguous() and ids.dim() == 3
    assert kv_block_table.dtype == torch.int32 and kv_block_table.stride(1) == 1
    B, _, k = ids.shape
    st = load().msa_indexer_expand_pages(_ptr(ids), B, k, _ptr(seq_lens), _ptr(kv_block_table),
                                         int(kv_block_table.stride(0)), page_tokens,
                                         _ptr(out_pages), _ptr(out_num_pages), _stream_ptr(stream))
    _check(st, "msa_indexer_expand_pages")


def msa_indexer_decode_mq_fp8(q, kcache_fp8, kscale, block_table, seq_lens, k: int, n_sink: int,
                              n_window: int, out_ids, out_scores, workspace, *,
                              max_batch: Optional[int] = None, max_model_len: int,
                              out_block_scores=None, split_blocks: int = 0, stream=None) -> None:
    """msa_indexer_decode_mq_fp8(): q bf16 [B, q_len, 4, 128] on the E4M3 cache."""
    import torch
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 4
    assert tuple(q.shape[2:]) == (MSA_NUM_HEADS, MSA_HEAD_DIM)
    assert kcache_fp8.element_size() == 1 and kcache_fp8.is_contiguous(), "kcache_fp8: 1-byte E4M3 codes"
    assert tuple(kcache_fp8.shape[1:]) == (MSA_PAGE_TOKENS, MSA_HEAD_DIM)
    assert kscale.dtype == torch.float32 and kscale.is_contiguous()
    assert tuple(kscale.shape) == tuple(kcache_fp8.shape[:2])
    assert block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.stride(1) == 1
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    B, q_len = int(q.shape[0]), int(q.shape[1])
    num_pages, bt_stride = int(kcache_fp8.shape[0]), int(block_table.stride(0))
    st = load().msa_indexer_decode_mq_fp8(
        _ptr(q), q_len, _ptr(kcache_fp8), _ptr(kscale), num_pages, _ptr(block_table), bt_stride,
        _ptr(seq_lens), B, B if max_batch is None else max_batch, max_model_len, k, n_sink,
        n_window, _ptr(out_ids), _ptr(out_scores), _ptr(out_block_scores), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), split_blocks, _stream_ptr(stream))
    _check(st, "msa_indexer_decode_mq_fp8")


def msa_indexer_decode_pages(q, kcache_pool, block_table, seq_lens, k: int, n_sink: int,
                             n_window: int, out_ids, out_scores, workspace, kv_block_table,
                             out_pages, out_num_pages, *, max_batch: Optional[int] = None,
                             max_model_len: int, page_tokens: int = 16, out_block_scores=None,
                             split_blocks: int = 0, stream=None) -> None:
    """msa_indexer_decode_pages(): decode with the page expansion fused into the merge."""
    import torch
    assert kv_block_table.dtype == torch.int32 and kv_block_table.stride(1) == 1
    B, num_pages, bt_stride = _shape_args(q, kcache_pool, block_table, seq_lens)
    st = load().msa_indexer_decode_pages(
        _ptr(q), _ptr(kcache_pool), num_pages, _ptr(block_table), bt_stride, _ptr(seq_lens), B,
        B if max_batch is None else max_batch, max_model_len, k, n_sink, n_window, _ptr(out_ids),
        _ptr(out_scores), _ptr(out_block_scores), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), split_blocks, _ptr(kv_block_table),
        int(kv_block_table.stride(0)), page_tokens, _ptr(out_pages), _ptr(out_num_pages),
        _stream_ptr(stream))
    _check(st, "msa_indexer_decode_pages")


def msa_indexer_workspace_bytes_mq(max_batch: int, max_model_len: int, k: int,
                                   split_blocks: int = 0, q_len: int = 1) -> int:
    return int(load().msa_indexer_workspace_bytes_mq(max_batch, max_model_len, k, split_blocks,
                                                     q_len))


def msa_indexer_decode_mq(q, kcache_pool, block_table, seq_lens, k: int, n_sink: int,
                          n_window: int, out_ids, out_scores, workspace, *,
                          max_batch: Optional[int] = None, max_model_len: int,
                          out_block_scores=None, split_blocks: int = 0, stream=None) -> None:
    """msa_indexer_decode_mq(): q is bf16 [B, q_len, 4, 128] (the last q_len tokens)."""
    import torch
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and q.dim() == 4
    assert tuple(q.shape[2:]) == (MSA_NUM_HEADS, MSA_HEAD_DIM)
    assert kcache_pool.dtype == torch.bfloat16 and kcache_pool.is_contiguous()
    assert block_table.dtype == torch.int32 and block_table.stride(1) == 1
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    B, q_len = int(q.shape[0]), int(q.shape[1])
    st = load().msa_indexer_decode_mq(
        _ptr(q), q_len, _ptr(kcache_pool), int(kcache_pool.shape[0]), _ptr(block_table),
        int(block_table.stride(0)), _ptr(seq_lens), B, B if max_batch is None else max_batch,
        max_model_len, k, n_sink, n_window, _ptr(out_ids), _ptr(out_scores),
        _ptr(out_block_scores), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
        split_blocks, _stream_ptr(stream))
    _check(st, "msa_indexer_decode_mq")


def msa_indexer_prefill_workspace_bytes(max_total_q: int, max_model_len: int) -> int:
    return int(load().msa_indexer_prefill_workspace_bytes(max_total_q, max_model_len))


def msa_indexer_prefill(q, cu_seqlens_q, kcache_pool, block_table, seq_lens, k: int, n_sink: int,
                        n_window: int, out_ids, out_scores, workspace, *, max_model_len: int,
                        out_block_scores=None, stream=None) -> None:
    """msa_indexer_prefill(): q bf16 [total_q, 4, 128], cu_seqlens_q int32 [B + 1]."""
    import torch
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and tuple(q.shape[1:]) == (4, 128)
    assert cu_seqlens_q.dtype == torch.int32 and cu_seqlens_q.is_contiguous()
    assert kcache_pool.dtype == torch.bfloat16 and kcache_pool.is_contiguous()
    assert block_table.dtype == torch.int32 and block_table.stride(1) == 1
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    st = load().msa_indexer_prefill(
        _ptr(q), _ptr(cu_seqlens_q), int(q.shape[0]), _ptr(kcache_pool), int(kcache_pool.shape[0]),
        _ptr(block_table), int(block_table.stride(0)), _ptr(seq_lens), int(seq_lens.shape[0]),
        max_model_len, k, n_sink, n_window, _ptr(out_ids), _ptr(out_scores), _ptr(out_block_scores),
        _ptr(workspace), int(workspace.numel() * workspace.element_size()), _stream_ptr(stream))
    _check(st, "msa_indexer_prefill")


def msa_indexer_prefill_score(q, cu_seqlens_q, kcache_pool, block_table, seq_lens, out_block_scores,
                              workspace, *, max_model_len: int, stream=None) -> None:
    """msa_indexer_prefill_score(): block scores only, fp32 [total_q, 4, ceil(max_model_len/128)]."""
    import torch
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and tuple(q.shape[1:]) == (4, 128)
    assert cu_seqlens_q.dtype == torch.int32 and cu_seqlens_q.is_contiguous()
    assert kcache_pool.dtype == torch.bfloat16 and kcache_pool.is_contiguous()
    assert block_table.dtype == torch.int32 and block_table.stride(1) == 1
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    assert out_block_scores.dtype == torch.float32 and out_block_scores.is_contiguous()
    st = load().msa_indexer_prefill_score(
        _ptr(q), _ptr(cu_seqlens_q), int(q.shape[0]), _ptr(kcache_pool), int(kcache_pool.shape[0]),
        _ptr(block_table), int(block_table.stride(0)), _ptr(seq_lens), int(seq_lens.shape[0]),
        max_model_len, _ptr(out_block_scores), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _stream_ptr(stream))
    _check(st, "msa_indexer_prefill_score")


def _prefill_fp8_args(q, cu_seqlens_q, kcache_fp8, kscale, block_table, seq_lens):
    import torch
    assert q.dtype == torch.bfloat16 and q.is_contiguous() and tuple(q.shape[1:]) == (4, 128)
    assert cu_seqlens_q.dtype == torch.int32 and cu_seqlens_q.is_contiguous()
    assert kcache_fp8.element_size() == 1 and kcache_fp8.is_contiguous(), "kcache_fp8: 1-byte E4M3 codes"
    assert tuple(kcache_fp8.shape[1:]) == (MSA_PAGE_TOKENS, MSA_HEAD_DIM)
    assert kscale.dtype == torch.float32 and kscale.is_contiguous()
    assert tuple(kscale.shape) == tuple(kcache_fp8.shape[:2])
    assert block_table.dtype == torch.int32 and block_table.stride(1) == 1
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()


def msa_indexer_prefill_fp8(q, cu_seqlens_q, kcache_fp8, kscale, block_table, seq_lens, k: int,
                            n_sink: int, n_window: int, out_ids, out_scores, workspace, *,
                            max_model_len: int, out_block_scores=None, stream=None) -> None:
    """msa_indexer_prefill_fp8(): prefill scoring on the E4M3 cache."""
    _prefill_fp8_args(q, cu_seqlens_q, kcache_fp8, kscale, block_table, seq_lens)
    st = load().msa_indexer_prefill_fp8(
        _ptr(q), _ptr(cu_seqlens_q), int(q.shape[0]), _ptr(kcache_fp8), _ptr(kscale),
        int(kcache_fp8.shape[0]), _ptr(block_table), int(block_table.stride(0)), _ptr(seq_lens),
        int(seq_lens.shape[0]), max_model_len, k, n_sink, n_window, _ptr(out_ids), _ptr(out_scores),
        _ptr(out_block_scores), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
        _stream_ptr(stream))
    _check(st, "msa_indexer_prefill_fp8")


def msa_indexer_prefill_score_fp8(q, cu_seqlens_q, kcache_fp8, kscale, block_table, seq_lens,
                                  out_block_scores, workspace, *, max_model_len: int,
                                  stream=None) -> None:
    """msa_indexer_prefill_score_fp8(): block scores only, on the E4M3 cache."""
    _prefill_fp8_args(q, cu_seqlens_q, kcache_fp8, kscale, block_table, seq_lens)
    st = load().msa_indexer_prefill_score_fp8(
        _ptr(q), _ptr(cu_seqlens_q), int(q.shape[0]), _ptr(kcache_fp8), _ptr(kscale),
        int(kcache_fp8.shape[0]), _ptr(block_table), int(block_table.stride(0)), _ptr(seq_lens),
        int(seq_lens.shape[0]), max_model_len, _ptr(out_block_scores), _ptr(workspace),
        int(workspace.numel() * workspace.element_size()), _stream_ptr(stream))
    _check(st, "msa_indexer_prefill_score_fp8")


def msa_indexer_test_withhold_pages(on: bool) -> None:
    """Test hook: while set, bf16 decode and prefill passes load nothing and their waits run out (see the C header)."""
    load().msa_indexer_test_withhold_pages(1 if on else 0)


def msa_indexer_get_error(workspace, *, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    st = load().msa_indexer_get_error(_ptr(workspace), _stream_ptr(stream), ctypes.byref(flags))
    _check(st, "msa_indexer_get_error")
    return int(flags.value)


def new_workspace(max_batch: int, max_model_len: int, k: int, split_blocks: int = 0,
                  device=None, q_len: int = 1):
    """A zero-filled uint8 CUDA tensor of msa_indexer_workspace_bytes_mq() bytes."""
    import torch
    n = msa_indexer_workspace_bytes_mq(max_batch, max_model_len, k, split_blocks, q_len)
    if n == 0:
        raise MsaError(MSA_ERR_UNSUPPORTED, "msa_indexer_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")
