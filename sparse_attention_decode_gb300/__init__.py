"""Decode-time MSA lightning indexer for GB300 (sm_103a).

The compute lives in ``libmsa_indexer.so`` (hand-written CUDA kernels behind
a C ABI, declared in ``include/msa_indexer.h``); this package only builds and
binds it.  PyTorch supplies device memory and streams.
"""

from ._binding import (  # noqa: F401
    EXPORTED,
    MSA_ERR_CUDA,
    MSA_ERR_INVALID_ARG,
    MSA_ERR_UNSUPPORTED,
    MSA_ERR_WORKSPACE_TOO_SMALL,
    MSA_FAULT_PAGE_ID,
    MSA_FAULT_SEQ_LEN,
    MSA_FAULT_SLOTS,
    MSA_FAULT_TIMEOUT,
    MSA_HEAD_DIM,
    MSA_MAX_BATCH,
    MSA_MAX_TOPK,
    MSA_NOALLOC_WORKSPACE_BYTES,
    MSA_NUM_HEADS,
    MSA_OK,
    MSA_PAGE_TOKENS,
    MsaError,
    library_path,
    load,
    msa_indexer_decode,
    msa_indexer_decode_noalloc,
    msa_indexer_decode_fp8,
    msa_indexer_decode_mq,
    msa_indexer_decode_mq_fp8,
    msa_indexer_decode_pages,
    msa_indexer_prefill,
    msa_indexer_prefill_fp8,
    msa_indexer_prefill_score,
    msa_indexer_prefill_score_fp8,
    msa_indexer_prefill_workspace_bytes,
    msa_indexer_workspace_bytes_mq,
    msa_indexer_score_fp8,
    msa_indexer_expand_pages,
    msa_indexer_get_error,
    msa_indexer_merge,
    msa_indexer_score,
    msa_indexer_test_withhold_pages,
    msa_indexer_workspace_bytes,
    msa_status_string,
    new_workspace,
)
