/*
 * msa_indexer.h -- C ABI of the decode-time MSA lightning indexer on GB300.
 *
 * What the library computes.  For each decode request b and each of the four
 * index-query heads h, every 128-token block j of the request's paged,
 * single-head index-K cache gets the score
 *
 *     s[b,h,j] = max over valid tokens t of block j of  sum_d q[b,h,d] * K[page(b,j),t,d]
 *
 * with fp32 accumulation and no scale (TensorRT-LLM PR #17008, "Description":
 * a full-kv_len MQA max-score pass that scores every KV block so top-k can
 * pick 16; vLLM blog "Following the Bottleneck: Optimizing MiniMax M3 on AMD
 * Instinct MI355X", section 2: the positive score scale was removed because
 * only the top-k order matters).  Each head then keeps its own top-k blocks
 * (vLLM PR #57832, "Solution", steps 3-4), with the first n_sink and the last
 * n_window blocks pinned inside the k outputs (same page, "Solution": forced
 * init/sink and sliding-window blocks are pinned; SGLang PR #41488,
 * "Modifications": initial/recent block priorities are preserved).
 *
 * Fixed shapes: 4 index heads, head dim 128, 128-token pages, bf16 inputs
 * (vLLM PR #57832, "Problem": index heads == KV heads == 4, one shared
 * index-K head; SGLang PR #41488, "Modifications": dimension 128, 128-token
 * blocks, top-k 16).
 *
 * Output order per (b, h): the pinned blocks in increasing block id, then the
 * other selected blocks by higher score first and, on equal fp32 scores,
 * lower block id first.  Ids are logical block indices within the request.
 * Unused slots (fewer than k blocks, or an empty request) hold id -1 and
 * score -inf.  The reported score of every selected block, pinned ones
 * included, is its fp32 block score.
 *
 * Memory.  Every pointer is device memory owned by the caller; the library
 * allocates, frees and synchronises nothing inside msa_indexer_decode /
 * _score / _merge.  All work is enqueued on `stream` (a cudaStream_t passed
 * as void*; NULL = the legacy default stream), so the calls can be recorded
 * into a CUDA graph.  Kernel shapes depend only on the bounds (batch,
 * max_model_len, split_blocks) and the SM count, never on the live seq_lens
 * (vLLM PR #57832, "CUDA graph capture": kernel shapes must be
 * capture-stable and come from max_model_len; block counts are runtime
 * values).
 *
 * Errors.  Argument errors are returned synchronously before anything is
 * enqueued.  Bad device data is not an error status (the host never reads
 * it): a seq_len outside [0, min(max_model_len, 128*bt_stride)] makes that
 * request empty (ids -1 / scores -inf); a block-table entry outside
 * [0, num_pages) makes that block score -inf and excludes it from the
 * selection.  Both set a bit in the workspace fault word, read (and cleared)
 * by msa_indexer_get_error().  No kernel traps or waits without bound: every
 * wait inside a kernel gives up after a fixed number of polls and sets
 * MSA_FAULT_TIMEOUT; the merge (decode) or the top-k (prefill) of a pass in
 * which that happened writes -1 / -inf to every output row, and the workspace
 * stays usable for the next call.
 *
 * Concurrency.  The library keeps no state between calls except in the
 * caller's workspace.  Calls that may overlap on the GPU need separate
 * workspaces.
 */
#ifndef MSA_INDEXER_H
#define MSA_INDEXER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSA_NUM_HEADS 4
#define MSA_HEAD_DIM 128
#define MSA_PAGE_TOKENS 128
#define MSA_MAX_TOPK 32     /* largest k accepted */
#define MSA_MAX_BATCH 4096  /* largest batch / max_batch accepted */
#define MSA_MAX_GRID 1024   /* bound on score CTAs used to size auto-mode workspaces */

typedef enum msa_status {
    MSA_OK = 0,
    MSA_ERR_INVALID_ARG = 1,         /* a null pointer, a bad size or an unaligned pointer */
    MSA_ERR_UNSUPPORTED = 2,         /* a size the kernels do not handle (k > MSA_MAX_TOPK, ...) */
    MSA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below msa_indexer_workspace_bytes() */
    MSA_ERR_CUDA = 4                 /* a CUDA runtime call or a launch failed */
} msa_status;

/* Bits of the workspace fault word (see msa_indexer_get_error). */
#define MSA_FAULT_SEQ_LEN 0x1u /* a seq_len outside [0, min(max_model_len, 128*bt_stride)] */
#define MSA_FAULT_PAGE_ID 0x2u /* a block-table entry outside [0, num_pages) */
#define MSA_FAULT_TIMEOUT 0x4u /* a bounded wait inside a kernel ran out (the call's rows are -1 / -inf) */
#define MSA_FAULT_SLOTS 0x8u   /* the workspace held fewer candidate slots than needed */

/*
 * Bytes of device workspace the calls below need for any batch <= max_batch
 * and any seq_len <= max_model_len, with top-k `k` and split width
 * `split_blocks` (0 = automatic).  Depends on the bounds only.  Returns 0
 * for arguments the library rejects.
 *
 * The workspace must be zero-filled once before its first use (for example
 * cudaMemset or torch.zeros); afterwards the library keeps it consistent.
 * It is 256-byte aligned storage owned by the caller.
 *
 * No passage of the pages defines this call; it is this library's own.  It
 * follows from two things the pages do fix: buffers are persistent and
 * allocated once (vLLM PR #57832, "CUDA graph capture": the indexer keeps
 * persistent buffers; TensorRT-LLM PR #17008, "Changes": graph-safe plan
 * buffers sized for the maximum work), and shapes come from bounds such as
 * max_model_len, never from the live lengths (vLLM PR #57832, same section).
 */
size_t msa_indexer_workspace_bytes(int max_batch, int max_model_len, int k, int split_blocks);

/*
 * One decode step of the indexer: block scores, pins, per-head top-k.
 * Enqueues two kernels on `stream`: msa_indexer_score() then
 * msa_indexer_merge().
 *
 *   q             bf16 [batch, 4, 128], contiguous, 16-byte aligned; the
 *                 post-RoPE index queries (SGLang PR #41488, "Modifications":
 *                 the existing post-RoPE queries are used).
 *   kcache_pool   bf16 [num_pages, 128, 128] (page, token, dim), contiguous,
 *                 16-byte aligned; the paged single-head index-K cache.
 *   num_pages     pages in the pool, 1 <= num_pages <= 2^24.
 *   block_table   int32 [batch, bt_stride]; entry (b, j) is the physical
 *                 page of logical block j of request b.  Only entries
 *                 j < ceil(seq_lens[b] / 128) are read.
 *   bt_stride     row stride of block_table in entries, >= 1.
 *   seq_lens      int32 [batch]: tokens of request b, the current one included.
 *   batch         requests, 0 <= batch <= max_batch (0 enqueues nothing).
 *   max_batch     the bound the workspace was sized for, <= MSA_MAX_BATCH.
 *   max_model_len the bound on seq_len the workspace was sized for, >= 1.
 *   k             outputs per head, 1 <= k <= MSA_MAX_TOPK.
 *   n_sink        leading blocks pinned, >= 0.
 *   n_window      trailing blocks pinned, >= 0; n_sink + n_window <= k.
 *   out_ids       int32 [batch, 4, k]: selected logical block ids.
 *   out_scores    fp32  [batch, 4, k]: their fp32 block scores.
 *   out_block_scores  optional fp32 [batch, 4, bt_stride]: every block's
 *                 score (entries j >= ceil(seq_len/128) are left untouched);
 *                 NULL to skip.
 *   workspace     caller-owned device scratch of workspace_bytes bytes,
 *                 >= msa_indexer_workspace_bytes(max_batch, max_model_len,
 *                 k, split_blocks), 256-byte aligned, zero-filled before its
 *                 first use.
 *   split_blocks  pages each score work unit covers; 0 = automatic (the
 *                 batch's pages spread evenly over one CTA per SM).  Any
 *                 value gives bitwise-identical results.
 *   stream        cudaStream_t as void*.
 *
 * Returns MSA_OK when both kernels were enqueued.
 */
msa_status msa_indexer_decode(const void *q, const void *kcache_pool, int64_t num_pages,
                              const int32_t *block_table, int64_t bt_stride,
                              const int32_t *seq_lens, int batch, int max_batch,
                              int max_model_len, int k, int n_sink, int n_window,
                              int32_t *out_ids, float *out_scores, float *out_block_scores,
                              void *workspace, size_t workspace_bytes, int split_blocks,
                              void *stream);

/*
 * The first stage of msa_indexer_decode alone: gathers every page of every
 * request once (all four heads scored while the tile is resident), forms the
 * block scores and the packed (score, block id) keys, and leaves each work
 * unit's own top-k per head in the workspace.  Keeping the full top-k per
 * unit makes the later merge exact (vLLM PR #57832, "Solution": a block in a
 * head's global top-k is necessarily in its own shard's top-k).  Same
 * arguments as msa_indexer_decode minus the outputs.
 */
msa_status msa_indexer_score(const void *q, const void *kcache_pool, int64_t num_pages,
                             const int32_t *block_table, int64_t bt_stride,
                             const int32_t *seq_lens, int batch, int max_batch,
                             int max_model_len, int k, int n_sink, int n_window,
                             float *out_block_scores, void *workspace, size_t workspace_bytes,
                             int split_blocks, void *stream);

/*
 * msa_indexer_score / msa_indexer_decode on an FP8 E4M3 index-K cache (the
 * cache format SGLang PR #41488 measured: "BF16 queries, FP8 E4M3 index
 * cache").  The pages do not give the scale convention; here every token has
 * one fp32 scale: K[t, d] = e4m3(code[t, d]) * kscale[page, t].
 *
 *   kcache_fp8  uint8 [num_pages, 128, 128] E4M3 codes (page, token, dim),
 *               contiguous, 16-byte aligned.
 *   kscale      fp32 [num_pages, 128] per-token scales, 16-byte aligned.
 *
 * Everything else is as for the bf16 calls (same workspace, same outputs,
 * same msa_indexer_merge).  The products run on f16 tensor cores: E4M3 codes
 * convert exactly to f16, and q is converted to f16 after multiplying each
 * head by a power of two that puts its largest |q| in [2^13, 2^14), which is
 * exact for bf16 inputs whose magnitude lies within 2^-14 .. 2^14 of that
 * largest value.
 */
msa_status msa_indexer_score_fp8(const void *q, const void *kcache_fp8, const float *kscale,
                                 int64_t num_pages, const int32_t *block_table, int64_t bt_stride,
                                 const int32_t *seq_lens, int batch, int max_batch,
                                 int max_model_len, int k, int n_sink, int n_window,
                                 float *out_block_scores, void *workspace, size_t workspace_bytes,
                                 int split_blocks, void *stream);

msa_status msa_indexer_decode_fp8(const void *q, const void *kcache_fp8, const float *kscale,
                                  int64_t num_pages, const int32_t *block_table, int64_t bt_stride,
                                  const int32_t *seq_lens, int batch, int max_batch,
                                  int max_model_len, int k, int n_sink, int n_window,
                                  int32_t *out_ids, float *out_scores, float *out_block_scores,
                                  void *workspace, size_t workspace_bytes, int split_blocks,
                                  void *stream);

/*
 * Several query positions per request (msa_indexer_decode_mq) on the E4M3
 * cache of msa_indexer_decode_fp8: q is bf16 [batch, q_len, 4, 128] with
 * q_len in {1, 2, 4}; position i sees the first seq_len - (q_len - 1 - i)
 * tokens; outputs are [batch, q_len, 4, k] (out_block_scores
 * [batch, q_len, 4, bt_stride]).  The workspace is sized by
 * msa_indexer_workspace_bytes_mq.  Two kernels.
 */
msa_status msa_indexer_decode_mq_fp8(const void *q, int q_len, const void *kcache_fp8,
                                     const float *kscale, int64_t num_pages,
                                     const int32_t *block_table, int64_t bt_stride,
                                     const int32_t *seq_lens, int batch, int max_batch,
                                     int max_model_len, int k, int n_sink, int n_window,
                                     int32_t *out_ids, float *out_scores, float *out_block_scores,
                                     void *workspace, size_t workspace_bytes, int split_blocks,
                                     void *stream);

/*
 * Several query positions per request: speculative-decode verification runs
 * the indexer for the last q_len tokens at once (vLLM PR #57832, "Test
 * Plan": query_len 1/4; vLLM blog "Following the Bottleneck", section 2: one
 * workgroup per request processes all draft positions together, reusing the
 * key loads).  Position i (0-based) sees the first seq_len - (q_len - 1 - i)
 * tokens (TensorRT-LLM PR #17008, "Description": the causal clamp
 * eff_kv = min(q_end + offset_q, kv_len)); pins and the top-k are per
 * position and head.  Each index-K page is read once for all q_len x 4
 * (position, head) columns.
 *
 *   q          bf16 [batch, q_len, 4, 128], q_len in {1, 2, 4}.
 *   out_ids    int32 [batch, q_len, 4, k]; out_scores fp32 [batch, q_len, 4, k];
 *   out_block_scores  optional fp32 [batch, q_len, 4, bt_stride].
 *   workspace  >= msa_indexer_workspace_bytes_mq(..., q_len) bytes.
 *
 * Other arguments as for msa_indexer_decode (bf16 cache).
 */
size_t msa_indexer_workspace_bytes_mq(int max_batch, int max_model_len, int k, int split_blocks,
                                      int q_len);

msa_status msa_indexer_decode_mq(const void *q, int q_len, const void *kcache_pool,
                                 int64_t num_pages, const int32_t *block_table, int64_t bt_stride,
                                 const int32_t *seq_lens, int batch, int max_batch,
                                 int max_model_len, int k, int n_sink, int n_window,
                                 int32_t *out_ids, float *out_scores, float *out_block_scores,
                                 void *workspace, size_t workspace_bytes, int split_blocks,
                                 void *stream);

/*
 * The second stage alone: merges the per-unit top-k lists that the last
 * msa_indexer_score() on this workspace left, per (request, head), into the
 * exact top-k (vLLM PR #57832, "Solution", step 4: merge per head) and
 * writes out_ids / out_scores.  `batch` and `k` must equal those of that
 * msa_indexer_score() call.
 */
msa_status msa_indexer_merge(int batch, int k, int32_t *out_ids, float *out_scores,
                             const void *workspace, size_t workspace_bytes, void *stream);

/*
 * Expands each selected 128-token block into the ids of the smaller KV-cache
 * pages it spans, so a sparse attention kernel that reads the KV cache in
 * `page_tokens`-token pages can consume the selection through a compact page
 * table without moving KV data (vLLM blog "Following the Bottleneck:
 * Optimizing MiniMax M3 on AMD Instinct MI355X", section 3 "Which bytes
 * move?", figure 5: each selected block id becomes eight 16-token page ids).
 *
 *   ids            int32 [batch, 4, k]: selected block ids as written by
 *                  msa_indexer_decode (-1 = none; ids outside the request
 *                  are ignored).
 *   seq_lens       int32 [batch]: the same lengths the selection used.
 *   kv_block_table int32 [batch, kv_bt_stride]: small page p of request b ->
 *                  physical KV page.  Entries p < min(ceil(seq_len /
 *                  page_tokens), kv_bt_stride) are read.
 *   page_tokens    a divisor of 128 (16 for eight pages per block).
 *   out_pages      int32 [batch, 4, k * 128 / page_tokens]: per (request,
 *                  head) the selected blocks in increasing block id, each as
 *                  its existing small pages in order, then -1.
 *   out_num_pages  int32 [batch, 4]: entries used in each row of out_pages.
 *
 * All device memory, enqueued on `stream`; one kernel, no workspace.
 */
msa_status msa_indexer_expand_pages(const int32_t *ids, int batch, int k, const int32_t *seq_lens,
                                    const int32_t *kv_block_table, int64_t kv_bt_stride,
                                    int page_tokens, int32_t *out_pages, int32_t *out_num_pages,
                                    void *stream);

/*
 * msa_indexer_decode followed by msa_indexer_expand_pages, with the
 * expansion fused into the merge kernel (the last warp step of each (request,
 * head) merge), so the selection reaches the page table without a third
 * launch.  Arguments are those of the two calls; out_pages / out_num_pages
 * get exactly what msa_indexer_expand_pages would write for this call's
 * out_ids.  Two kernels.
 */
msa_status msa_indexer_decode_pages(const void *q, const void *kcache_pool, int64_t num_pages,
                                    const int32_t *block_table, int64_t bt_stride,
                                    const int32_t *seq_lens, int batch, int max_batch,
                                    int max_model_len, int k, int n_sink, int n_window,
                                    int32_t *out_ids, float *out_scores, float *out_block_scores,
                                    void *workspace, size_t workspace_bytes, int split_blocks,
                                    const int32_t *kv_block_table, int64_t kv_bt_stride,
                                    int page_tokens, int32_t *out_pages, int32_t *out_num_pages,
                                    void *stream);

/*
 * Prefill scoring: every new token of every request selects blocks over its
 * own causal prefix (vLLM PR #57832: the prefill branch scores iq[nd:] with
 * cu_seqlens_q and takes the per-token top-k).  Request b's new tokens are
 * its last n_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] tokens; new token t
 * sits at position seq_lens[b] - n_b + t and sees tokens [0, position].
 * Pins and top-k are per (token, head), over that token's block count.
 *
 *   q             bf16 [total_q, 4, 128]: rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1
 *                 are request b's new tokens in order (may be NULL when
 *                 total_q is 0: nothing is launched).
 *   cu_seqlens_q  int32 [batch + 1], non-decreasing, cu_seqlens_q[batch] <= total_q.
 *   seq_lens      int32 [batch]: tokens of request b including its new ones.
 *   out_ids / out_scores  [total_q, 4, k].
 *   out_block_scores      optional fp32 [total_q, 4, ceil(max_model_len/128)]:
 *                 block scores of each token's visible blocks (others untouched).
 *   workspace     >= msa_indexer_prefill_workspace_bytes(total_q, max_model_len)
 *                 bytes (256 when out_block_scores is given), 256-byte aligned,
 *                 zero-filled before first use.
 *
 * Requests with inconsistent rows or lengths produce -1 / -inf and set
 * MSA_FAULT_SEQ_LEN; bad pages set MSA_FAULT_PAGE_ID (read with
 * msa_indexer_get_error on this workspace).  bf16 cache; two kernels.
 */
size_t msa_indexer_prefill_workspace_bytes(int max_total_q, int max_model_len);

/*
 * msa_indexer_prefill on the E4M3 cache of msa_indexer_decode_fp8
 * (kcache_fp8 uint8 [num_pages, 128, 128] codes, kscale fp32 [num_pages, 128]
 * per-token scales, 16-byte aligned).  The keys are widened to f16 exactly
 * and each query row is scaled to f16 by a power of two (exact for values
 * within 2^-14..2^14 of the row's largest |q|) before the tensor-core
 * product; the per-token scale multiplies each key's product before the max.
 * Other arguments, layouts and errors as msa_indexer_prefill.  Two kernels.
 */
msa_status msa_indexer_prefill_fp8(const void *q, const int32_t *cu_seqlens_q, int total_q,
                                   const void *kcache_fp8, const float *kscale, int64_t num_pages,
                                   const int32_t *block_table, int64_t bt_stride,
                                   const int32_t *seq_lens, int batch, int max_model_len, int k,
                                   int n_sink, int n_window, int32_t *out_ids, float *out_scores,
                                   float *out_block_scores, void *workspace,
                                   size_t workspace_bytes, void *stream);

/* The block-score half of msa_indexer_prefill_fp8 (see msa_indexer_prefill_score). */
msa_status msa_indexer_prefill_score_fp8(const void *q, const int32_t *cu_seqlens_q, int total_q,
                                         const void *kcache_fp8, const float *kscale,
                                         int64_t num_pages, const int32_t *block_table,
                                         int64_t bt_stride, const int32_t *seq_lens, int batch,
                                         int max_model_len, float *out_block_scores,
                                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * The block-score half of msa_indexer_prefill: writes out_block_scores
 * (required, fp32 [total_q, 4, ceil(max_model_len/128)], each token's
 * visible blocks only) and nothing else.  The workspace needs only its
 * 256-byte header (the fault word and pass count).  After MSA_FAULT_TIMEOUT
 * the block scores of that pass are incomplete.  One kernel.
 */
msa_status msa_indexer_prefill_score(const void *q, const int32_t *cu_seqlens_q, int total_q,
                                     const void *kcache_pool, int64_t num_pages,
                                     const int32_t *block_table, int64_t bt_stride,
                                     const int32_t *seq_lens, int batch, int max_model_len,
                                     float *out_block_scores, void *workspace,
                                     size_t workspace_bytes, void *stream);

msa_status msa_indexer_prefill(const void *q, const int32_t *cu_seqlens_q, int total_q,
                               const void *kcache_pool, int64_t num_pages,
                               const int32_t *block_table, int64_t bt_stride,
                               const int32_t *seq_lens, int batch, int max_model_len, int k,
                               int n_sink, int n_window, int32_t *out_ids, float *out_scores,
                               float *out_block_scores, void *workspace, size_t workspace_bytes,
                               void *stream);

/*
 * Reads the workspace fault word (MSA_FAULT_* bits) into *flags and clears
 * it.  Synchronises `stream`.  Returns MSA_ERR_INVALID_ARG for null
 * pointers, MSA_ERR_CUDA if a CUDA call fails.
 *
 * No passage of the pages defines this call; it is this library's own way
 * of reporting bad device data without a host read inside the decode call.
 * The pages treat unsupported configurations as start-up errors (vLLM PR
 * #57832, "Solution": enabling the path with a non-bf16 index cache fails at
 * start-up) and a short plan mirror after capture as a hard error
 * (TensorRT-LLM PR #17008, "Changes"); device
 * data cannot be checked on the host without a synchronisation, so it is
 * flagged here instead.
 */
msa_status msa_indexer_get_error(void *workspace, void *stream, uint32_t *flags);

/*
 * Test hook for the bounded waits.  No passage of the pages corresponds; it
 * exists so that a test can make the kernels' waits run out without any
 * fault: while `on` is non-zero, bf16 one-position decode and score passes
 * with k <= 16 enqueued afterwards run a separately built copy of the score
 * kernel that loads no index-K page and never signals one, so every
 * consumer's first page wait runs out after a short poll limit (2^14 polls)
 * instead of the normal one; bf16 prefill and prefill-score passes likewise
 * run a copy of the prefill scoring kernel that loads no query row and no
 * page.  No asynchronous copy is in flight at any time.  The pass then sets
 * MSA_FAULT_TIMEOUT, and its merge or top-k writes -1 / -inf to every output
 * row (a prefill-score pass leaves its block scores incomplete).  Other
 * shapes, and the E4M3 prefill, return MSA_ERR_UNSUPPORTED while it is set.
 * Set it back to 0 for normal operation.  The flag is process-wide: do not
 * set it while other threads run calls.
 */
void msa_indexer_test_withhold_pages(int on);

/*
 * msa_indexer_decode without a caller-supplied workspace.  The pages describe
 * no such call; it exists for callers that cannot allocate device memory
 * themselves: a plugin inside a host framework whose allocator owns all of
 * the GPU's memory, or code that may not call cudaMalloc (which can
 * synchronise the device) on its per-token path.
 *
 * The scratch lives in one fixed array of MSA_NOALLOC_WORKSPACE_BYTES in the
 * library's device memory (every GPU that loads the library keeps it until
 * the process exits).  The call allocates and frees nothing.  Each call looks
 * up the array's device address in the current context (a host-side query
 * that enqueues nothing), so a caller's own context, or a new one after
 * cudaDeviceReset, gets its own copy.  Loading the library's module into a
 * context can happen on the first call in it; make that first call before
 * any stream capture.
 *
 * Arguments are those of msa_indexer_decode with max_batch = batch and the
 * automatic split.  A batch whose scratch would not fit returns
 * MSA_ERR_UNSUPPORTED before anything is enqueued; the scratch a batch needs
 * is what msa_indexer_decode checks a caller's workspace against, with the
 * grid of this GPU (at most its SM count of score CTAs) in place of
 * MSA_MAX_GRID:
 *   256 + round_up(4*(batch+1), 256) + (7*CTAs + batch) * 4 * kmax * 8 bytes,
 * kmax = 16 for k <= 16 else 32.  On GB300 (152 SMs) every batch up to 1024
 * fits for any k.  Every call uses the same array and leaves its contents
 * behind.  The words that must start at zero (two ticket counters in the
 * header) are zero when the module is loaded into a context and every call
 * returns them to zero; everything else a call reads it wrote earlier on the
 * GPU.  Calls that can overlap on the GPU (different streams,
 * different threads) race on the array: serialise them.  Data faults are
 * handled as in msa_indexer_decode but are not reported.
 */
#define MSA_NOALLOC_WORKSPACE_BYTES (4u * 1024u * 1024u)
msa_status msa_indexer_decode_noalloc(const void *q, const void *kcache_pool, int64_t num_pages,
                                      const int32_t *block_table, int64_t bt_stride,
                                      const int32_t *seq_lens, int batch, int max_model_len, int k,
                                      int n_sink, int n_window, int32_t *out_ids,
                                      float *out_scores, float *out_block_scores, void *stream);

/*
 * A static, human-readable name for a status code.  No passage of the pages
 * defines it; it belongs to this library's status codes (above).
 */
const char *msa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MSA_INDEXER_H */
