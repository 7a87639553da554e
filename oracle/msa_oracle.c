/*
 * CPU oracle for the decode-time MSA lightning indexer -- TEST INFRASTRUCTURE.
 *
 * This file is a plain, slow, deliberately unoptimised restatement of what
 * the decode indexer computes.  Only the tests, the package smoke check and
 * the CPU-baseline leg of the benchmark load it.  The CUDA library never
 * links it, includes it or calls it, and it shares no code with that library.
 *
 * What it computes (for every request b, index head h in [0,4), block j):
 *
 *   1. Block score.  s[b,h,j] = max over the valid tokens t of block j of
 *      sum_d q[b,h,d] * K[page(b,j), t, d], with no scale and no
 *      nonlinearity.  The indexer is an MQA pass over the whole context whose
 *      per-block result is the maximum token score (TensorRT-LLM PR #17008,
 *      "Description": a full-kv_len MQA max-score pass; SGLang PR #41488,
 *      "Modifications": max scoring).  No positive scale is applied because
 *      only the top-k order matters (vLLM blog "Following the Bottleneck:
 *      Optimizing MiniMax M3 on AMD Instinct MI355X", section 2 "What work
 *      repeats?").  Valid tokens are [0, seq_len): block j covers tokens
 *      [128 j, min(128 j + 128, seq_len)) (TensorRT-LLM PR #17008,
 *      "Description": the causal clamp eff_kv = min(q_end + offset_q, kv_len)).
 *      The whole sum is formed in double precision: bf16 -> double is exact,
 *      each product of two bf16 values is exact in double, and a 128-term
 *      double sum carries a relative error near 1e-14, far below the
 *      tolerance the GPU path is held to.
 *
 *   2. Pins.  The first n_sink blocks and the last n_window blocks of the
 *      request are always selected ("Forced init/sink and sliding-window
 *      blocks are pinned": vLLM PR #57832, "Solution"; "Initial/recent block
 *      priorities ... are preserved": SGLang PR #41488, "Modifications").
 *      pinned(j) = j < n_sink or j >= nb - n_window, with nb = ceil(seq_len/128).
 *      The pins take slots inside the k outputs (see the selection below).
 *
 *   3. Selection per head.  Each head selects on its own (vLLM PR #57832,
 *      "Solution" step 4 and the "Withdrawn" note: mixing heads is a bug).
 *      Output row = the pinned blocks in increasing block id, then the
 *      remaining blocks ordered by higher score first and, on equal scores,
 *      lower block id first, truncated to k entries.  When the request has
 *      fewer than k blocks every block is returned.  Unused slots hold id -1
 *      and score -inf.
 *
 *   4. Split-merge.  The context-parallel exactness argument (vLLM PR #57832,
 *      "Solution": a block in a head's global top-k is necessarily in the
 *      top-k of its own shard; SGLang PR #41488: keeping 16 candidates on
 *      every shard preserves the global top-16 even when all winners sit in
 *      one shard).  msa_oracle_select_split() partitions each row's blocks
 *      into contiguous splits, keeps the pins plus the top-k of every split,
 *      and selects again over that candidate set.  It must agree with the
 *      unsplit selection.
 *
 *   5. Page expansion.  The downstream sparse attention reads the KV cache in
 *      pages smaller than the indexer's 128-token blocks; each selected block
 *      is turned into the ids of the small pages it spans, through the KV
 *      cache's own block table, without moving KV data (vLLM blog "Following
 *      the Bottleneck", section 3 "Which bytes move?" and its figure 5: every
 *      selected block id becomes eight 16-token page ids in a compact page
 *      table).  msa_oracle_expand_pages() lists, per (request, head), the
 *      selected blocks in increasing block id, each expanded to its existing
 *      small pages in order, then pads with -1 and reports the count.
 *
 *   6. fp8 index-K cache.  The index cache may be stored as FP8 E4M3 (vLLM PR
 *      #57832, "Solution": the fp8 index cache is a separate path; SGLang PR
 *      #41488 measured "BF16 queries, FP8 E4M3 index cache").  The pages do
 *      not give the scale convention; the reading taken here is one fp32
 *      scale per token: K[t,d] = e4m3(code[t,d]) * scale[t].  E4M3 (OCP FP8):
 *      1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0
 *      encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; there is no inf.
 *      msa_oracle_block_scores_fp8() is step 1 on that cache, in fp64.
 *
 * Layouts (all host memory, row-major, caller-owned):
 *   q        uint16 bf16 bits [B][4][128]
 *   pool     uint16 bf16 bits [num_pages][128][128]   (page, token, dim)
 *   bt       int32 [B][bt_stride], logical block -> physical page
 *   seq_lens int32 [B]
 *   scores   double [B][4][bt_stride]; entries j >= nb are set to -inf
 *   out_ids  int32  [B][4][k];  out_scores double [B][4][k]
 *
 * Return value: 0 on success, a negative code for an argument the oracle
 * refuses (it is only ever fed valid inputs by the tests).
 */

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define HEADS 4
#define DIM 128
#define PAGE 128

/* A bf16 value is the upper half of an IEEE binary32 value. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* The value of an FP8 E4M3 code, from the format's definition. */
double msa_oracle_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int exponent = (code >> 3) & 0xF;
    int mantissa = code & 0x7;
    double magnitude;
    if (exponent == 0xF && mantissa == 0x7)
        return NAN;
    if (exponent == 0)
        magnitude = ldexp(mantissa / 8.0, -6);
    else
        magnitude = ldexp(1.0 + mantissa / 8.0, exponent - 7);
    return sign ? -magnitude : magnitude;
}

static int64_t blocks_of(int32_t seq_len)
{
    return ((int64_t)seq_len + PAGE - 1) / PAGE;
}

int msa_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the host threads later calls use (timing on one core or on all). */
void msa_oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Step 1: the score of every block of every request, for every head. */
int msa_oracle_block_scores(const uint16_t *q, const uint16_t *pool, int64_t num_pages,
                            const int32_t *bt, int64_t bt_stride, const int32_t *seq_lens,
                            int batch, double *scores)
{
    if (batch < 0 || bt_stride <= 0 || num_pages < 0)
        return -1;
    for (int b = 0; b < batch; ++b) {
        if (seq_lens[b] < 0 || blocks_of(seq_lens[b]) > bt_stride)
            return -2;
        for (int64_t j = 0; j < blocks_of(seq_lens[b]); ++j) {
            int32_t page = bt[(int64_t)b * bt_stride + j];
            if (page < 0 || page >= num_pages)
                return -3;
        }
    }

    int64_t units = (int64_t)batch * bt_stride;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t u = 0; u < units; ++u) {
        int b = (int)(u / bt_stride);
        int64_t j = u % bt_stride;
        int64_t nb = blocks_of(seq_lens[b]);
        for (int h = 0; h < HEADS; ++h) {
            double best = -INFINITY;
            if (j < nb) {
                int32_t page = bt[(int64_t)b * bt_stride + j];
                int64_t first_token = j * PAGE;
                int64_t valid = seq_lens[b] - first_token;
                if (valid > PAGE)
                    valid = PAGE;
                for (int64_t t = 0; t < valid; ++t) {
                    const uint16_t *krow = pool + ((int64_t)page * PAGE + t) * DIM;
                    const uint16_t *qrow = q + ((int64_t)b * HEADS + h) * DIM;
                    double dot = 0.0;
                    for (int d = 0; d < DIM; ++d)
                        dot += bf16_to_double(qrow[d]) * bf16_to_double(krow[d]);
                    if (dot > best)
                        best = dot;
                }
            }
            scores[((int64_t)b * HEADS + h) * bt_stride + j] = best;
        }
    }
    return 0;
}

typedef struct {
    double score;
    int64_t id;
} candidate;

/* Higher score first; on equal scores the lower block id first. */
static int by_score_then_id(const void *pa, const void *pb)
{
    const candidate *a = (const candidate *)pa;
    const candidate *b = (const candidate *)pb;
    if (a->score > b->score)
        return -1;
    if (a->score < b->score)
        return 1;
    if (a->id < b->id)
        return -1;
    if (a->id > b->id)
        return 1;
    return 0;
}

static int is_pinned(int64_t j, int64_t nb, int n_sink, int n_window)
{
    return j < n_sink || j >= nb - n_window;
}

/*
 * Select from the blocks listed in `ids` (count n, any order) of one head of
 * one request: the pinned ones in increasing id, then the others by
 * (score desc, id asc), truncated to k.  Writes k ids/scores, padded.
 */
static void select_from(const double *row_scores, const int64_t *ids, int64_t n, int64_t nb,
                        int k, int n_sink, int n_window, int32_t *out_ids, double *out_scores,
                        candidate *scratch)
{
    int64_t filled = 0;
    int64_t n_free = 0;

    /* pinned blocks, increasing id: ids[] may be unordered, so scan j upward */
    for (int64_t j = 0; j < nb && filled < k; ++j) {
        if (!is_pinned(j, nb, n_sink, n_window))
            continue;
        for (int64_t i = 0; i < n; ++i) {
            if (ids[i] == j) {
                out_ids[filled] = (int32_t)j;
                out_scores[filled] = row_scores[j];
                ++filled;
                break;
            }
        }
    }
    for (int64_t i = 0; i < n; ++i) {
        if (is_pinned(ids[i], nb, n_sink, n_window))
            continue;
        scratch[n_free].score = row_scores[ids[i]];
        scratch[n_free].id = ids[i];
        ++n_free;
    }
    qsort(scratch, (size_t)n_free, sizeof(candidate), by_score_then_id);
    for (int64_t i = 0; i < n_free && filled < k; ++i) {
        out_ids[filled] = (int32_t)scratch[i].id;
        out_scores[filled] = scratch[i].score;
        ++filled;
    }
    for (; filled < k; ++filled) {
        out_ids[filled] = -1;
        out_scores[filled] = -INFINITY;
    }
}

static int check_select_args(int batch, int64_t bt_stride, const int32_t *seq_lens, int k,
                             int n_sink, int n_window)
{
    if (batch < 0 || bt_stride <= 0 || k < 1 || n_sink < 0 || n_window < 0)
        return -1;
    if (n_sink + n_window > k)
        return -4;
    for (int b = 0; b < batch; ++b)
        if (seq_lens[b] < 0 || blocks_of(seq_lens[b]) > bt_stride)
            return -2;
    return 0;
}

/* Steps 2 and 3: pins plus the per-head top-k over all of a request's blocks. */
int msa_oracle_select(const double *scores, int batch, int64_t bt_stride, const int32_t *seq_lens,
                      int k, int n_sink, int n_window, int32_t *out_ids, double *out_scores)
{
    int rc = check_select_args(batch, bt_stride, seq_lens, k, n_sink, n_window);
    if (rc)
        return rc;
    int64_t *ids = (int64_t *)malloc((size_t)bt_stride * sizeof(int64_t));
    candidate *scratch = (candidate *)malloc((size_t)bt_stride * sizeof(candidate));
    if (!ids || !scratch) {
        free(ids);
        free(scratch);
        return -5;
    }
    for (int b = 0; b < batch; ++b) {
        int64_t nb = blocks_of(seq_lens[b]);
        for (int64_t j = 0; j < nb; ++j)
            ids[j] = j;
        for (int h = 0; h < HEADS; ++h) {
            int64_t row = (int64_t)b * HEADS + h;
            select_from(scores + row * bt_stride, ids, nb, nb, k, n_sink, n_window,
                        out_ids + row * k, out_scores + row * k, scratch);
        }
    }
    free(ids);
    free(scratch);
    return 0;
}

/*
 * Step 4: the same selection reached through contiguous splits of
 * `split_blocks` blocks.  Every split keeps its pins and its own top-k of the
 * rest; the final selection runs over the union of what the splits kept.
 */
int msa_oracle_select_split(const double *scores, int batch, int64_t bt_stride,
                            const int32_t *seq_lens, int k, int n_sink, int n_window,
                            int64_t split_blocks, int32_t *out_ids, double *out_scores)
{
    int rc = check_select_args(batch, bt_stride, seq_lens, k, n_sink, n_window);
    if (rc)
        return rc;
    if (split_blocks < 1)
        return -1;
    int64_t *ids = (int64_t *)malloc((size_t)bt_stride * sizeof(int64_t));
    int64_t *kept = (int64_t *)malloc((size_t)bt_stride * sizeof(int64_t));
    candidate *scratch = (candidate *)malloc((size_t)bt_stride * sizeof(candidate));
    int32_t *sid = (int32_t *)malloc((size_t)(k + bt_stride) * sizeof(int32_t));
    double *ssc = (double *)malloc((size_t)(k + bt_stride) * sizeof(double));
    if (!ids || !kept || !scratch || !sid || !ssc) {
        free(ids);
        free(kept);
        free(scratch);
        free(sid);
        free(ssc);
        return -5;
    }
    for (int b = 0; b < batch; ++b) {
        int64_t nb = blocks_of(seq_lens[b]);
        for (int h = 0; h < HEADS; ++h) {
            int64_t row = (int64_t)b * HEADS + h;
            const double *rs = scores + row * bt_stride;
            int64_t n_kept = 0;
            for (int64_t s0 = 0; s0 < nb; s0 += split_blocks) {
                int64_t s1 = s0 + split_blocks < nb ? s0 + split_blocks : nb;
                int64_t n = 0;
                for (int64_t j = s0; j < s1; ++j)
                    ids[n++] = j;
                /* the split's own selection: its pins, then its top-k of the rest */
                int64_t pins_here = 0;
                for (int64_t j = s0; j < s1; ++j)
                    pins_here += is_pinned(j, nb, n_sink, n_window);
                int split_k = k + (int)pins_here;
                select_from(rs, ids, n, nb, split_k, n_sink, n_window, sid, ssc, scratch);
                for (int i = 0; i < split_k; ++i)
                    if (sid[i] >= 0)
                        kept[n_kept++] = sid[i];
            }
            select_from(rs, kept, n_kept, nb, k, n_sink, n_window, out_ids + row * k,
                        out_scores + row * k, scratch);
        }
    }
    free(ids);
    free(kept);
    free(scratch);
    free(sid);
    free(ssc);
    return 0;
}

static int cmp_int(const void *pa, const void *pb)
{
    int a = *(const int *)pa, b = *(const int *)pb;
    return (a > b) - (a < b);
}

/*
 * Step 5: ids int32 [B][4][k] (as from msa_oracle_select, -1 = none);
 * kv_bt int32 [B][kv_stride]: small page p of request b -> physical page;
 * out_pages int32 [B][4][k * (128 / page_tokens)]; out_num int32 [B][4].
 */
int msa_oracle_expand_pages(const int32_t *ids, int batch, int k, const int32_t *seq_lens,
                            const int32_t *kv_bt, int64_t kv_stride, int page_tokens,
                            int32_t *out_pages, int32_t *out_num)
{
    if (batch < 0 || k < 1 || page_tokens < 1 || PAGE % page_tokens != 0 || kv_stride < 1)
        return -1;
    const int per_block = PAGE / page_tokens;
    const int64_t width = (int64_t)k * per_block;
    int *sel = (int *)malloc((size_t)k * sizeof(int));
    if (!sel)
        return -5;
    for (int b = 0; b < batch; ++b) {
        int64_t small_pages = seq_lens[b] > 0 ? ((int64_t)seq_lens[b] + page_tokens - 1) / page_tokens : 0;
        if (small_pages > kv_stride) {
            free(sel);
            return -2;
        }
        for (int h = 0; h < HEADS; ++h) {
            const int32_t *row = ids + ((int64_t)b * HEADS + h) * k;
            int32_t *out = out_pages + ((int64_t)b * HEADS + h) * width;
            int n_sel = 0;
            for (int r = 0; r < k; ++r)
                if (row[r] >= 0)
                    sel[n_sel++] = row[r];
            qsort(sel, (size_t)n_sel, sizeof(int), cmp_int);
            int64_t n = 0;
            for (int i = 0; i < n_sel; ++i) {
                for (int s = 0; s < per_block; ++s) {
                    int64_t p = (int64_t)sel[i] * per_block + s;
                    if (p < small_pages)
                        out[n++] = kv_bt[(int64_t)b * kv_stride + p];
                }
            }
            out_num[b * HEADS + h] = (int32_t)n;
            for (; n < width; ++n)
                out[n] = -1;
        }
    }
    free(sel);
    return 0;
}

/* Step 6: block scores on the fp8 cache: pool8 uint8 [num_pages][128][128]
 * E4M3 codes, kscale float [num_pages][128] per-token scales. */
int msa_oracle_block_scores_fp8(const uint16_t *q, const uint8_t *pool8, const float *kscale,
                                int64_t num_pages, const int32_t *bt, int64_t bt_stride,
                                const int32_t *seq_lens, int batch, double *scores)
{
    if (batch < 0 || bt_stride <= 0 || num_pages < 0)
        return -1;
    for (int b = 0; b < batch; ++b) {
        if (seq_lens[b] < 0 || blocks_of(seq_lens[b]) > bt_stride)
            return -2;
        for (int64_t j = 0; j < blocks_of(seq_lens[b]); ++j) {
            int32_t page = bt[(int64_t)b * bt_stride + j];
            if (page < 0 || page >= num_pages)
                return -3;
        }
    }
    int64_t units = (int64_t)batch * bt_stride;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t u = 0; u < units; ++u) {
        int b = (int)(u / bt_stride);
        int64_t j = u % bt_stride;
        int64_t nb = blocks_of(seq_lens[b]);
        for (int h = 0; h < HEADS; ++h) {
            double best = -INFINITY;
            if (j < nb) {
                int32_t page = bt[(int64_t)b * bt_stride + j];
                int64_t valid = seq_lens[b] - j * PAGE;
                if (valid > PAGE)
                    valid = PAGE;
                for (int64_t t = 0; t < valid; ++t) {
                    const uint8_t *krow = pool8 + ((int64_t)page * PAGE + t) * DIM;
                    const uint16_t *qrow = q + ((int64_t)b * HEADS + h) * DIM;
                    double scale = (double)kscale[(int64_t)page * PAGE + t];
                    double dot = 0.0;
                    for (int d = 0; d < DIM; ++d)
                        dot += bf16_to_double(qrow[d]) * (msa_oracle_e4m3_value(krow[d]) * scale);
                    if (dot > best)
                        best = dot;
                }
            }
            scores[((int64_t)b * HEADS + h) * bt_stride + j] = best;
        }
    }
    return 0;
}
