// Decode-time MSA lightning indexer for GB300 (sm_103a): kernels and C ABI.
//
// Two kernels per decode step:
//
//  score_kernel  (persistent, one CTA per SM)
//    a1  plan: page counts per request from the live seq_lens and their
//        prefix sums; the batch's pages are cut into equal chunks, so a long
//        request is spread over many CTAs and short ones share a CTA.
//    a2  gather: a producer warp issues one 2-D TMA pair per 32 KiB page
//        (page = block_table[b, j]) into a ring of shared-memory stages.
//    a3  score: a consumer warp multiplies the resident 128x128 tile by the
//        four query heads with mma.sync m16n8k16 (bf16 in, fp32 accumulate);
//        the tile is read once for all four heads.
//    a4  block max over the valid tokens (rows past seq_len are masked).
//    a5  pin and pack into 64-bit keys (keys.cuh).
//    a6  per-(chunk, request) top-kmax list per head in the workspace.
//
//  merge_kernel  (one CTA per (head, request))
//    a7  exact top-k of that request's chunk lists, decoded to ids/scores.
//
// The exactness of the split is the context-parallel argument of vLLM
// PR #57832 ("Solution"): a block in a head's global top-k is in the top-k of
// its own shard, so keeping the full top-k per shard and merging is exact.
// Splitting the KV axis across CTAs to shorten each CTA's serial chain is
// TensorRT-LLM PR #17008 ("Changes": num_kv_splits); max is exact, so the
// block scores do not depend on the split.

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "../../include/msa_indexer.h"
#include "keys.cuh"
#include "layout.cuh"
#include "ptx.cuh"
#include "host_util.cuh"

namespace msa {

// Cache formats.  A page of the index-K cache is 128 tokens x 128 dims:
//  Bf16Fmt: 32 KiB of bf16, moved as two 64x128 TMA boxes (128B swizzle);
//  Fp8Fmt:  16 KiB of E4M3 codes (one 128x128-byte TMA box) + 512 B of
//           per-token fp32 scales (one bulk copy).
// Pipeline shape per format: page number `it` (counted per CTA) is scored by
// consumer warp it % kConsumers in stage stage_of(it); every stage belongs to
// one consumer warp, so each full/empty barrier has a single waiter that sees
// its phases strictly in order (no warp can lap another warp's stage).  fp8
// pages arrive twice as often and cost more to score per byte, so that
// format runs four consumer warps.
struct Bf16Fmt {
    static constexpr bool kFp8 = false;
    static constexpr int kConsumers = 2;
    static constexpr int kStagesPer = 3;
    static constexpr int kDataBytes = kPageBytes;
    static constexpr int kScaleBytes = 0;
};

// bf16 pages for four query positions: 16 columns double each page's MMAs,
// so four consumer warps (one per SM sub-partition, one 32 KiB stage each)
// share the pages; measured 202 -> 175 us per call on the long-context batch.
// One-position passes of a few pages per SM use it too (wide_pass): there
// the pages come from L2 and the consumers' scoring, not HBM, sets the pace
// (16 x 8700 tokens: 10.35 -> 9.73 us a call; 32 x 128K tokens, which
// needs three stages per consumer to keep HBM busy, 155.6 -> 156.3 us).
struct Bf16Wide4Fmt {
    static constexpr bool kFp8 = false;
    static constexpr int kConsumers = 4;
    static constexpr int kStagesPer = 1;
    static constexpr int kDataBytes = kPageBytes;
    static constexpr int kScaleBytes = 0;
};

struct Fp8Fmt {
    static constexpr bool kFp8 = true;
    static constexpr int kConsumers = 4;
    static constexpr int kStagesPer = 3;
    static constexpr int kDataBytes = kPage * kDim;  // 16 KiB of E4M3 codes
    static constexpr int kScaleBytes = kPage * 4;    // 512 B: one fp32 per token
};

// fp8 pages for two or four query positions: the wider candidate lists leave
// room for two stages per consumer warp.
struct Fp8MqFmt {
    static constexpr bool kFp8 = true;
    static constexpr int kConsumers = 4;
    static constexpr int kStagesPer = 2;
    static constexpr int kDataBytes = kPage * kDim;
    static constexpr int kScaleBytes = kPage * 4;
};

template <class F>
struct Pipe {
    static constexpr int kConsumers = F::kConsumers;
    static constexpr int kStages = F::kConsumers * F::kStagesPer;
    static constexpr int kProducerWarp = kConsumers;
    static constexpr int kThreads = 32 * (kConsumers + 1);
    static constexpr int kConsumerThreads = 32 * kConsumers;
    static constexpr uint32_t kTxBytes = F::kDataBytes + F::kScaleBytes;

    __host__ __device__ static constexpr int stage_of(uint32_t it)
    {
        return static_cast<int>(it % kConsumers) +
               kConsumers * static_cast<int>((it / kConsumers) % F::kStagesPer);
    }
    // Use index of page `it` in its stage (its phase number on the barriers).
    __host__ __device__ static constexpr uint32_t use_of(uint32_t it) { return it / kStages; }
};

// Query columns of one request: NQ positions x 4 heads (column c = 4 * position
// + head), scored as the n dimension of m16n8k16 in kFrags fragments of 8.
template <int NQ>
struct Cols {
    static constexpr int kCols = 4 * NQ;
    static constexpr int kFrags = (kCols + 7) / 8;
};

struct ScoreParams {
    CUtensorMap tmap;  // pool as [num_pages*128 rows][128 elements] (format-specific boxes)
    const uint16_t *q;
    const float *kscale;  // fp8 only: [num_pages, 128] per-token scales
    const int32_t *block_table;
    const int32_t *seq_lens;
    float *out_block_scores;
    uint8_t *ws;
    int64_t bt_stride;
    int64_t num_pages;
    int batch;
    int seq_limit;
    int n_sink;
    int n_window;
    int split_blocks;
    int slot_capacity;
    int l2_keep_pages;  // passes of at most this many pages keep them in L2
};

constexpr int kChunkQueue = 8;  // chunk ids the producer may post ahead of the consumers

// Polls before a barrier wait gives up.  TH selects the kernel built for the
// bounded-wait test hook (msa_indexer_test_withhold_pages): its producer
// loads and signals no page, and its waits give up after far fewer polls.
// Both are compile-time: a wait bound read at run time slowed the E4M3
// kernel's page waits by ~11 %.
constexpr uint32_t kTestSpinLimit = 1u << 14;
template <bool TH>
constexpr uint32_t kWaitPolls = TH ? kTestSpinLimit : kSpinLimit;

template <class F>
struct SmemCtl {
    static constexpr int S = Pipe<F>::kStages;
    uint64_t full[S];                // page landed (1 producer arrival + TMA bytes)
    uint64_t empty[S];               // page consumed (its owner warp)
    uint64_t cq_full[kChunkQueue];   // chunk id posted (producer)
    uint64_t cq_empty[kChunkQueue];  // chunk id read (every consumer warp)
    uint64_t list_bar[2];            // lists of a segment written (every consumer thread)
    int2 meta[S];                    // (valid tokens, page ok)
    int chunk_q[kChunkQueue];
    int warp_sums[F::kConsumers + 1];
    volatile int abort_flag;
    uint32_t epoch;  // the workspace's pass count when this pass started
    Partition part;  // this pass's chunking, the same in every CTA
};

template <int KMAX, class F, int NQ = 1>
struct SmemLayout {
    static constexpr size_t stages = 0;  // kStages x kDataBytes, 1024-aligned
    static constexpr size_t scales = stages + static_cast<size_t>(Pipe<F>::kStages) * F::kDataBytes;
    static constexpr size_t ctl = round_up(scales + static_cast<size_t>(Pipe<F>::kStages) * F::kScaleBytes, 16);
    static constexpr size_t lists = round_up(ctl + sizeof(SmemCtl<F>), 16);
    static constexpr size_t list_entries = 2 * F::kConsumers * Cols<NQ>::kCols * KMAX;
    static constexpr size_t prefix = lists + list_entries * sizeof(uint64_t);
    static __host__ __device__ size_t bytes(int batch)
    {
        return 1024 /* alignment slack */ + prefix + sizeof(int32_t) * (batch + 1);
    }
};

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

// The request that owns batch page p: the largest b with prefix[b] <= p.
__device__ __forceinline__ int find_row(const int *prefix, int batch, int p)
{
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= p)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Pages of a request of L tokens; a length outside [0, seq_limit] is an
// empty request.  The score kernel's prefix and a decode call's merge both
// count pages with this rule.
__device__ __forceinline__ int pages_for_length(int L, int seq_limit)
{
    return (L < 0 || L > seq_limit) ? 0 : (L + kPage - 1) / kPage;
}

__device__ __forceinline__ int pages_of_request(const ScoreParams &p, int b)
{
    return pages_for_length(p.seq_lens[b], p.seq_limit);
}

// a1: prefix[b] = pages of requests 0..b-1, computed by every CTA from the
// live seq_lens (the grid itself never depends on them).
template <class F>
__device__ void build_prefix(const ScoreParams &p, int *prefix, SmemCtl<F> *ctl, WorkspaceHeader *hdr)
{
    constexpr int kThreads = Pipe<F>::kThreads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = p.batch;
    const int per = (B + kThreads - 1) / kThreads;
    const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
    // the pass count, loaded beside the lengths (it is needed only if a wait runs out)
    const uint32_t epoch = tid == 0 ? __ldcg(&hdr->epoch) : 0u;
    int local = 0;
    for (int b = r0; b < r1; ++b) {
        const int L = p.seq_lens[b];
        if ((L < 0 || L > p.seq_limit) && blockIdx.x == 0)
            atomicOr(&hdr->fault, MSA_FAULT_SEQ_LEN);
        local += pages_of_request(p, b);
    }
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        ctl->warp_sums[warp] = x;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w)
        before += ctl->warp_sums[w];
    int run = before + x - local;
    for (int b = r0; b < r1; ++b) {
        prefix[b] = run;
        run += pages_of_request(p, b);
    }
    if (tid == kThreads - 1)
        prefix[B] = before + x;
    if (tid == 0)
        ctl->epoch = epoch;
    __syncthreads();
}

// a3 + a4: the block scores of one resident page for every query column.
// The page sits in two 16 KiB halves (dims 0-63, 64-127), each 128 rows of
// 128 bytes with the TMA 128-byte swizzle (16-byte chunk index XOR row % 8).
// A = 16 tokens x 16 dims via ldmatrix; B = q (16 dims x 8 columns per
// fragment; with one position the columns are heads 0-3 and four zero
// columns).  C row = token, column = query column.  vrows[f] = valid token
// rows of this lane's columns in fragment f (positions see different
// lengths).  Returns m[f][0..1] = max over valid rows of columns 8f + 2t and
// 8f + 2t + 1 (t = lane % 4), reduced over the warp.
template <int NQ>
__device__ __forceinline__ void score_page(uint32_t stage,
                                           const uint32_t (&bq)[Cols<NQ>::kFrags][8][2],
                                           const int (&vrows)[Cols<NQ>::kFrags], uint32_t lane_off,
                                           const uint32_t (&xo)[4], int lane,
                                           float (&m)[Cols<NQ>::kFrags][2])
{
    constexpr int NF = Cols<NQ>::kFrags;
    const float neg_inf = -__int_as_float(0x7f800000);
#pragma unroll
    for (int f = 0; f < NF; ++f)
        m[f][0] = m[f][1] = neg_inf;
#pragma unroll
    for (int mt0 = 0; mt0 < 8; mt0 += 4) {
        float acc[4][NF][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int f = 0; f < NF; ++f)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[u][f][e] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint32_t a[4];
                ldsm_x4(a, stage + (ks >> 2) * kHalfPageBytes + (mt0 + u) * 16 * 128 + lane_off +
                               xo[ks & 3]);
#pragma unroll
                for (int f = 0; f < NF; ++f)
                    mma_bf16_16816(acc[u][f], a, bq[f][ks][0], bq[f][ks][1]);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int row = (mt0 + u) * 16 + (lane >> 2);
#pragma unroll
            for (int f = 0; f < NF; ++f) {
                const bool v0 = row < vrows[f], v1 = row + 8 < vrows[f];
                m[f][0] = fmaxf(m[f][0], v0 ? acc[u][f][0] : neg_inf);
                m[f][1] = fmaxf(m[f][1], v0 ? acc[u][f][1] : neg_inf);
                m[f][0] = fmaxf(m[f][0], v1 ? acc[u][f][2] : neg_inf);
                m[f][1] = fmaxf(m[f][1], v1 ? acc[u][f][3] : neg_inf);
            }
        }
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
#pragma unroll
        for (int f = 0; f < NF; ++f) {
            m[f][0] = fmaxf(m[f][0], __shfl_xor_sync(0xffffffffu, m[f][0], o));
            m[f][1] = fmaxf(m[f][1], __shfl_xor_sync(0xffffffffu, m[f][1], o));
        }
    }
}

// Wait for phase `parity` of barrier `bar`, polling at most `limit` times.
__device__ __forceinline__ bool mbar_wait_n(uint32_t bar, uint32_t parity, uint32_t limit)
{
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity))
            return true;
    return false;
}

// A wait of this CTA ran out: the fault bit for the caller, and the pass is
// marked so that the merge empties every output row (its lists are incomplete).
template <class F>
__device__ __forceinline__ void give_up(SmemCtl<F> *ctl, WorkspaceHeader *hdr)
{
    atomicOr(&hdr->fault, MSA_FAULT_TIMEOUT);
    atomicExch(&hdr->aborted, ctl->epoch + 1u);
    ctl->abort_flag = 1;
}

// Bounded wait for the whole warp; false (and the CTA's abort flag set) when
// the wait ran out or another warp already gave up.
template <class F>
__device__ __forceinline__ bool warp_wait(SmemCtl<F> *ctl, WorkspaceHeader *hdr, uint32_t bar,
                                          uint32_t parity, uint32_t limit)
{
    bool ok = false;
    if (!ctl->abort_flag) {
        ok = mbar_wait_n(bar, parity, limit);
        if (!ok)
            give_up(ctl, hdr);
    }
    return __all_sync(0xffffffffu, ok);
}

// a3 + a4 on an fp8 page.  The stage holds 128 rows of 128 E4M3 bytes with
// the TMA 128-byte swizzle (16-byte chunk index XOR row % 8).  Lane (g, t)
// gets bytes 4t..4t+3 of chunk ks of rows g and g+8 of each 16-row tile
// (ldmatrix in its 16-bit view) and converts them exactly to f16 (e4m3 -> f16
// is exact): bytes 4t, 4t+1 fill the A-fragment columns 2t, 2t+1 and bytes
// 4t+2, 4t+3 the columns 2t+8, 2t+9.
// q (bf16) is laid out with the same byte-to-column map, times a per-head
// power of two that keeps it in f16's normal range; f16 mma with fp32
// accumulation.  The per-token scale multiplies each row before the max, the
// per-head power of two is undone after it.
template <int NF>
__device__ __forceinline__ void score_page_fp8(uint32_t stage, const float *scl,
                                               const uint32_t (&bq)[NF][8][2], const int (&vrows)[NF],
                                               int lane, float (&m)[NF][2])
{
    const float neg_inf = -__int_as_float(0x7f800000);
    const int g = lane >> 2;
#pragma unroll
    for (int f = 0; f < NF; ++f)
        m[f][0] = m[f][1] = neg_inf;
#pragma unroll
    for (int mt0 = 0; mt0 < 8; mt0 += 4) {
        float acc[4][NF][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int f = 0; f < NF; ++f)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[u][f][e] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < 8; ks += 2) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                // one ldmatrix.x4 (16-bit view: a lane gets 4 bytes of one row):
                // r0/r1 = rows g / g+8 of chunk ks, r2/r3 = the same of chunk ks+1
                const uint32_t row = static_cast<uint32_t>((mt0 + u) * 16 + ((lane >> 3) & 1) * 8 + (lane & 7));
                const uint32_t chunk = static_cast<uint32_t>(ks + (lane >> 4));
                uint32_t r[4];
                ldsm_x4(r, stage + row * 128 + ((chunk ^ (lane & 7)) << 4));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t a[4];
                    a[0] = e4m3x2_to_f16x2(static_cast<uint16_t>(r[2 * h] & 0xffffu));
                    a[2] = e4m3x2_to_f16x2(static_cast<uint16_t>(r[2 * h] >> 16));
                    a[1] = e4m3x2_to_f16x2(static_cast<uint16_t>(r[2 * h + 1] & 0xffffu));
                    a[3] = e4m3x2_to_f16x2(static_cast<uint16_t>(r[2 * h + 1] >> 16));
#pragma unroll
                    for (int f = 0; f < NF; ++f)
                        mma_f16_16816(acc[u][f], a, bq[f][ks + h][0], bq[f][ks + h][1]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int row = (mt0 + u) * 16 + g;
            const float s0 = scl[row], s1 = scl[row + 8];
#pragma unroll
            for (int f = 0; f < NF; ++f) {
                const bool v0 = row < vrows[f], v1 = row + 8 < vrows[f];
                m[f][0] = fmaxf(m[f][0], v0 ? acc[u][f][0] * s0 : neg_inf);
                m[f][1] = fmaxf(m[f][1], v0 ? acc[u][f][1] * s0 : neg_inf);
                m[f][0] = fmaxf(m[f][0], v1 ? acc[u][f][2] * s1 : neg_inf);
                m[f][1] = fmaxf(m[f][1], v1 ? acc[u][f][3] * s1 : neg_inf);
            }
        }
    }
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            m[f][0] = fmaxf(m[f][0], __shfl_xor_sync(0xffffffffu, m[f][0], o));
            m[f][1] = fmaxf(m[f][1], __shfl_xor_sync(0xffffffffu, m[f][1], o));
        }
}

// The query fragments of request b for the page scorer of format F.
// Column c = 8f + g of fragment f is q row b * kCols + c (position c / 4,
// head c % 4); columns past kCols are zero.
// bf16: the B fragments of m16n8k16.
// fp8: f16 pairs in the byte-to-column map of score_page_fp8, each column
// scaled by 2^e so its largest |q| lands in [2^13, 2^14); inv_lo[f] /
// inv_hi[f] receive 2^-e of columns 8f + 2t and 8f + 2t + 1 (t = lane % 4).
template <class F, int NQ>
__device__ __forceinline__ void load_query(const ScoreParams &p, int b, int lane,
                                           uint32_t (&bq)[Cols<NQ>::kFrags][8][2],
                                           float (&inv_lo)[Cols<NQ>::kFrags],
                                           float (&inv_hi)[Cols<NQ>::kFrags])
{
    constexpr int NC = Cols<NQ>::kCols;
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int f = 0; f < Cols<NQ>::kFrags; ++f) {
        const int c = 8 * f + g;
        const uint16_t *qrow = p.q + (static_cast<size_t>(b) * NC + (c < NC ? c : 0)) * kDim;
        if constexpr (!F::kFp8) {
            const uint32_t *qw = reinterpret_cast<const uint32_t *>(qrow);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                bq[f][ks][0] = c < NC ? __ldg(qw + 8 * ks + t) : 0u;
                bq[f][ks][1] = c < NC ? __ldg(qw + 8 * ks + 4 + t) : 0u;
            }
            inv_lo[f] = inv_hi[f] = 1.0f;
        } else {
            const uint2 *q8 = reinterpret_cast<const uint2 *>(qrow);  // 4 bf16 per load
            float v[8][4];
            float amax = 0.0f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint2 raw = c < NC ? __ldg(q8 + 4 * ks + t) : make_uint2(0u, 0u);
                v[ks][0] = __uint_as_float(raw.x << 16);
                v[ks][1] = __uint_as_float(raw.x & 0xffff0000u);
                v[ks][2] = __uint_as_float(raw.y << 16);
                v[ks][3] = __uint_as_float(raw.y & 0xffff0000u);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    amax = fmaxf(amax, fabsf(v[ks][e]));
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            int ex = 0;
            if (amax > 0.0f)
                frexpf(amax, &ex);              // amax = m * 2^ex, m in [0.5, 1)
            const int sh = max(-100, min(100, 14 - ex));
            const float up = __int_as_float((127 + sh) << 23), down = __int_as_float((127 - sh) << 23);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                bq[f][ks][0] = f32x2_to_f16x2(v[ks][0] * up, v[ks][1] * up);
                bq[f][ks][1] = f32x2_to_f16x2(v[ks][2] * up, v[ks][3] * up);
            }
            inv_lo[f] = __shfl_sync(0xffffffffu, down, (8 * t) & 31);
            inv_hi[f] = __shfl_sync(0xffffffffu, down, (8 * t + 4) & 31);
        }
    }
}

template <int KMAX, class F, int NQ, bool TH>
__device__ void run_consumer(const ScoreParams &p, const Partition &part, uint8_t *smem,
                             SmemCtl<F> *ctl, const int *prefix, WorkspaceHeader *hdr,
                             uint64_t *g_slots)
{
    using P = Pipe<F>;
    using CL = SmemLayout<KMAX, F, NQ>;
    constexpr int C = P::kConsumers;
    constexpr int NC = Cols<NQ>::kCols;    // query columns: NQ positions x 4 heads
    constexpr int NF = Cols<NQ>::kFrags;   // n8 fragments
    constexpr int NR = NC * KMAX / 32;     // list registers per lane
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int t = lane & 3;
    const float neg_inf = -__int_as_float(0x7f800000);
    uint64_t *listbuf = reinterpret_cast<uint64_t *>(smem + CL::lists);

    // ldmatrix lane geometry (bf16): matrix mi = lane / 8 (rows +8 for odd,
    // dims +8 for mi >= 2), row-in-matrix r = lane % 8.
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t lane_off = static_cast<uint32_t>(((mi & 1) * 8 + rr) * 128);
    uint32_t xo[4];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4)
        xo[c4] = static_cast<uint32_t>((((c4 * 2 + (mi >> 1)) ^ rr) & 7) << 4);
    // position of this lane's columns 8f + 2t, 8f + 2t + 1 (clamped for padding columns)
    int lane_pos[NF];
#pragma unroll
    for (int f = 0; f < NF; ++f)
        lane_pos[f] = min((8 * f + 2 * t) >> 2, NQ - 1);

    const uint32_t stage0 = smem_addr(smem + CL::stages);
    const float *scales = reinterpret_cast<const float *>(smem + CL::scales);
    uint32_t bq[NF][8][2];
    float inv_lo[NF], inv_hi[NF];
#pragma unroll
    for (int f = 0; f < NF; ++f)
        inv_lo[f] = inv_hi[f] = 1.0f;
    int q_row = -1;
    uint32_t it = 0;       // pages of this CTA so far (same count as the producer's)
    uint32_t segments = 0; // (chunk, request) segments finished so far

    for (uint32_t n = 0;; ++n) {
        // next chunk id from the producer
        const int qs = static_cast<int>(n % kChunkQueue);
        if (!warp_wait(ctl, hdr, smem_addr(&ctl->cq_full[qs]), (n / kChunkQueue) & 1u, kWaitPolls<TH>))
            break;
        const int c = ctl->chunk_q[qs];
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&ctl->cq_empty[qs]));
        if (c < 0)
            break;
        int p0, p1;
        part.range(c, p0, p1);
        int pg = p0;
        while (pg < p1) {
            const int b = find_row(prefix, p.batch, pg);
            const int row_first = prefix[b], row_end = prefix[b + 1];
            const int seg_end = min(p1, row_end);
            // position i sees the first seq_len - (NQ - 1 - i) tokens
            const int seq_len = p.seq_lens[b];
            int nb_pos[NQ];
#pragma unroll
            for (int i = 0; i < NQ; ++i) {
                const int len = seq_len - (NQ - 1 - i);
                nb_pos[i] = len > 0 ? (len + kPage - 1) / kPage : 0;
            }
            uint64_t lst[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r)
                lst[r] = 0;

            const int skip = (w - static_cast<int>(it % C) + C) % C;
            for (int x = pg + skip; x < seg_end; x += C) {
                const uint32_t my = it + static_cast<uint32_t>(x - pg);
                const int s = P::stage_of(my);
                const int j = x - row_first;

                if (b != q_row) {  // issue the query loads before waiting on the page
                    load_query<F, NQ>(p, b, lane, bq, inv_lo, inv_hi);
                    q_row = b;
                }

                const bool ready =
                    warp_wait(ctl, hdr, smem_addr(&ctl->full[s]), P::use_of(my) & 1u, kWaitPolls<TH>);
                const int2 meta = ctl->meta[s];
                float mk[NF][2];  // the page's column maxima (-inf when skipped)
#pragma unroll
                for (int f = 0; f < NF; ++f)
                    mk[f][0] = mk[f][1] = neg_inf;
                const bool ok = ready && meta.y != 0;
                if (ok) {
                    float m[NF][2];
                    const int rem = seq_len - j * kPage;  // tokens of the last position in this block on
                    int vrows[NF];
#pragma unroll
                    for (int f = 0; f < NF; ++f)
                        vrows[f] = min(kPage, rem - (NQ - 1 - lane_pos[f]));
                    if constexpr (F::kFp8) {
                        score_page_fp8<NF>(stage0 + s * F::kDataBytes, scales + s * kPage, bq, vrows,
                                           lane, m);
#pragma unroll
                        for (int f = 0; f < NF; ++f) {
                            m[f][0] *= inv_lo[f];
                            m[f][1] *= inv_hi[f];
                        }
                    } else {
                        score_page<NQ>(stage0 + s * F::kDataBytes, bq, vrows, lane_off, xo, lane, m);
                    }
#pragma unroll
                    for (int f = 0; f < NF; ++f) {
                        mk[f][0] = m[f][0];
                        mk[f][1] = m[f][1];
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&ctl->empty[s]));

                // Column cc's maximum is held by lanes with t = (cc % 8) / 2, as
                // mk[cc / 8][cc % 2].  Every column on every lane is needed only
                // for 32-wide lists or the block-score output.
                if (KMAX == 32 || p.out_block_scores != nullptr) {
                    float sc[NC];
#pragma unroll
                    for (int cc = 0; cc < NC; ++cc)
                        sc[cc] = __shfl_sync(0xffffffffu, mk[cc >> 3][cc & 1], (cc & 7) >> 1);
                    if (p.out_block_scores != nullptr && lane < NC) {
                        float v = sc[0];
#pragma unroll
                        for (int cc = 1; cc < NC; ++cc)
                            v = lane == cc ? sc[cc] : v;
                        p.out_block_scores[(static_cast<size_t>(b) * NC + lane) * p.bt_stride + j] = v;
                    }
                    if constexpr (KMAX == 32) {
#pragma unroll
                        for (int r = 0; r < NR; ++r) {
                            const int nbp = nb_pos[r >> 2];
                            const bool pinned = j < p.n_sink || j >= nbp - p.n_window;
                            const uint64_t key = (ok && j < nbp) ? pack_key(sc[r], j, pinned) : 0ull;
                            lst[r] = insert_desc<32>(lst[r], key, lane);
                        }
                    }
                }
                if constexpr (KMAX == 16) {
                    // list register r: lanes 0-15 hold column 2r, lanes 16-31 column
                    // 2r + 1.  Lane (lane & 16) | (r & 3) holds both as mk[r / 4][h]
                    // with h its own half, so one shuffle gives each half its column.
                    const int h = lane >> 4;
#pragma unroll
                    for (int r = 0; r < NR; ++r) {
                        const float v =
                            __shfl_sync(0xffffffffu, h ? mk[r >> 2][1] : mk[r >> 2][0], (lane & 16) | (r & 3));
                        const int nbp = nb_pos[r >> 1];  // position of columns 2r, 2r + 1
                        const bool pinned = j < p.n_sink || j >= nbp - p.n_window;
                        const uint64_t key = (ok && j < nbp) ? pack_key(v, j, pinned) : 0ull;
                        lst[r] = insert_desc<16>(lst[r], key, lane);
                    }
                }
            }
            it += static_cast<uint32_t>(seg_end - pg);
            pg = seg_end;

            // a6: combine the consumer warps' lists of this (chunk, request)
            // and store the result in slot c + b.  Double-buffered: buffer
            // `buf` is written again two segments later, after every warp has
            // passed the next segment's barrier (and so has finished reading
            // this one).
            const int buf = static_cast<int>(segments & 1u);
            uint64_t *lb = listbuf + static_cast<size_t>(buf) * C * NC * KMAX;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const int col = r * (32 / KMAX) + lane / KMAX;
                lb[(w * NC + col) * KMAX + lane % KMAX] = lst[r];
            }
            mbar_arrive(smem_addr(&ctl->list_bar[buf]));  // every consumer thread
            const bool lists_ready =
                warp_wait(ctl, hdr, smem_addr(&ctl->list_bar[buf]), (segments >> 1) & 1u,
                          kWaitPolls<TH>);
            ++segments;
            if (!lists_ready)
                continue;
            const int slot = c + b;
            if (slot >= p.slot_capacity) {
                if (lane == 0)
                    atomicOr(&hdr->fault, MSA_FAULT_SLOTS);
                continue;
            }
            auto L = [&](int src, int col, int rank) { return lb[(src * NC + col) * KMAX + rank]; };
            auto store = [&](int col, int rank, uint64_t v) {
                g_slots[(static_cast<size_t>(slot) * NC + col) * KMAX + rank] = v;
            };
            constexpr int kPerWarp = NC / C;  // columns each warp merges
            if constexpr (C == 2 && KMAX == 16) {
                // two columns per pass: lanes 0-15 and 16-31
#pragma unroll
                for (int pp = 0; pp < kPerWarp / 2; ++pp) {
                    const int col = w * kPerWarp + 2 * pp + (lane >> 4), r = lane & 15;
                    store(col, r, merge_top<16>(L(0, col, r), L(1, col, 15 - r), lane));
                }
            } else if constexpr (C == 2) {
#pragma unroll
                for (int pp = 0; pp < kPerWarp; ++pp) {
                    const int col = w * kPerWarp + pp;
                    store(col, lane, merge_top<32>(L(0, col, lane), L(1, col, 31 - lane), lane));
                }
            } else if constexpr (C == 4 && KMAX == 16) {
                // per column: lanes 0-15 merge lists 0,1, lanes 16-31 lists 2,3, then the halves
#pragma unroll
                for (int pp = 0; pp < kPerWarp; ++pp) {
                    const int col = w * kPerWarp + pp;
                    const int half = lane >> 4, r = lane & 15;
                    uint64_t v = merge_top<16>(L(2 * half, col, r), L(2 * half + 1, col, 15 - r), lane);
                    v = merge_top<16>(v, __shfl_sync(0xffffffffu, v, 31 - lane), lane);
                    if (lane < 16)
                        store(col, r, v);
                }
            } else {
                static_assert(C == 4, "two or four consumer warps");
#pragma unroll
                for (int pp = 0; pp < kPerWarp; ++pp) {
                    const int col = w * kPerWarp + pp;
                    uint64_t v = merge_top<32>(L(0, col, lane), L(1, col, 31 - lane), lane);
                    const uint64_t u = merge_top<32>(L(2, col, lane), L(3, col, 31 - lane), lane);
                    v = merge_top<32>(v, __shfl_sync(0xffffffffu, u, 31 - lane), lane);
                    store(col, lane, v);
                }
            }
        }
    }
}

// Lane-parallel lookup of up to 32 pages [pb, pe) of the batch: lane i gets
// page pb + i's physical page, valid-token count and a validity bit.
struct PageLookup {
    int page, valid, ok;
};

__device__ __forceinline__ PageLookup lookup_pages(const ScoreParams &p, const int *prefix,
                                                   WorkspaceHeader *hdr, int pb, int pe, int lane)
{
    PageLookup r{0, 0, 0};
    const int pg = pb + lane;
    if (pg < pe) {
        const int b = find_row(prefix, p.batch, pg);
        const int j = pg - prefix[b];
        r.page = p.block_table[static_cast<int64_t>(b) * p.bt_stride + j];
        r.valid = min(kPage, p.seq_lens[b] - j * kPage);
        r.ok = (r.page >= 0 && r.page < p.num_pages) ? 1 : 0;
        if (!r.ok)
            atomicOr(&hdr->fault, MSA_FAULT_PAGE_ID);
    }
    return r;
}

// A pool ticket (valid in lane 0).
__device__ __forceinline__ unsigned take_ticket(WorkspaceHeader *hdr, int lane)
{
    return lane == 0 ? atomicAdd(&hdr->pool_next, 1u) : 0u;
}

// The chunk behind a ticket; tickets past the batch are skipped.  -1: none left.
__device__ __forceinline__ int resolve_ticket(const Partition &part, WorkspaceHeader *hdr,
                                              unsigned ticket, int lane)
{
    if (part.pool == 0)
        return -1;
    int c = part.pool_chunk(static_cast<int>(__shfl_sync(0xffffffffu, ticket, 0)));
    while (c == -2)
        c = part.pool_chunk(static_cast<int>(__shfl_sync(0xffffffffu, take_ticket(hdr, lane), 0)));
    return c;
}

template <int KMAX, class F, int NQ, bool TH>
__device__ void run_producer(const ScoreParams &p, const Partition &part, uint8_t *smem,
                             SmemCtl<F> *ctl, const int *prefix, WorkspaceHeader *hdr)
{
    using P = Pipe<F>;
    const int lane = threadIdx.x & 31;
    const uint32_t stage0 = smem_addr(smem + SmemLayout<KMAX, F, NQ>::stages);
    const uint32_t scale0 = smem_addr(smem + SmemLayout<KMAX, F, NQ>::scales);
    uint32_t it = 0;  // pages issued
    uint32_t n = 0;   // chunk ids posted
    // K is read once per pass: evicted first, unless the whole pass fits in
    // half of L2, where repeated calls on the same pages can find them there
    const uint64_t stream_policy =
        part.total <= p.l2_keep_pages ? l2_evict_normal_policy() : l2_evict_first_policy();

    auto post = [&](int c) {
        if (lane == 0) {
            const int qs = static_cast<int>(n % kChunkQueue);
            if (n >= kChunkQueue && !ctl->abort_flag &&
                !mbar_wait_n(smem_addr(&ctl->cq_empty[qs]), ((n / kChunkQueue) - 1) & 1u,
                             kWaitPolls<TH>))
                give_up(ctl, hdr);
            ctl->chunk_q[qs] = c;
            mbar_arrive(smem_addr(&ctl->cq_full[qs]));
        }
        ++n;
        __syncwarp();
    };

    // This CTA's static chunk first, then pool chunks.  A batch of up to 32
    // pages is always issued before anything that waits on global memory
    // (the next batch's lookups, a pool ticket): the pages already in the
    // stage ring keep the consumers and HBM busy across those waits.
    int cur = part.first_chunk(blockIdx.x);
    if (cur < 0 && part.pool > 0)
        cur = resolve_ticket(part, hdr, take_ticket(hdr, lane), lane);
    int a = 0, e = 0;
    PageLookup look{0, 0, 0};
    if (cur >= 0) {
        post(cur);  // consumers can start their query loads at once
        part.range(cur, a, e);
        look = lookup_pages(p, prefix, hdr, a, e, lane);
    }
    while (cur >= 0) {
        const int cnt = min(32, e - a);
        for (int i = 0; i < cnt; ++i, ++it) {
            const int page = __shfl_sync(0xffffffffu, look.page, i);
            const int valid = __shfl_sync(0xffffffffu, look.valid, i);
            const int ok = __shfl_sync(0xffffffffu, look.ok, i);
            if (lane == 0) {
                const int s = P::stage_of(it);
                const uint32_t full = smem_addr(&ctl->full[s]);
                if (it >= P::kStages && !ctl->abort_flag) {
                    if (!mbar_wait_n(smem_addr(&ctl->empty[s]), (P::use_of(it) - 1) & 1u,
                                     kWaitPolls<TH>))
                        give_up(ctl, hdr);
                }
                // with the test hook set nothing is loaded or signalled until a
                // wait has run out: every stage stays empty, no copy is in flight
                const bool withheld = TH && !ctl->abort_flag;
                const bool issue = ok && !ctl->abort_flag && !withheld;
                ctl->meta[s] = make_int2(valid, issue ? 1 : 0);
                if (issue) {
                    const uint32_t dst = stage0 + s * F::kDataBytes;
                    mbar_arrive_expect_tx(full, P::kTxBytes);
                    if constexpr (F::kFp8) {
                        tma_load_2d_hint(dst, &p.tmap, 0, page * kPage, full, stream_policy);
                        bulk_load_hint(scale0 + s * F::kScaleBytes,
                                       p.kscale + static_cast<size_t>(page) * kPage, F::kScaleBytes,
                                       full, stream_policy);
                    } else {
                        tma_load_2d_hint(dst, &p.tmap, 0, page * kPage, full, stream_policy);
                        tma_load_2d_hint(dst + kHalfPageBytes, &p.tmap, 64, page * kPage, full,
                                         stream_policy);
                    }
                } else if (!withheld) {
                    mbar_arrive(full);
                }
            }
            __syncwarp();
        }
        if (a + 32 < e) {  // next batch of the same chunk
            a += 32;
            look = lookup_pages(p, prefix, hdr, a, e, lane);
            continue;
        }
        cur = part.pool > 0 ? resolve_ticket(part, hdr, take_ticket(hdr, lane), lane) : -1;
        if (cur < 0)
            break;
        post(cur);
        part.range(cur, a, e);
        look = lookup_pages(p, prefix, hdr, a, e, lane);
    }
    post(-1);  // no more chunks

    // This CTA takes no more tickets; the last CTA to get here resets the
    // ticket counters for the next pass (every other CTA has stopped claiming)
    // and counts the pass: every CTA read the pass count at its start, before
    // its own arrival here.
    if (lane == 0) {
        __threadfence();
        if (atomicAdd(&hdr->done, 1u) == gridDim.x - 1) {
            atomicExch(&hdr->pool_next, 0u);
            atomicExch(&hdr->done, 0u);
            atomicAdd(&hdr->epoch, 1u);
        }
    }
    // Drain: no copy may still be landing in shared memory when the CTA exits.
    // (With the test hook no copy was ever issued.)
    if (lane == 0 && !TH) {
        const uint32_t cnt = it < P::kStages ? it : P::kStages;
        for (uint32_t i = 0; i < cnt; ++i) {
            const uint32_t q = it - 1 - i;
            if (!mbar_wait_n(smem_addr(&ctl->full[P::stage_of(q)]), P::use_of(q) & 1u,
                             kWaitPolls<TH>))
                give_up(ctl, hdr);
        }
    }
}

template <int KMAX, class F, int NQ, bool TH = false>
__global__ void __launch_bounds__(Pipe<F>::kThreads, 1)
    score_kernel(const __grid_constant__ ScoreParams p)
{
    using P = Pipe<F>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    SmemCtl<F> *ctl = reinterpret_cast<SmemCtl<F> *>(smem + SmemLayout<KMAX, F, NQ>::ctl);
    int *prefix = reinterpret_cast<int *>(smem + SmemLayout<KMAX, F, NQ>::prefix);
    WorkspaceHeader *hdr = reinterpret_cast<WorkspaceHeader *>(p.ws);
    uint64_t *g_slots = reinterpret_cast<uint64_t *>(p.ws + slots_offset(p.batch));
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P::kStages; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), 1);
            mbar_init(smem_addr(&ctl->empty[s]), 1);
        }
        for (int i = 0; i < kChunkQueue; ++i) {
            mbar_init(smem_addr(&ctl->cq_full[i]), 1);
            mbar_init(smem_addr(&ctl->cq_empty[i]), P::kConsumers);
        }
        for (int i = 0; i < 2; ++i)
            mbar_init(smem_addr(&ctl->list_bar[i]), P::kConsumerThreads);
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == P::kProducerWarp && (threadIdx.x & 31) == 0)
        prefetch_tensormap(&p.tmap);
    // Everything above touched only this CTA's shared memory and the kernel
    // parameters; global memory is read and written only after the previous
    // kernel on the stream has finished.  The merge grid is released only
    // after this wait: a decode call's merge reads the call's lengths before
    // its own wait, which is safe because whatever wrote them has finished
    // by now.
    griddep_wait();
    griddep_launch_dependents();

    build_prefix<F>(p, prefix, ctl, hdr);  // ends with __syncthreads

    if (threadIdx.x == 0)
        ctl->part = Partition::make(prefix[p.batch], gridDim.x, p.split_blocks);
    __syncthreads();
    const Partition &part = ctl->part;
    if (blockIdx.x == 0) {
        int *g_prefix = reinterpret_cast<int *>(p.ws + prefix_offset());
        for (int b = threadIdx.x; b <= p.batch; b += P::kThreads)
            g_prefix[b] = prefix[b];
        if (threadIdx.x == 0) {
            hdr->part = part;
            hdr->batch = p.batch;
            hdr->kmax = KMAX;
        }
    }

    if (warp == P::kProducerWarp)
        run_producer<KMAX, F, NQ, TH>(p, part, smem, ctl, prefix, hdr);
    else
        run_consumer<KMAX, F, NQ, TH>(p, part, smem, ctl, prefix, hdr, g_slots);
}

// Selected blocks -> small KV pages for one (request, head) row, by one full
// warp: the <= 32 selected ids (`id` of lane < k, else -1) are sorted
// ascending across the lanes (bitonic), each lane counts the small pages of
// its block, a lane prefix gives the output offsets, and each lane copies
// its pages' ids from the KV block table.
struct ExpandArgs {
    const int32_t *seq_lens;
    const int32_t *kv_bt;
    int64_t kv_stride;
    int per_block;
    int page_tokens;
    int32_t *out_pages;  // null: no expansion
    int32_t *out_num;
};

__device__ __forceinline__ void expand_row(const ExpandArgs &ex, int b, size_t row, int k, int id,
                                           int lane)
{
    const int L = ex.seq_lens[b];
    const int nb = L > 0 ? (L + kPage - 1) / kPage : 0;
    long long small = L > 0 ? (static_cast<long long>(L) + ex.page_tokens - 1) / ex.page_tokens : 0;
    if (small > ex.kv_stride)
        small = ex.kv_stride;
    int key = (id >= 0 && id < nb) ? id : 0x7fffffff;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int j = size >> 1; j > 0; j >>= 1) {
            const int other = __shfl_xor_sync(0xffffffffu, key, j);
            const bool ascending = (lane & size) == 0;
            const bool low = (lane & j) == 0;
            key = (low == ascending) ? min(key, other) : max(key, other);
        }
    }
    const bool valid = key != 0x7fffffff;
    const long long first = valid ? static_cast<long long>(key) * ex.per_block : 0;
    int count = 0;
    if (valid && first < small)
        count = static_cast<int>(min(static_cast<long long>(ex.per_block), small - first));
    int incl = count;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    const int width = k * ex.per_block;
    int32_t *out = ex.out_pages + row * width;
    const int32_t *src = ex.kv_bt + static_cast<size_t>(b) * ex.kv_stride;
    for (int s = 0; s < count; ++s)
        out[incl - count + s] = src[first + s];
    for (int e = total + lane; e < width; e += 32)
        out[e] = -1;
    if (lane == 0)
        ex.out_num[row] = total;
}

// a7: one CTA per (query column, request): column = 4 * position + head.  The
// request's chunk lists are staged in shared memory a tile at a time (all of a
// thread's loads in flight together); each group of KMAX lanes merges its
// (up to 8) lists of the tile pairwise and folds the result into a running
// top-KMAX, and a tree over the groups, whose first level (the two groups of
// a warp, at KMAX 16) is a shuffle, yields the request's top-KMAX.
constexpr int kMergeThreads = 256;
constexpr int kMergeTileKeys = 2048;  // 16 KiB of keys staged per pass

// What a decode call tells its merge beyond the workspace: with the lengths
// (batch <= kMergeThreads) each merge CTA finds its request's page range and
// the pass's chunking itself, before the score grid has finished, instead of
// reading them from the workspace after it.  Null seq_lens: the workspace.
struct MergeHint {
    const int32_t *seq_lens;
    int seq_limit;
    int grid;          // the score grid
    int split_blocks;
};

template <int KMAX>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const uint8_t *ws, int batch, int k,
                                                              int cols, int slot_capacity,
                                                              int32_t *out_ids, float *out_scores,
                                                              const ExpandArgs ex, const MergeHint hint)
{
    constexpr int kGroups = kMergeThreads / KMAX;
    constexpr int kTileLists = kMergeTileKeys / KMAX;
    __shared__ uint64_t tile[kMergeTileKeys];
    __shared__ uint64_t tree[kMergeThreads];
    __shared__ int sums[2][kMergeThreads / 32];

    const int h = blockIdx.x, b = blockIdx.y;
    const int lane = threadIdx.x & 31, grp = threadIdx.x / KMAX, rank = threadIdx.x % KMAX;
    const WorkspaceHeader *hdr = reinterpret_cast<const WorkspaceHeader *>(ws);
    const uint64_t *slots = reinterpret_cast<const uint64_t *>(ws + slots_offset(batch));

    int c_first = 0, n_lists = 0;
    if (hint.seq_lens != nullptr) {
        // The lengths are inputs of the call: whatever wrote them finished
        // before the score grid got past its own wait, and only then was this
        // grid released.  Pages before this request and in the whole batch,
        // as the score kernel counts them.
        int pg = 0;
        if (threadIdx.x < batch)
            pg = pages_for_length(hint.seq_lens[threadIdx.x], hint.seq_limit);
        const int mine = __shfl_sync(0xffffffffu, pg, b & 31);  // valid in the warp holding b
        int before = threadIdx.x < b ? pg : 0, all = pg;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            before += __shfl_xor_sync(0xffffffffu, before, o);
            all += __shfl_xor_sync(0xffffffffu, all, o);
        }
        if (lane == 0) {
            sums[0][threadIdx.x >> 5] = before;
            sums[1][threadIdx.x >> 5] = all;
        }
        if ((threadIdx.x >> 5) == (b >> 5) && lane == 0)
            tree[0] = static_cast<uint64_t>(mine);
        __syncthreads();
        int p0 = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kMergeThreads / 32; ++w) {
            p0 += sums[0][w];
            total += sums[1][w];
        }
        const int p1 = p0 + static_cast<int>(tree[0]);
        __syncthreads();
        const Partition part = Partition::make(total, hint.grid, hint.split_blocks);
        if (p1 > p0 && part.unit > 0 && p1 <= part.total) {
            c_first = part.chunk_of(p0);
            n_lists = min(part.chunk_of(p1 - 1) - c_first + 1, slot_capacity);
        }
    }
    // the score grid's workspace writes are complete and visible after this
    griddep_wait();
    griddep_launch_dependents();

    // a wait of the score pass ran out: its lists are incomplete, every row is left empty
    const bool pass_ok = hdr->aborted != hdr->epoch;
    if (hint.seq_lens == nullptr) {
        const int *prefix = reinterpret_cast<const int *>(ws + prefix_offset());
        const Partition &part = hdr->part;
        const int p0 = prefix[b], p1 = prefix[b + 1];
        if (pass_ok && p1 > p0 && part.unit > 0 && p1 <= part.total) {
            c_first = part.chunk_of(p0);
            n_lists = min(part.chunk_of(p1 - 1) - c_first + 1, slot_capacity);
        }
    }

    constexpr int kPer = kMergeTileKeys / kMergeThreads;  // keys a thread stages per tile
    constexpr int kLevels = 3;                              // lists per group per tile: <= 2^kLevels
    static_assert(kTileLists == kGroups << kLevels, "a tile holds 8 lists per group");
    auto rev = [&](uint64_t x) { return __shfl_sync(0xffffffffu, x, lane ^ (KMAX - 1)); };
    uint64_t run = 0;
    for (int t0 = 0; t0 < n_lists; t0 += kTileLists) {
        const int nt = min(kTileLists, n_lists - t0);
        // all of a thread's loads in flight at once, then the stores
        uint64_t v[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = threadIdx.x + i * kMergeThreads;
            const int slot = c_first + t0 + e / KMAX + b;
            v[i] = (e < nt * KMAX && slot < slot_capacity)
                       ? slots[(static_cast<size_t>(slot) * cols + h) * KMAX + e % KMAX]
                       : 0ull;
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            tile[threadIdx.x + i * kMergeThreads] = v[i];
        __syncthreads();
        // group grp's lists grp + kGroups m (m < 8), merged pairwise: each level's
        // merges are independent of one another, so their latencies overlap
        // (folding them into one running list one by one does not)
        const int per = (nt + kGroups - 1) / kGroups;  // lists per group, uniform over the CTA
        auto list = [&](int m, bool reversed) {
            const int li = grp + kGroups * m;
            return li < nt ? tile[li * KMAX + (reversed ? KMAX - 1 - rank : rank)] : 0ull;
        };
        uint64_t a0 = list(0, false);
        if (per > 1) {
            uint64_t a2 = 0, a4 = 0, a6 = 0;
            a0 = merge_top<KMAX>(a0, list(1, true), lane);
            if (per > 2) {
                a2 = merge_top<KMAX>(list(2, false), list(3, true), lane);
                if (per > 4) {
                    a4 = merge_top<KMAX>(list(4, false), list(5, true), lane);
                    a6 = merge_top<KMAX>(list(6, false), list(7, true), lane);
                    a4 = merge_top<KMAX>(a4, rev(a6), lane);
                }
                a0 = merge_top<KMAX>(a0, rev(a2), lane);
                if (per > 4)
                    a0 = merge_top<KMAX>(a0, rev(a4), lane);
            }
        }
        run = t0 == 0 ? a0 : merge_top<KMAX>(run, rev(a0), lane);
        __syncthreads();
    }
    const int used = min(n_lists, kGroups);  // groups holding anything
    int first_step = 1;
    if constexpr (KMAX == 16) {
        // the two groups of a warp: each half merges the other's list, read
        // reversed straight from its lanes
        if (used > 1)
            run = merge_top<KMAX>(run, __shfl_sync(0xffffffffu, run, lane ^ 31), lane);
        first_step = 2;
    }
    tree[threadIdx.x] = run;
    __syncthreads();
#pragma unroll
    for (int step = first_step; step < kGroups; step <<= 1) {
        if (step >= used)
            break;  // uniform across the CTA
        const bool active = (grp % (2 * step)) == 0 && grp + step < kGroups;
        const uint64_t other = active ? tree[(grp + step) * KMAX + (KMAX - 1 - rank)] : 0ull;
        run = merge_top<KMAX>(run, other, lane);
        __syncthreads();
        tree[threadIdx.x] = run;
        __syncthreads();
    }
    if (!pass_ok)
        run = 0;  // the empty key
    int id = -1;
    if (grp == 0 && rank < k) {
        float score;
        unpack_key(run, id, score);
        const size_t o = (static_cast<size_t>(b) * cols + h) * k + rank;
        out_ids[o] = id;
        out_scores[o] = score;
    }
    // fused page expansion (decode, one position): warp 0 holds the list
    if (ex.out_pages != nullptr && threadIdx.x < 32)
        expand_row(ex, b, static_cast<size_t>(b) * cols + h, k, id, lane);
}

// Selected blocks -> small KV pages, one warp per (request, head).
__global__ void __launch_bounds__(128) expand_pages_kernel(const int32_t *ids, int k, const ExpandArgs ex)
{
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.x, h = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t row = static_cast<size_t>(b) * kHeads + h;
    expand_row(ex, b, row, k, lane < k ? ids[row * k + lane] : -1, lane);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <int KMAX, class F, int NQ, bool TH = false>
static bool ensure_smem_attr(int dev)
{
    static std::atomic<bool> done[kMaxDevices];
    if (dev >= 0 && dev < kMaxDevices && done[dev].load(std::memory_order_acquire))
        return true;
    const size_t bytes = SmemLayout<KMAX, F, NQ>::bytes(MSA_MAX_BATCH);
    if (cudaFuncSetAttribute(score_kernel<KMAX, F, NQ, TH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(bytes)) != cudaSuccess)
        return false;
    if (dev >= 0 && dev < kMaxDevices)
        done[dev].store(true, std::memory_order_release);
    return true;
}

static bool bounds_ok(int max_batch, int max_model_len, int k, int split_blocks)
{
    if (max_batch < 1 || max_batch > MSA_MAX_BATCH || max_model_len < 1)
        return false;
    if (k < 1 || k > MSA_MAX_TOPK || split_blocks < 0)
        return false;
    return static_cast<int64_t>(max_batch) * blocks_for(max_model_len) < (int64_t{1} << 30);
}

static int64_t chunk_bound(int batch, int64_t max_blocks, int split_blocks, int grid)
{
    return chunk_capacity(grid, static_cast<int64_t>(batch) * max_blocks, split_blocks);
}

static msa_status validate(const void *q, const void *kcache_pool, int64_t num_pages,
                           const int32_t *block_table, int64_t bt_stride, const int32_t *seq_lens,
                           int batch, int max_batch, int max_model_len, int k, int n_sink,
                           int n_window, const void *workspace, int split_blocks)
{
    if (!q || !kcache_pool || !block_table || !seq_lens || !workspace)
        return MSA_ERR_INVALID_ARG;
    if (batch < 0 || batch > max_batch || max_batch < 1 || max_model_len < 1)
        return MSA_ERR_INVALID_ARG;
    if (max_batch > MSA_MAX_BATCH)
        return MSA_ERR_UNSUPPORTED;
    if (k < 1 || n_sink < 0 || n_window < 0 || split_blocks < 0)
        return MSA_ERR_INVALID_ARG;
    if (k > MSA_MAX_TOPK)
        return MSA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(n_sink) + n_window > k)
        return MSA_ERR_INVALID_ARG;
    if (num_pages < 1 || bt_stride < 1)
        return MSA_ERR_INVALID_ARG;
    if (num_pages > (int64_t{1} << 24))  // TMA row coordinate page*128 must fit in int32
        return MSA_ERR_UNSUPPORTED;
    if (!bounds_ok(max_batch, max_model_len, k, split_blocks))
        return MSA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(kcache_pool) & 15) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3) || (reinterpret_cast<uintptr_t>(seq_lens) & 3))
        return MSA_ERR_INVALID_ARG;
    return MSA_OK;
}

// The longest request the block table and max_model_len allow.
static int seq_limit_for(int64_t bt_stride, int max_model_len)
{
    return static_cast<int>(bt_stride * kPage < max_model_len ? bt_stride * kPage : max_model_len);
}

static int score_grid(int sms, int batch, int64_t max_blocks, int split_blocks)
{
    const int64_t work = static_cast<int64_t>(batch) * max_blocks;
    int64_t units = split_blocks > 0 ? (work + split_blocks - 1) / split_blocks : work;
    int64_t g = sms;
    if (g > MSA_MAX_GRID)
        g = MSA_MAX_GRID;
    if (units < g)
        g = units;
    return static_cast<int>(g < 1 ? 1 : g);
}

// Test hook for the bounded waits (msa_indexer_test_withhold_pages): while it
// is set, bf16 one-position passes with k <= 16 run score_kernel<16, Bf16Fmt,
// 1, true> (no page loaded, short waits) and bf16 prefill passes the pair
// kernel's copy that loads nothing; other shapes are refused.
static std::atomic<int> g_withhold_pages{0};

bool test_withhold_pages() { return g_withhold_pages.load(std::memory_order_relaxed) != 0; }

// The pool as a 2-D tensor map: rows = num_pages * 128 tokens, 128 elements
// per row, 128-byte swizzle.  bf16: 64x128 boxes (two per page); fp8
// (unsigned bytes): one 128x128 box per page.
template <class F>
static bool make_pool_map(CUtensorMap *map, const void *pool, int64_t num_pages)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc)
        return false;
    const cuuint64_t elem = F::kFp8 ? 1 : 2;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDim),
                                static_cast<cuuint64_t>(num_pages) * kPage};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDim) * elem};
    const cuuint32_t box[2] = {F::kFp8 ? 128u : 64u, static_cast<cuuint32_t>(kPage)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, F::kFp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KMAX, class F, int NQ>
static msa_status launch_score(const void *q, const void *kcache_pool, const float *kscale,
                               int64_t num_pages, const int32_t *block_table, int64_t bt_stride,
                               const int32_t *seq_lens, int batch, int max_model_len, int n_sink,
                               int n_window, float *out_block_scores, void *workspace,
                               int slot_capacity, int grid, int split_blocks, cudaStream_t st,
                               int dev)
{
    ScoreParams p;
    std::memset(&p, 0, sizeof p);
    const bool withhold = g_withhold_pages.load(std::memory_order_relaxed) != 0;
    if (withhold && !(KMAX == 16 && NQ == 1 && std::is_same<F, Bf16Fmt>::value))
        return MSA_ERR_UNSUPPORTED;
    if (!make_pool_map<F>(&p.tmap, kcache_pool, num_pages))
        return MSA_ERR_CUDA;
    p.q = static_cast<const uint16_t *>(q);
    p.kscale = kscale;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.out_block_scores = out_block_scores;
    p.ws = static_cast<uint8_t *>(workspace);
    p.bt_stride = bt_stride;
    p.num_pages = num_pages;
    p.batch = batch;
    p.seq_limit = seq_limit_for(bt_stride, max_model_len);
    p.n_sink = n_sink;
    p.n_window = n_window;
    p.split_blocks = split_blocks;
    p.slot_capacity = slot_capacity;
    p.l2_keep_pages = static_cast<int>(device_l2_bytes(dev) / 2 / (F::kDataBytes + F::kScaleBytes));
    const size_t smem = SmemLayout<KMAX, F, NQ>::bytes(batch);
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(Pipe<F>::kThreads), smem, st, attr);
    if constexpr (KMAX == 16 && NQ == 1 && std::is_same<F, Bf16Fmt>::value) {
        if (withhold) {
            if (!ensure_smem_attr<16, Bf16Fmt, 1, true>(dev))
                return MSA_ERR_CUDA;
            return cudaLaunchKernelEx(&cfg, score_kernel<16, Bf16Fmt, 1, true>, p) == cudaSuccess
                       ? MSA_OK
                       : MSA_ERR_CUDA;
        }
    }
    if (!ensure_smem_attr<KMAX, F, NQ>(dev))
        return MSA_ERR_CUDA;
    return cudaLaunchKernelEx(&cfg, score_kernel<KMAX, F, NQ>, p) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

struct Plan {
    int grid;
    int slot_capacity;
    int dev;
};

static msa_status plan(int batch, int max_batch, int max_model_len, int k, int split_blocks,
                       size_t workspace_bytes, Plan &out, int nq = 1)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MSA_ERR_CUDA;
    const int sms = device_sms(dev);
    if (sms <= 0)
        return MSA_ERR_CUDA;
    const int64_t max_blocks = blocks_for(max_model_len);
    const int grid = score_grid(sms, batch, max_blocks, split_blocks);
    const int kmax = kmax_for(k);
    const size_t off = slots_offset(batch);
    const int64_t need_slots = chunk_bound(batch, max_blocks, split_blocks, grid) + batch;
    if (workspace_bytes < off)
        return MSA_ERR_WORKSPACE_TOO_SMALL;
    const int64_t cap = static_cast<int64_t>((workspace_bytes - off) / (slot_bytes(kmax) * nq));
    if (cap < need_slots)
        return MSA_ERR_WORKSPACE_TOO_SMALL;
    out.grid = grid;
    out.slot_capacity = static_cast<int>(cap > (int64_t{1} << 30) ? (int64_t{1} << 30) : cap);
    out.dev = dev;
    (void)max_batch;
    return MSA_OK;
}

// A one-position bf16 pass whose bound is one to 64 pages per SM runs the
// four-consumer format (Bf16Wide4Fmt).  Fewer pages than SMs leave most
// CTAs one page or none, where the wider CTA only costs.
constexpr int64_t kWideMaxPagesPerSm = 64;
static bool wide_pass(int batch, int max_model_len, int dev)
{
    const int64_t work = static_cast<int64_t>(batch) * blocks_for(max_model_len);
    const int sms = device_sms(dev);
    return !g_withhold_pages.load(std::memory_order_relaxed) && sms > 0 && work >= sms &&
           work <= kWideMaxPagesPerSm * sms;
}

template <class F, int NQ = 1>
static msa_status score_entry(const void *q, const void *kcache_pool, const float *kscale,
                              int64_t num_pages, const int32_t *block_table, int64_t bt_stride,
                              const int32_t *seq_lens, int batch, int max_batch, int max_model_len,
                              int k, int n_sink, int n_window, float *out_block_scores,
                              void *workspace, size_t workspace_bytes, int split_blocks,
                              void *stream)
{
    msa_status st = validate(q, kcache_pool, num_pages, block_table, bt_stride, seq_lens, batch,
                             max_batch, max_model_len, k, n_sink, n_window, workspace, split_blocks);
    if (st != MSA_OK)
        return st;
    if (F::kFp8 && (!kscale || (reinterpret_cast<uintptr_t>(kscale) & 15)))
        return MSA_ERR_INVALID_ARG;
    if (batch == 0)
        return MSA_OK;
    Plan pl;
    st = plan(batch, max_batch, max_model_len, k, split_blocks, workspace_bytes, pl, NQ);
    if (st != MSA_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if constexpr (std::is_same<F, Bf16Fmt>::value && NQ == 1) {
        if (wide_pass(batch, max_model_len, pl.dev)) {
            if (kmax_for(k) == 16)
                return launch_score<16, Bf16Wide4Fmt, 1>(q, kcache_pool, kscale, num_pages, block_table,
                                                         bt_stride, seq_lens, batch, max_model_len, n_sink,
                                                         n_window, out_block_scores, workspace,
                                                         pl.slot_capacity, pl.grid, split_blocks, s, pl.dev);
            return launch_score<32, Bf16Wide4Fmt, 1>(q, kcache_pool, kscale, num_pages, block_table,
                                                     bt_stride, seq_lens, batch, max_model_len, n_sink,
                                                     n_window, out_block_scores, workspace,
                                                     pl.slot_capacity, pl.grid, split_blocks, s, pl.dev);
        }
    }
    if (kmax_for(k) == 16)
        return launch_score<16, F, NQ>(q, kcache_pool, kscale, num_pages, block_table, bt_stride,
                                       seq_lens, batch, max_model_len, n_sink, n_window,
                                       out_block_scores, workspace, pl.slot_capacity, pl.grid,
                                       split_blocks, s, pl.dev);
    return launch_score<32, F, NQ>(q, kcache_pool, kscale, num_pages, block_table, bt_stride,
                                   seq_lens, batch, max_model_len, n_sink, n_window,
                                   out_block_scores, workspace, pl.slot_capacity, pl.grid,
                                   split_blocks, s, pl.dev);
}

}  // namespace msa

using namespace msa;

extern "C" size_t msa_indexer_workspace_bytes_mq(int max_batch, int max_model_len, int k,
                                                 int split_blocks, int q_len)
{
    if (!bounds_ok(max_batch, max_model_len, k, split_blocks))
        return 0;
    if (q_len != 1 && q_len != 2 && q_len != 4)
        return 0;
    const int64_t chunks = chunk_bound(max_batch, blocks_for(max_model_len), split_blocks, MSA_MAX_GRID);
    return slots_offset(max_batch) +
           static_cast<size_t>(chunks + max_batch) * slot_bytes(kmax_for(k)) * q_len;
}

extern "C" size_t msa_indexer_workspace_bytes(int max_batch, int max_model_len, int k,
                                              int split_blocks)
{
    return msa_indexer_workspace_bytes_mq(max_batch, max_model_len, k, split_blocks, 1);
}


extern "C" msa_status msa_indexer_score(const void *q, const void *kcache_pool, int64_t num_pages,
                                        const int32_t *block_table, int64_t bt_stride,
                                        const int32_t *seq_lens, int batch, int max_batch,
                                        int max_model_len, int k, int n_sink, int n_window,
                                        float *out_block_scores, void *workspace,
                                        size_t workspace_bytes, int split_blocks, void *stream)
{
    return score_entry<Bf16Fmt>(q, kcache_pool, nullptr, num_pages, block_table, bt_stride,
                                seq_lens, batch, max_batch, max_model_len, k, n_sink, n_window,
                                out_block_scores, workspace, workspace_bytes, split_blocks, stream);
}

extern "C" msa_status msa_indexer_score_fp8(const void *q, const void *kcache_fp8,
                                            const float *kscale, int64_t num_pages,
                                            const int32_t *block_table, int64_t bt_stride,
                                            const int32_t *seq_lens, int batch, int max_batch,
                                            int max_model_len, int k, int n_sink, int n_window,
                                            float *out_block_scores, void *workspace,
                                            size_t workspace_bytes, int split_blocks, void *stream)
{
    return score_entry<Fp8Fmt>(q, kcache_fp8, kscale, num_pages, block_table, bt_stride, seq_lens,
                               batch, max_batch, max_model_len, k, n_sink, n_window,
                               out_block_scores, workspace, workspace_bytes, split_blocks, stream);
}

static msa_status merge_entry(int batch, int k, int cols, int32_t *out_ids, float *out_scores,
                              const void *workspace, size_t workspace_bytes, void *stream,
                              const ExpandArgs &ex = ExpandArgs{}, MergeHint hint = MergeHint{})
{
    if (batch > kMergeThreads)
        hint.seq_lens = nullptr;
    if (!out_ids || !out_scores || !workspace || batch < 0 || batch > MSA_MAX_BATCH)
        return MSA_ERR_INVALID_ARG;
    if (k < 1)
        return MSA_ERR_INVALID_ARG;
    if (k > MSA_MAX_TOPK)
        return MSA_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(workspace) & 255)
        return MSA_ERR_INVALID_ARG;
    if (batch == 0)
        return MSA_OK;
    const int kmax = kmax_for(k);
    const size_t off = slots_offset(batch);
    const size_t per_slot = slot_bytes(kmax) / kHeads * cols;
    if (workspace_bytes < off + per_slot)
        return MSA_ERR_WORKSPACE_TOO_SMALL;
    const int64_t cap = static_cast<int64_t>((workspace_bytes - off) / per_slot);
    const int capacity = static_cast<int>(cap > (int64_t{1} << 30) ? (int64_t{1} << 30) : cap);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint8_t *ws = static_cast<const uint8_t *>(workspace);
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>(cols), static_cast<unsigned>(batch)),
                                        dim3(kMergeThreads), 0, s, attr);
    cudaError_t e = kmax == 16
                        ? cudaLaunchKernelEx(&cfg, merge_kernel<16>, ws, batch, k, cols, capacity,
                                             out_ids, out_scores, ex, hint)
                        : cudaLaunchKernelEx(&cfg, merge_kernel<32>, ws, batch, k, cols, capacity,
                                             out_ids, out_scores, ex, hint);
    return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

// The hint a decode call passes its merge: the lengths, their limit and the
// score grid and split its score pass was launched with (as plan() sizes it).
static MergeHint merge_hint(const int32_t *seq_lens, int batch, int64_t bt_stride, int max_model_len,
                            int split_blocks)
{
    MergeHint h{nullptr, 0, 0, 0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return h;
    const int sms = device_sms(dev);
    if (sms <= 0)
        return h;
    h.seq_lens = seq_lens;
    h.seq_limit = seq_limit_for(bt_stride, max_model_len);
    h.grid = score_grid(sms, batch, blocks_for(max_model_len), split_blocks);
    h.split_blocks = split_blocks;
    return h;
}

extern "C" msa_status msa_indexer_merge(int batch, int k, int32_t *out_ids, float *out_scores,
                                        const void *workspace, size_t workspace_bytes,
                                        void *stream)
{
    return merge_entry(batch, k, kHeads, out_ids, out_scores, workspace, workspace_bytes, stream);
}

extern "C" msa_status msa_indexer_decode(const void *q, const void *kcache_pool, int64_t num_pages,
                                         const int32_t *block_table, int64_t bt_stride,
                                         const int32_t *seq_lens, int batch, int max_batch,
                                         int max_model_len, int k, int n_sink, int n_window,
                                         int32_t *out_ids, float *out_scores,
                                         float *out_block_scores, void *workspace,
                                         size_t workspace_bytes, int split_blocks, void *stream)
{
    if (!out_ids || !out_scores)
        return MSA_ERR_INVALID_ARG;
    msa_status st = msa_indexer_score(q, kcache_pool, num_pages, block_table, bt_stride, seq_lens,
                                      batch, max_batch, max_model_len, k, n_sink, n_window,
                                      out_block_scores, workspace, workspace_bytes, split_blocks,
                                      stream);
    if (st != MSA_OK || batch == 0)
        return st;
    return merge_entry(batch, k, kHeads, out_ids, out_scores, workspace, workspace_bytes, stream,
                       ExpandArgs{}, merge_hint(seq_lens, batch, bt_stride, max_model_len, split_blocks));
}

// ---------------------------------------------------------------------------
// Allocation-free variant: the scratch of msa_indexer_decode in a fixed
// device array of this library, for callers that cannot allocate.
// ---------------------------------------------------------------------------

namespace msa {

static __device__ __align__(256) uint8_t g_noalloc_workspace[MSA_NOALLOC_WORKSPACE_BYTES];

// Device address of g_noalloc_workspace in the current context.  In host code
// the array's name only stands in for it; the kernels must be given this
// address.  It is looked up on every call (a host-side query that allocates
// nothing and enqueues nothing): each context that loads the library (the
// primary one, a framework's own, a new one after cudaDeviceReset) holds its
// own copy of the array at its own address.  Each copy is zero-filled when
// the module is loaded into its context, which is what the words that must
// start at zero (the header's ticket counters) need; the score kernel
// returns them to zero at the end of every pass.
static void *noalloc_workspace()
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess)
        return nullptr;
    return p;
}

}  // namespace msa

extern "C" msa_status msa_indexer_decode_noalloc(const void *q, const void *kcache_pool,
                                                 int64_t num_pages, const int32_t *block_table,
                                                 int64_t bt_stride, const int32_t *seq_lens,
                                                 int batch, int max_model_len, int k, int n_sink,
                                                 int n_window, int32_t *out_ids, float *out_scores,
                                                 float *out_block_scores, void *stream)
{
    if (!out_ids || !out_scores)
        return MSA_ERR_INVALID_ARG;
    const int max_batch = batch > 0 ? batch : 1;
    // argument checks that need no device (a placeholder stands in for the scratch)
    msa_status st = validate(q, kcache_pool, num_pages, block_table, bt_stride, seq_lens, batch,
                             max_batch, max_model_len, k, n_sink, n_window,
                             reinterpret_cast<const void *>(uintptr_t{256}), 0);
    if (st != MSA_OK || batch == 0)
        return st;
    // the same sizing msa_indexer_decode applies to a caller's workspace
    Plan pl;
    st = plan(batch, max_batch, max_model_len, k, 0, MSA_NOALLOC_WORKSPACE_BYTES, pl);
    if (st == MSA_ERR_WORKSPACE_TOO_SMALL)
        return MSA_ERR_UNSUPPORTED;
    if (st != MSA_OK)
        return st;
    void *ws = noalloc_workspace();
    if (ws == nullptr)
        return MSA_ERR_CUDA;
    return msa_indexer_decode(q, kcache_pool, num_pages, block_table, bt_stride, seq_lens, batch,
                              max_batch, max_model_len, k, n_sink, n_window, out_ids, out_scores,
                              out_block_scores, ws, MSA_NOALLOC_WORKSPACE_BYTES, 0, stream);
}

extern "C" msa_status msa_indexer_expand_pages(const int32_t *ids, int batch, int k,
                                               const int32_t *seq_lens,
                                               const int32_t *kv_block_table,
                                               int64_t kv_bt_stride, int page_tokens,
                                               int32_t *out_pages, int32_t *out_num_pages,
                                               void *stream)
{
    if (!ids || !seq_lens || !kv_block_table || !out_pages || !out_num_pages)
        return MSA_ERR_INVALID_ARG;
    if (batch < 0 || k < 1 || kv_bt_stride < 1 || page_tokens < 1 || kPage % page_tokens != 0)
        return MSA_ERR_INVALID_ARG;
    if (k > MSA_MAX_TOPK || batch > MSA_MAX_BATCH)
        return MSA_ERR_UNSUPPORTED;
    if (batch == 0)
        return MSA_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>(batch)), dim3(32 * kHeads), 0, s, attr);
    ExpandArgs ex{seq_lens, kv_block_table, kv_bt_stride, kPage / page_tokens, page_tokens, out_pages,
                  out_num_pages};
    const cudaError_t e = cudaLaunchKernelEx(&cfg, expand_pages_kernel, ids, k, ex);
    return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

extern "C" msa_status msa_indexer_decode_pages(
    const void *q, const void *kcache_pool, int64_t num_pages, const int32_t *block_table,
    int64_t bt_stride, const int32_t *seq_lens, int batch, int max_batch, int max_model_len, int k,
    int n_sink, int n_window, int32_t *out_ids, float *out_scores, float *out_block_scores,
    void *workspace, size_t workspace_bytes, int split_blocks, const int32_t *kv_block_table,
    int64_t kv_bt_stride, int page_tokens, int32_t *out_pages, int32_t *out_num_pages, void *stream)
{
    if (!out_ids || !out_scores || !kv_block_table || !out_pages || !out_num_pages)
        return MSA_ERR_INVALID_ARG;
    if (kv_bt_stride < 1 || page_tokens < 1 || kPage % page_tokens != 0)
        return MSA_ERR_INVALID_ARG;
    msa_status st = msa_indexer_score(q, kcache_pool, num_pages, block_table, bt_stride, seq_lens,
                                      batch, max_batch, max_model_len, k, n_sink, n_window,
                                      out_block_scores, workspace, workspace_bytes, split_blocks,
                                      stream);
    if (st != MSA_OK || batch == 0)
        return st;
    const ExpandArgs ex{seq_lens, kv_block_table, kv_bt_stride, kPage / page_tokens, page_tokens,
                        out_pages, out_num_pages};
    return merge_entry(batch, k, kHeads, out_ids, out_scores, workspace, workspace_bytes, stream, ex,
                       merge_hint(seq_lens, batch, bt_stride, max_model_len, split_blocks));
}

extern "C" msa_status msa_indexer_decode_mq(const void *q, int q_len, const void *kcache_pool,
                                            int64_t num_pages, const int32_t *block_table,
                                            int64_t bt_stride, const int32_t *seq_lens, int batch,
                                            int max_batch, int max_model_len, int k, int n_sink,
                                            int n_window, int32_t *out_ids, float *out_scores,
                                            float *out_block_scores, void *workspace,
                                            size_t workspace_bytes, int split_blocks, void *stream)
{
    if (!out_ids || !out_scores)
        return MSA_ERR_INVALID_ARG;
    if (q_len < 1)
        return MSA_ERR_INVALID_ARG;
    if (q_len != 1 && q_len != 2 && q_len != 4)
        return MSA_ERR_UNSUPPORTED;
    msa_status st;
    if (q_len == 1)
        st = score_entry<Bf16Fmt, 1>(q, kcache_pool, nullptr, num_pages, block_table, bt_stride,
                                     seq_lens, batch, max_batch, max_model_len, k, n_sink, n_window,
                                     out_block_scores, workspace, workspace_bytes, split_blocks,
                                     stream);
    else if (q_len == 2)
        st = score_entry<Bf16Fmt, 2>(q, kcache_pool, nullptr, num_pages, block_table, bt_stride,
                                     seq_lens, batch, max_batch, max_model_len, k, n_sink, n_window,
                                     out_block_scores, workspace, workspace_bytes, split_blocks,
                                     stream);
    else
        st = score_entry<Bf16Wide4Fmt, 4>(q, kcache_pool, nullptr, num_pages, block_table, bt_stride,
                                     seq_lens, batch, max_batch, max_model_len, k, n_sink, n_window,
                                     out_block_scores, workspace, workspace_bytes, split_blocks,
                                     stream);
    if (st != MSA_OK || batch == 0)
        return st;
    return merge_entry(batch, k, kHeads * q_len, out_ids, out_scores, workspace, workspace_bytes,
                       stream, ExpandArgs{},
                       merge_hint(seq_lens, batch, bt_stride, max_model_len, split_blocks));
}

extern "C" msa_status msa_indexer_decode_mq_fp8(const void *q, int q_len, const void *kcache_fp8,
                                                const float *kscale, int64_t num_pages,
                                                const int32_t *block_table, int64_t bt_stride,
                                                const int32_t *seq_lens, int batch, int max_batch,
                                                int max_model_len, int k, int n_sink, int n_window,
                                                int32_t *out_ids, float *out_scores,
                                                float *out_block_scores, void *workspace,
                                                size_t workspace_bytes, int split_blocks,
                                                void *stream)
{
    if (!out_ids || !out_scores)
        return MSA_ERR_INVALID_ARG;
    if (q_len < 1)
        return MSA_ERR_INVALID_ARG;
    if (q_len != 1 && q_len != 2 && q_len != 4)
        return MSA_ERR_UNSUPPORTED;
    msa_status st;
    if (q_len == 1)
        st = score_entry<Fp8Fmt, 1>(q, kcache_fp8, kscale, num_pages, block_table, bt_stride,
                                    seq_lens, batch, max_batch, max_model_len, k, n_sink, n_window,
                                    out_block_scores, workspace, workspace_bytes, split_blocks,
                                    stream);
    else if (q_len == 2)
        st = score_entry<Fp8MqFmt, 2>(q, kcache_fp8, kscale, num_pages, block_table, bt_stride,
                                      seq_lens, batch, max_batch, max_model_len, k, n_sink,
                                      n_window, out_block_scores, workspace, workspace_bytes,
                                      split_blocks, stream);
    else
        st = score_entry<Fp8MqFmt, 4>(q, kcache_fp8, kscale, num_pages, block_table, bt_stride,
                                      seq_lens, batch, max_batch, max_model_len, k, n_sink,
                                      n_window, out_block_scores, workspace, workspace_bytes,
                                      split_blocks, stream);
    if (st != MSA_OK || batch == 0)
        return st;
    return merge_entry(batch, k, kHeads * q_len, out_ids, out_scores, workspace, workspace_bytes,
                       stream, ExpandArgs{},
                       merge_hint(seq_lens, batch, bt_stride, max_model_len, split_blocks));
}

extern "C" msa_status msa_indexer_decode_fp8(const void *q, const void *kcache_fp8,
                                             const float *kscale, int64_t num_pages,
                                             const int32_t *block_table, int64_t bt_stride,
                                             const int32_t *seq_lens, int batch, int max_batch,
                                             int max_model_len, int k, int n_sink, int n_window,
                                             int32_t *out_ids, float *out_scores,
                                             float *out_block_scores, void *workspace,
                                             size_t workspace_bytes, int split_blocks,
                                             void *stream)
{
    if (!out_ids || !out_scores)
        return MSA_ERR_INVALID_ARG;
    msa_status st = msa_indexer_score_fp8(q, kcache_fp8, kscale, num_pages, block_table, bt_stride,
                                          seq_lens, batch, max_batch, max_model_len, k, n_sink,
                                          n_window, out_block_scores, workspace, workspace_bytes,
                                          split_blocks, stream);
    if (st != MSA_OK || batch == 0)
        return st;
    return merge_entry(batch, k, kHeads, out_ids, out_scores, workspace, workspace_bytes, stream,
                       ExpandArgs{}, merge_hint(seq_lens, batch, bt_stride, max_model_len, split_blocks));
}

extern "C" void msa_indexer_test_withhold_pages(int on)
{
    g_withhold_pages.store(on != 0 ? 1 : 0, std::memory_order_relaxed);
}

extern "C" msa_status msa_indexer_get_error(void *workspace, void *stream, uint32_t *flags)
{
    if (!workspace || !flags)
        return MSA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t *word = &static_cast<WorkspaceHeader *>(workspace)->fault;
    uint32_t host = 0;
    if (cudaMemcpyAsync(&host, word, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MSA_ERR_CUDA;
    if (cudaMemsetAsync(word, 0, sizeof host, s) != cudaSuccess)
        return MSA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess)
        return MSA_ERR_CUDA;
    *flags = host;
    return MSA_OK;
}

extern "C" const char *msa_status_string(int status)
{
    switch (status) {
    case MSA_OK:
        return "ok";
    case MSA_ERR_INVALID_ARG:
        return "invalid argument";
    case MSA_ERR_UNSUPPORTED:
        return "unsupported size";
    case MSA_ERR_WORKSPACE_TOO_SMALL:
        return "workspace too small";
    case MSA_ERR_CUDA:
        return "CUDA error";
    default:
        return "unknown status";
    }
}
