// Prefill scoring: every new token of a request scores the blocks of its own
// causal prefix (vLLM PR #57832: the prefill branch scores iq[nd:] over the
// block table with cu_seqlens_q, then takes the per-token top-k).  New token t
// of request b (n_b new tokens, seq_len_b tokens in all) sits at position
// seq_len_b - n_b + t and sees tokens [0, position].
//
// prefill_score_kernel: one CTA per tile of 32 new tokens of one request
// (128 rows = 32 tokens x 4 heads).  A producer warp streams the request's
// pages (those the tile's last token sees) through a 3-stage TMA ring; each
// of 8 consumer warps holds its 16 rows of q as mma.sync A fragments and
// multiplies them with every resident page (keys as the n dimension via
// ldmatrix), takes the masked max over the page's visible keys per row and
// writes the block score.  Every consumer reads every stage, so the empty
// barriers count 8 arrivals and each consumer sees the phases in order.
//
// rows_topk_kernel: one warp per (token, head) row: pins and top-k over the
// row's block scores (bitonic sort of 32 keys at a time into a running list).
#pragma once

namespace msa {

constexpr int kPfTokens = 32;                    // new tokens per tile
constexpr int kPfConsumers = 8;                  // 4 tokens x 4 heads = 16 rows each
constexpr int kPfStages = 3;
constexpr int kPfThreads = 32 * (kPfConsumers + 1);

struct PrefillParams {
    CUtensorMap tmap;  // bf16 pool, 64x128 boxes, 128B swizzle
    const uint16_t *q;         // [total_q, 4, 128]
    const int32_t *cu_q;       // [batch + 1]
    const int32_t *block_table;
    const int32_t *seq_lens;
    float *scores;             // [total_q, 4, bs_stride]
    uint32_t *fault;
    int64_t bt_stride;
    int64_t bs_stride;
    int64_t num_pages;
    int batch;
    int seq_limit;
    int total_q;
};

struct PrefillSmem {
    uint64_t full[kPfStages];
    uint64_t empty[kPfStages];
    int ok[kPfStages];
    int b, tile, n_new, seq_len, tok0, nb_tile;
};

constexpr size_t kPfSmemBytes = 1024 /* alignment slack */ + kPfStages * kPageBytes + sizeof(PrefillSmem);

// New tokens of request b, or -1 for a request the kernel refuses: rows
// outside [0, total_q) or out of order, a length past the limit or negative,
// or more new tokens than tokens.
__device__ __forceinline__ int pf_new_tokens(const PrefillParams &p, int b, int *seq_out)
{
    const int c0 = p.cu_q[b], c1 = p.cu_q[b + 1];
    const int n = c1 - c0;
    const int L = p.seq_lens[b];
    *seq_out = L;
    if (c0 < 0 || c1 > p.total_q || n < 0 || L < 0 || L > p.seq_limit || n > L)
        return -1;
    return n;
}

__global__ void __launch_bounds__(kPfThreads, 2) prefill_score_kernel(const __grid_constant__ PrefillParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    PrefillSmem *ctl = reinterpret_cast<PrefillSmem *>(smem + kPfStages * kPageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPfStages; ++s) {
            mbar_init(smem_addr(&ctl->full[s]), 1);
            mbar_init(smem_addr(&ctl->empty[s]), kPfConsumers);
        }
        fence_barrier_init();
    }
    griddep_wait();
    griddep_launch_dependents();

    // which (request, tile) this CTA scores: a serial scan by one thread
    // (batch sizes of a prefill step are small)
    if (threadIdx.x == 0) {
        int before = 0, found = -1;
        for (int b = 0; b < p.batch; ++b) {
            int L;
            const int n = pf_new_tokens(p, b, &L);
            if (n < 0) {
                atomicOr(p.fault, MSA_FAULT_SEQ_LEN);
                continue;
            }
            const int tiles = (n + kPfTokens - 1) / kPfTokens;
            if (found < 0 && static_cast<int>(blockIdx.x) < before + tiles) {
                found = b;
                ctl->b = b;
                ctl->tile = blockIdx.x - before;
                ctl->n_new = n;
                ctl->seq_len = L;
            }
            before += tiles;
        }
        if (found < 0) {
            ctl->b = -1;
        } else {
            ctl->tok0 = ctl->tile * kPfTokens;
            const int last = min(ctl->n_new, ctl->tok0 + kPfTokens) - 1;  // last token of the tile
            const int pos_last = ctl->seq_len - ctl->n_new + last;
            ctl->nb_tile = pos_last / kPage + 1;
        }
    }
    __syncthreads();
    if (ctl->b < 0)
        return;  // past the last tile (uniform across the CTA)
    const int b = ctl->b, n_new = ctl->n_new, seq_len = ctl->seq_len, tok0 = ctl->tok0;
    const int nb_tile = ctl->nb_tile;
    const uint32_t stage0 = smem_addr(smem);

    if (warp == kPfConsumers) {
        // producer
        const uint64_t pol = l2_evict_first_policy();
        for (int jb = 0; jb < nb_tile; jb += 32) {
            const int j_l = jb + lane;
            int page = 0, ok = 0;
            if (j_l < nb_tile) {
                page = p.block_table[static_cast<int64_t>(b) * p.bt_stride + j_l];
                ok = (page >= 0 && page < p.num_pages) ? 1 : 0;
                if (!ok)
                    atomicOr(p.fault, MSA_FAULT_PAGE_ID);
            }
            const int cnt = min(32, nb_tile - jb);
            for (int i = 0; i < cnt; ++i) {
                const int j = jb + i;
                const int pg = __shfl_sync(0xffffffffu, page, i);
                const int pok = __shfl_sync(0xffffffffu, ok, i);
                if (lane == 0) {
                    const int s = j % kPfStages;
                    const uint32_t full = smem_addr(&ctl->full[s]);
                    if (j >= kPfStages &&
                        !mbar_wait(smem_addr(&ctl->empty[s]), ((j / kPfStages) - 1) & 1u))
                        atomicOr(p.fault, MSA_FAULT_TIMEOUT);
                    ctl->ok[s] = pok;
                    if (pok) {
                        const uint32_t dst = stage0 + s * kPageBytes;
                        mbar_arrive_expect_tx(full, kPageBytes);
                        tma_load_2d_hint(dst, &p.tmap, 0, pg * kPage, full, pol);
                        tma_load_2d_hint(dst + kHalfPageBytes, &p.tmap, 64, pg * kPage, full, pol);
                    } else {
                        mbar_arrive(full);
                    }
                }
                __syncwarp();
            }
        }
        if (lane == 0) {  // drain: no copy may land after the CTA exits
            for (int j = max(0, nb_tile - kPfStages); j < nb_tile; ++j)
                if (!mbar_wait(smem_addr(&ctl->full[j % kPfStages]), (j / kPfStages) & 1u))
                    atomicOr(p.fault, MSA_FAULT_TIMEOUT);
        }
        return;
    }

    // consumer warp: rows 4*tl + h for its 4 tokens tl (C rows g and g+8)
    const int g = lane >> 2, t = lane & 3;
    const int tl0 = tok0 + 4 * warp + (g >> 2);  // token (within the request's new tokens) of row g
    const int tl1 = tl0 + 2;                     // token of row g + 8
    const int head = g & 3;
    const int pos0 = seq_len - n_new + tl0, pos1 = seq_len - n_new + tl1;
    const bool live0 = tl0 < n_new, live1 = tl1 < n_new;
    const int warp_first = tok0 + 4 * warp;
    const int warp_last = min(n_new, warp_first + 4) - 1;
    const int wpos_min = seq_len - n_new + warp_first;
    const int wpos_max = seq_len - n_new + warp_last;
    const bool warp_live = warp_first < n_new;

    // A fragments of the warp's 16 rows (zero for tokens past the request's new tokens)
    uint32_t a[8][4];
    {
        const int64_t r0 = static_cast<int64_t>(p.cu_q[b]) + tl0, r1 = static_cast<int64_t>(p.cu_q[b]) + tl1;
        const uint32_t *q0 = reinterpret_cast<const uint32_t *>(p.q + (r0 * kHeads + head) * kDim);
        const uint32_t *q1 = reinterpret_cast<const uint32_t *>(p.q + (r1 * kHeads + head) * kDim);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            a[ks][0] = live0 ? __ldg(q0 + 8 * ks + t) : 0u;
            a[ks][1] = live1 ? __ldg(q1 + 8 * ks + t) : 0u;
            a[ks][2] = live0 ? __ldg(q0 + 8 * ks + 4 + t) : 0u;
            a[ks][3] = live1 ? __ldg(q1 + 8 * ks + 4 + t) : 0u;
        }
    }
    // ldmatrix geometry for B (keys x dims): matrix mi = lane / 8: keys +8 for
    // mi >= 2, dims +8 for odd mi; key-in-matrix r = lane % 8
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t key_off = static_cast<uint32_t>(((mi >> 1) * 8 + rr) * 128);
    uint32_t xo[4];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4)
        xo[c4] = static_cast<uint32_t>((((c4 * 2 + (mi & 1)) ^ rr) & 7) << 4);
    const float neg_inf = -__int_as_float(0x7f800000);
    float *out0 = p.scores + ((static_cast<int64_t>(p.cu_q[b]) + tl0) * kHeads + head) * p.bs_stride;
    float *out1 = p.scores + ((static_cast<int64_t>(p.cu_q[b]) + tl1) * kHeads + head) * p.bs_stride;

    for (int j = 0; j < nb_tile; ++j) {
        const int s = j % kPfStages;
        bool ready = false;
        if (mbar_wait(smem_addr(&ctl->full[s]), (j / kPfStages) & 1u))
            ready = true;
        else if (lane == 0)
            atomicOr(p.fault, MSA_FAULT_TIMEOUT);
        ready = __all_sync(0xffffffffu, ready);
        const bool page_ok = ready && ctl->ok[s] != 0;
        const int first_key = j * kPage;
        // a page past every row of this warp is skipped (still waited and released)
        if (page_ok && warp_live && first_key <= wpos_max) {
            const uint32_t stage = stage0 + s * kPageBytes;
            const bool full_page = first_key + kPage - 1 <= wpos_min;
            float mx0 = neg_inf, mx1 = neg_inf;
#pragma unroll 2
            for (int nf2 = 0; nf2 < 8; ++nf2) {
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t bf[4];
                    ldsm_x4(bf, stage + (ks >> 2) * kHalfPageBytes + nf2 * 16 * 128 + key_off + xo[ks & 3]);
                    mma_bf16_16816(acc[0], a[ks], bf[0], bf[1]);
                    mma_bf16_16816(acc[1], a[ks], bf[2], bf[3]);
                }
#pragma unroll
                for (int fr = 0; fr < 2; ++fr) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int kp = first_key + nf2 * 16 + fr * 8 + 2 * t + e;
                        const bool v0 = full_page || kp <= pos0;
                        const bool v1 = full_page || kp <= pos1;
                        mx0 = fmaxf(mx0, v0 ? acc[fr][e] : neg_inf);
                        mx1 = fmaxf(mx1, v1 ? acc[fr][2 + e] : neg_inf);
                    }
                }
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            if (t == 0) {
                if (live0 && first_key <= pos0)
                    out0[j] = mx0;
                if (live1 && first_key <= pos1)
                    out1[j] = mx1;
            }
        } else if (!page_ok && ready && warp_live && t == 0) {
            if (live0 && first_key <= pos0)
                out0[j] = neg_inf;
            if (live1 && first_key <= pos1)
                out1[j] = neg_inf;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_addr(&ctl->empty[s]));
    }
}

// Sorts 32 keys (one per lane) into descending order across the warp.
__device__ __forceinline__ uint64_t sort32_desc(uint64_t v, int lane)
{
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int j = size >> 1; j > 0; j >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool desc = (lane & size) == 0;  // always true at size 32
            const bool low = (lane & j) == 0;
            v = (low == desc) ? umax64(v, o) : umin64(v, o);
        }
    }
    return v;
}

// One warp per (token, head) row of the prefill: pins and top-k of its blocks.
template <int KMAX>
__global__ void __launch_bounds__(256) rows_topk_kernel(const float *scores, int64_t bs_stride,
                                                        const int32_t *cu_q, const int32_t *seq_lens,
                                                        int batch, int total_q, int seq_limit, int k,
                                                        int n_sink, int n_window, int32_t *out_ids,
                                                        float *out_scores)
{
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);  // (token, head)
    if (row >= static_cast<int64_t>(total_q) * kHeads)
        return;
    const int tok = static_cast<int>(row / kHeads);
    // the request of this token: the last b with cu_q[b] <= tok
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu_q[mid] <= tok)
            lo = mid;
        else
            hi = mid - 1;
    }
    const int b = lo;
    const int n = cu_q[b + 1] - cu_q[b], L = seq_lens[b];
    int nb = 0;
    if (cu_q[b] >= 0 && cu_q[b] <= tok && tok < cu_q[b + 1] && cu_q[b + 1] <= total_q && L >= 0 &&
        L <= seq_limit && n <= L) {
        const int pos = L - n + (tok - cu_q[b]);
        nb = pos / kPage + 1;
    }
    const float *srow = scores + row * bs_stride;
    uint64_t run = 0;
    for (int c0 = 0; c0 < nb; c0 += 32) {
        const int j = c0 + lane;
        uint64_t key = 0;
        if (j < nb)
            key = pack_key(srow[j], j, j < n_sink || j >= nb - n_window);
        if (j < nb && srow[j] == -__int_as_float(0x7f800000))
            key = 0;  // a block whose page was out of range
        const uint64_t sorted = sort32_desc(key, lane);
        if constexpr (KMAX == 16)
            run = merge_top<16>(run, __shfl_sync(0xffffffffu, sorted, (15 - lane) & 31), lane);
        else
            run = merge_top<32>(run, __shfl_sync(0xffffffffu, sorted, 31 - lane), lane);
    }
    if (lane < k) {
        int id;
        float score;
        unpack_key(run, id, score);
        out_ids[row * k + lane] = id;
        out_scores[row * k + lane] = score;
    }
}

}  // namespace msa
