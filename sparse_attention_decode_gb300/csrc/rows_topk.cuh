// Per-row top-k of the prefill's block scores (the second prefill kernel).
//
// One warp per (token, head) row: the row's blocks are its token's visible
// blocks; pins (the first n_sink and the last n_window of them) come first,
// then the highest-scoring free blocks (vLLM PR #57832, "Solution" step 3:
// packed (score, block id) keys; the prefill branch takes a per-token top-k
// over cu_seqlens_q).  Included by prefill.cu after its request helpers.
#pragma once

namespace msa {

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

constexpr int kKeysPerLane = 16;  // rows_topk_kernel takes 32 x 16 = 512 blocks at a time

// Rows (one warp each) per CTA of rows_topk_kernel<KMAX>: 16 KiB of
// candidate space per CTA either way.
template <int KMAX>
__host__ __device__ constexpr int rows_per_cta() { return KMAX == 16 ? 8 : 4; }

// Sorts 32 values (one per lane) into descending order across the warp.
__device__ __forceinline__ uint32_t sort32_desc_u32(uint32_t v, int lane)
{
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int j = size >> 1; j > 0; j >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool desc = (lane & size) == 0;
            const bool low = (lane & j) == 0;
            v = (low == desc) ? max(v, o) : min(v, o);
        }
    }
    return v;
}

// The 32-bit coarse key of a packed key: all pinned blocks share the top
// value, free blocks keep the order bits of their score, empty is 0.  It
// never decreases along the packed-key order (equal scores tie).
__device__ __forceinline__ uint32_t coarse_of(uint64_t key)
{
    if (key == 0)
        return 0;
    return (key >> 63) ? 0xFFFFFFFFu : static_cast<uint32_t>(key >> 31);
}

// Merges 32 keys (one per lane, any order) into the running top-KMAX list.
template <int KMAX>
__device__ __forceinline__ uint64_t merge32(uint64_t run, uint64_t key, int lane)
{
    const uint64_t sorted = sort32_desc(key, lane);
    if constexpr (KMAX == 16)
        return merge_top<16>(run, __shfl_sync(0xffffffffu, sorted, (15 - lane) & 31), lane);
    else
        return merge_top<32>(run, __shfl_sync(0xffffffffu, sorted, 31 - lane), lane);
}

// One warp per (token, head) row of the prefill: pins and top-k of its
// blocks.  The pins enter the running list first; then the blocks go 512 (16
// per lane) at a time through a filter on 32-bit coarse keys (the order bits
// of the score): until the running list is full, the KMAX-th largest of the
// 32 lane maxima is a lower bound on the coarse key of the group's KMAX-th
// largest block (KMAX lanes hold one at least that large, and a pin ranks
// above its coarse key); once it is full, its last key is the bound.  Only
// blocks at or above the bound can enter the list.  They are compacted into shared memory (without ties at most KMAX
// lanes x 16; a group whose ties overflow that is merged whole instead),
// pins and out-of-range blocks dropped, and inserted one at a time when there
// are few, else sorted 32 at a time and merged.  The list ends as the
// descending top-KMAX of all keys.
template <int KMAX>
__global__ void __launch_bounds__(32 * rows_per_cta<KMAX>()) rows_topk_kernel(
    const float *scores, int64_t bs_stride, const int32_t *cu_q, const int32_t *seq_lens, int batch,
    int total_q, int seq_limit, int k, int n_sink, int n_window, int32_t *out_ids, float *out_scores)
{
    constexpr int kRowsPerCta = rows_per_cta<KMAX>();
    constexpr int kCandCap = KMAX * kKeysPerLane;
    __shared__ float cand_s[kRowsPerCta][kCandCap];  // candidate scores
    __shared__ int cand_j[kRowsPerCta][kCandCap];    // and their block ids
    // No early trigger: this grid runs in many waves, and a dependent persistent
    // scoring grid launched before its last wave slows that wave (its CTAs are
    // released at this grid's exit instead).
    griddep_wait();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + wid;  // (token, head)
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
    const Req r = req_info(cu_q, seq_lens, total_q, seq_limit, lo);
    int nb = 0;
    if (r.ok && r.c0 <= tok && tok < r.c0 + r.n)
        nb = (r.len - r.n + (tok - r.c0)) / kPage + 1;
    const float *srow = scores + row * bs_stride;
    const float neg_inf = -__int_as_float(0x7f800000);
    float *buf_s = cand_s[wid];
    int *buf_j = cand_j[wid];
    // The pins (the first n_sink and the last n_window visible blocks, ids
    // ascending) go into the list first: their ids are known, and a block
    // whose page was out of range (-inf) is left out.
    const int ns = min(n_sink, nb);
    const int w0 = max(ns, nb - n_window);  // first window block that is not a sink
    const int npin = ns + (nb - w0);        // <= n_sink + n_window <= k <= KMAX
    uint64_t pk = 0;
    if (lane < npin) {
        const int id = lane < ns ? lane : w0 + (lane - ns);
        const float sv = srow[id];
        pk = sv == neg_inf ? 0ull : pack_key(sv, id, true);
    }
    // lanes hold the pins in id order, which is their key order: already the
    // sorted list unless a pin was dropped (-inf), which a merge compacts
    const unsigned pin_lanes = __ballot_sync(0xffffffffu, pk != 0ull);
    const unsigned all_pins = npin >= 32 ? 0xffffffffu : ((1u << npin) - 1u);
    uint64_t run = pin_lanes == all_pins ? pk : merge32<KMAX>(0ull, pk, lane);
    for (int g0 = 0; g0 < nb; g0 += 32 * kKeysPerLane) {
        float v[kKeysPerLane];
#pragma unroll
        for (int i = 0; i < kKeysPerLane; ++i) {
            const int j = g0 + 32 * i + lane;
            v[i] = j < nb ? srow[j] : neg_inf;
        }
        // coarse keys of every block as a free one (-0 as +0, as pack_key);
        // pins and -inf are sorted out among the few candidates
        uint32_t ck[kKeysPerLane];
        uint32_t cmx = 0;
#pragma unroll
        for (int i = 0; i < kKeysPerLane; ++i) {
            ck[i] = float_order_bits(v[i] + 0.0f);
            cmx = max(cmx, ck[i]);
        }
        // Once the list is full its last key is the bound (nothing below it can
        // enter); before that, the KMAX-th largest lane maximum.  Always above
        // -inf's coarse key, so padding and out-of-range blocks never qualify.
        const uint64_t tail = __shfl_sync(0xffffffffu, run, KMAX - 1);
        const uint32_t lane_bound =
            tail != 0ull ? 0u : __shfl_sync(0xffffffffu, sort32_desc_u32(cmx, lane), KMAX - 1);
        const uint32_t bound = max(max(lane_bound, coarse_of(tail)), float_order_bits(neg_inf) + 1u);
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < kKeysPerLane; ++i)
            cnt += ck[i] >= bound ? 1 : 0;
        int off = cnt;  // inclusive prefix over the lanes
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, off, o);
            if (lane >= o)
                off += u;
        }
        const int total = __shfl_sync(0xffffffffu, off, 31);
        off -= cnt;
        if (total <= kCandCap) {
#pragma unroll
            for (int i = 0; i < kKeysPerLane; ++i) {
                if (ck[i] >= bound) {
                    buf_s[off] = v[i];
                    buf_j[off] = g0 + 32 * i + lane;
                    ++off;
                }
            }
            __syncwarp();
            if (total <= 8) {
                // a few candidates: insert them one at a time
                for (int c = 0; c < total; ++c) {
                    const int j = buf_j[c];
                    const uint64_t key = (j < ns || j >= w0) ? 0ull : pack_key(buf_s[c], j, false);
                    run = insert_desc<KMAX>(run, key, lane);
                }
            } else {
                for (int c0 = 0; c0 < total; c0 += 32) {
                    uint64_t key = 0;
                    if (c0 + lane < total) {
                        const int j = buf_j[c0 + lane];
                        if (j >= ns && j < w0)
                            key = pack_key(buf_s[c0 + lane], j, false);
                    }
                    run = merge32<KMAX>(run, key, lane);
                }
            }
            __syncwarp();
        } else {
            // many ties at the bound: merge every free block of the group
#pragma unroll
            for (int i = 0; i < kKeysPerLane; ++i) {
                const int j = g0 + 32 * i + lane;
                const bool free_ok = j < nb && j >= ns && j < w0 && v[i] != neg_inf;
                run = merge32<KMAX>(run, free_ok ? pack_key(v[i], j, false) : 0ull, lane);
            }
        }
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
