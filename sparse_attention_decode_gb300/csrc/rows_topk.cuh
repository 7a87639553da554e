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

constexpr int kTopkGroup = 1024;      // blocks a row pass takes at once: 32 per lane
constexpr int kTopkPerLane = kTopkGroup / 32;
constexpr int kTopkRowsPerCta = 8;    // warps per CTA, each filtering one row at a time
constexpr int kTopkCandCap = 64;      // candidates a row compacts before the all-blocks path

// Sorts 32 floats (one per lane) into descending order across the warp.
__device__ __forceinline__ float sort32_desc_f(float v, int lane)
{
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int j = size >> 1; j > 0; j >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, v, j);
            const bool desc = (lane & size) == 0;
            const bool low = (lane & j) == 0;
            v = (low == desc) ? fmaxf(v, o) : fminf(v, o);
        }
    }
    return v;
}

// A lower bound on the KMAX-th largest of a lane's 32 values `v` over the
// warp, from values that are themselves elements: KMAX = 16, the 16th
// largest of the 32 lane maxima; KMAX = 32, the 32nd largest of the 64 lane
// maxima and second maxima (the top 32 of two descending lists a and b is
// max(a[i], b[31 - i]) over i).  At least KMAX elements are >= it.
template <int KMAX>
__device__ __forceinline__ float group_bound(const float (&v)[kTopkPerLane], int lane)
{
    if constexpr (KMAX == 16) {
        float mx = v[0];
#pragma unroll
        for (int i = 1; i < kTopkPerLane; ++i)
            mx = fmaxf(mx, v[i]);
        return __shfl_sync(0xffffffffu, sort32_desc_f(mx, lane), 15);
    } else {
        float m1 = v[0], m2 = -__int_as_float(0x7f800000);
#pragma unroll
        for (int i = 1; i < kTopkPerLane; ++i) {
            m2 = fmaxf(m2, fminf(m1, v[i]));
            m1 = fmaxf(m1, v[i]);
        }
        const float a = sort32_desc_f(m1, lane);
        const float b = sort32_desc_f(m2, lane);
        float t = fmaxf(a, __shfl_sync(0xffffffffu, b, 31 - lane));
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
            t = fminf(t, __shfl_xor_sync(0xffffffffu, t, o));
        return t;
    }
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

// The fp32 score a list's last key stands for, as a bound on the scores that
// can still enter: +inf for a pinned key (no free block can), -inf for none.
__device__ __forceinline__ float tail_bound(uint64_t tail)
{
    if (tail == 0ull)
        return -__int_as_float(0x7f800000);
    if (tail >> 63)
        return __int_as_float(0x7f800000);
    int id;
    float s;
    unpack_key(tail, id, s);
    return s;
}

// 16-byte asynchronous copies global -> shared (cached in L2 only) and their
// per-thread groups.
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_addr(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

constexpr int kTopkCtasPerSm = 3;  // CTAs a SM holds (80 registers, 66 KiB each)

// Shared memory of rows_topk_kernel: per warp two group buffers (the row it
// filters and the next row's first group on its way) and the candidates.
struct TopkSmem {
    float group[kTopkRowsPerCta][2][kTopkGroup];
    int cand[kTopkRowsPerCta][kTopkCandCap];
};
constexpr size_t kTopkSmemBytes = sizeof(TopkSmem);

// Block scores [g0, min(g0 + 1024, nb)) of one row into `dst` (offsets
// 0..1023), 16 bytes a copy, lane l taking chunks 32 i + l.  With `vec` (row
// start and stride 16-byte aligned) the copies are asynchronous and one
// commit group is closed; otherwise plain loads and stores.  Values past nb
// in `dst` are left as they are: readers mask them.
__device__ __forceinline__ void fetch_group(float *dst, const float *srow, int g0, int nb, bool vec,
                                            int lane)
{
    const int n = min(kTopkGroup, nb - g0);
    if (vec) {
#pragma unroll
        for (int i = 0; i < kTopkGroup / 128; ++i) {
            const int o = 4 * (32 * i + lane);
            if (o < n)
                cp_async16(dst + o, srow + g0 + o);
        }
        cp_async_commit();
    } else {
        for (int o = lane; o < n; o += 32)
            dst[o] = __ldcs(srow + g0 + o);
    }
}

// The prefill per-row top-k.  Each warp takes rows (token, head) r, r + W,
// r + 2W, ... (W = warps in the grid) and, while it filters one, the first
// 1024 block scores of its next row are already being copied into shared
// memory.  For one row: the pins (the first n_sink and the last n_window
// visible blocks) start the running list.  The row's blocks are taken 1024
// at a time (lane l holds blocks g0 + 128 i + 4 l + e, i < 8, e < 4) and
// filtered on their fp32 scores against one bound: while the running list
// is not full, group_bound (KMAX blocks of the group score at least that
// much, so the list's KMAX-th key after this group is at least the key of
// such a block); once it is full, the score of its last key.  Only finite
// blocks at or above the bound can enter.  Each lane marks its qualifying
// blocks in a 32-bit mask and writes their offsets, one per set bit, into a
// compact candidate list (a few dozen for a random row; a group whose ties
// overflow kTopkCandCap is merged whole instead).  The candidates' keys
// (pins dropped) are sorted 32 at a time; while the list holds only pins
// they simply follow them, after that they are merged.  The list ends as the
// descending top-KMAX of all keys.
template <int KMAX>
__global__ void __launch_bounds__(32 * kTopkRowsPerCta, kTopkCtasPerSm) rows_topk_kernel(
    const float *scores, int64_t bs_stride, const int32_t *cu_q, const int32_t *seq_lens, int batch,
    int total_q, int seq_limit, int k, int n_sink, int n_window, int32_t *out_ids, float *out_scores,
    const WorkspaceHeader *hdr)
{
    extern __shared__ __align__(16) uint8_t topk_smem_raw[];
    TopkSmem &sm = *reinterpret_cast<TopkSmem *>(topk_smem_raw);
    // No early trigger: the next kernel on the stream (a persistent scoring
    // grid) is released at this grid's exit.
    griddep_wait();
    // a scoring pass whose wait ran out left its block scores incomplete:
    // every row of it is then written empty (-1 / -inf)
    const bool pass_ok = __ldcg(&hdr->aborted) != __ldcg(&hdr->epoch);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t rows = static_cast<int64_t>(total_q) * kHeads;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kTopkRowsPerCta;
    const float neg_inf = -__int_as_float(0x7f800000);
    int *buf_j = sm.cand[wid];
    const bool vec = ((reinterpret_cast<uintptr_t>(scores) & 15u) == 0) && ((bs_stride & 3) == 0);

    // the request table: with fewer than 32 requests, lane b holds cu_q[b]
    // and seq_lens[b] for the whole kernel
    const bool small = batch < 32;
    const int cq = small && lane <= batch ? cu_q[lane] : 0x7fffffff;
    const int sl = small && lane < batch ? seq_lens[lane] : 0;
    // blocks visible to row rw's token
    auto visible = [&](int64_t rw) {
        const int tok = static_cast<int>(rw / kHeads);
        Req r;
        if (small) {  // the last b with cu_q[b] <= tok
            const unsigned le = __ballot_sync(0xffffffffu, lane < batch && cq <= tok);
            const int b = le ? 31 - __clz(le) : 0;
            r = make_req(__shfl_sync(0xffffffffu, cq, b), __shfl_sync(0xffffffffu, cq, b + 1),
                         __shfl_sync(0xffffffffu, sl, b), total_q, seq_limit);
        } else {
            int lo = 0, hi = batch - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (cu_q[mid] <= tok)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            r = req_info(cu_q, seq_lens, total_q, seq_limit, lo);
        }
        return (pass_ok && r.ok && r.c0 <= tok && tok < r.c0 + r.n) ? (r.len - r.n + (tok - r.c0)) / kPage + 1
                                                                    : 0;
    };

    int64_t rw = static_cast<int64_t>(blockIdx.x) * kTopkRowsPerCta + wid;
    int nb = rw < rows ? visible(rw) : 0;
    int buf = 0;
    if (nb > 0)
        fetch_group(sm.group[wid][0], scores + rw * bs_stride, 0, nb, vec, lane);
    else if (vec)
        cp_async_commit();  // an empty group keeps one group per row
    for (; rw < rows; rw += stride) {
        const int64_t nx = rw + stride;
        const int nb_nx = nx < rows ? visible(nx) : 0;
        if (nb_nx > 0)
            fetch_group(sm.group[wid][buf ^ 1], scores + nx * bs_stride, 0, nb_nx, vec, lane);
        else if (vec)
            cp_async_commit();
        if (vec)
            cp_async_wait<1>();  // this lane's copies of the current row have landed
        __syncwarp();            // ... and every lane's
        float *gs = sm.group[wid][buf];
        const float *srow = scores + rw * bs_stride;

        // The pins (the first n_sink and the last n_window visible blocks, ids
        // ascending) go into the list first: their ids are known, and a block
        // whose page was out of range (-inf) is left out.
        const int ns = min(n_sink, nb);
        const int w0 = max(ns, nb - n_window);  // first window block that is not a sink
        const int npin = ns + (nb - w0);        // <= n_sink + n_window <= k <= KMAX
        const int pin_id = lane < ns ? lane : w0 + (lane - ns);
        float pin_s = neg_inf;
        if (lane < npin)
            pin_s = pin_id < kTopkGroup ? gs[pin_id] : srow[pin_id];
        uint64_t run = 0;  // empty row: no blocks, no pins
        for (int g0 = 0; g0 < nb; g0 += kTopkGroup) {
            if (g0 > 0) {  // a later group of a long row: loaded here, into the same buffer
                __syncwarp();
                fetch_group(gs, srow, g0, nb, vec, lane);
                if (vec)
                    cp_async_wait<0>();
                __syncwarp();
            }
            float v[kTopkPerLane];  // v[4 i + e] = block g0 + 128 i + 4 lane + e
#pragma unroll
            for (int i = 0; i < kTopkPerLane / 4; ++i) {
                const float4 x = reinterpret_cast<const float4 *>(gs)[32 * i + lane];
                v[4 * i] = x.x;
                v[4 * i + 1] = x.y;
                v[4 * i + 2] = x.z;
                v[4 * i + 3] = x.w;
            }
            if (g0 + kTopkGroup > nb) {  // the row's last, partial group
#pragma unroll
                for (int i = 0; i < kTopkPerLane; ++i)
                    if (g0 + 128 * (i >> 2) + 4 * lane + (i & 3) >= nb)
                        v[i] = neg_inf;
            }
            const bool only_pins = g0 == 0;
            if (only_pins) {
                // lanes hold the pins in id order, which is their key order: already
                // the sorted list unless a pin was dropped (-inf), which a merge compacts
                const uint64_t pk = lane < npin && pin_s != neg_inf ? pack_key(pin_s, pin_id, true) : 0ull;
                const unsigned pin_lanes = __ballot_sync(0xffffffffu, pk != 0ull);
                const unsigned all_pins = npin >= 32 ? 0xffffffffu : ((1u << npin) - 1u);
                run = pk;
                if (pin_lanes != all_pins)  // uniform: sort only when a pin was dropped
                    run = merge32<KMAX>(0ull, pk, lane);
            }
            const uint64_t tail = __shfl_sync(0xffffffffu, run, KMAX - 1);
            // while the list is not full, a bound from this group's own values
            float bound = tail == 0ull ? group_bound<KMAX>(v, lane) : tail_bound(tail);
            bound = fmaxf(bound, -3.402823466e38f);  // -inf (padding, bad pages) never qualifies
            unsigned mask = 0;
#pragma unroll
            for (int i = 0; i < kTopkPerLane; ++i)
                mask |= v[i] >= bound ? (1u << i) : 0u;
            const int cnt = __popc(mask);
            int off = cnt;  // inclusive prefix over the lanes
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, off, o);
                if (lane >= o)
                    off += u;
            }
            const int total = __shfl_sync(0xffffffffu, off, 31);
            off -= cnt;
            if (total <= kTopkCandCap) {
                while (mask != 0u) {  // this lane's candidates, one per set bit
                    const int i = __ffs(mask) - 1;
                    mask &= mask - 1u;
                    buf_j[off++] = 128 * (i >> 2) + 4 * lane + (i & 3);
                }
                __syncwarp();
                if (!only_pins && total <= 8) {
                    // a few candidates: insert them one at a time
                    for (int c = 0; c < total; ++c) {
                        const int j = g0 + buf_j[c];
                        const uint64_t key = (j < ns || j >= w0) ? 0ull : pack_key(gs[buf_j[c]], j, false);
                        run = insert_desc<KMAX>(run, key, lane);
                    }
                } else {
                    for (int c0 = 0; c0 < total; c0 += 32) {
                        uint64_t key = 0;
                        if (c0 + lane < total) {
                            const int o = buf_j[c0 + lane], j = g0 + o;
                            if (j >= ns && j < w0)
                                key = pack_key(gs[o], j, false);
                        }
                        if (only_pins && total <= 32) {
                            // the list holds pins only (np of them, lanes 0..np-1):
                            // the sorted candidates follow them
                            const uint64_t sorted = sort32_desc(key, lane);
                            const int np = __popc(__ballot_sync(0xffffffffu, run != 0ull) &
                                                  (KMAX == 32 ? 0xffffffffu : 0xffffu));
                            const uint64_t moved = __shfl_sync(0xffffffffu, sorted, (lane - np) & 31);
                            run = lane < np ? run : moved;
                        } else {
                            run = merge32<KMAX>(run, key, lane);
                        }
                    }
                }
                __syncwarp();
            } else {
                // many ties at the bound: merge every free block of the group
#pragma unroll
                for (int i = 0; i < kTopkPerLane; ++i) {
                    const int j = g0 + 128 * (i >> 2) + 4 * lane + (i & 3);
                    const bool free_ok = j < nb && j >= ns && j < w0 && v[i] != neg_inf;
                    run = merge32<KMAX>(run, free_ok ? pack_key(v[i], j, false) : 0ull, lane);
                }
            }
        }
        if (lane < k) {
            int id;
            float score;
            unpack_key(run, id, score);
            out_ids[rw * k + lane] = id;
            out_scores[rw * k + lane] = score;
        }
        __syncwarp();  // every lane is done with this buffer before it is refilled
        buf ^= 1;
        nb = nb_nx;
    }
    if (vec)
        cp_async_wait<0>();  // nothing left in flight
}

}  // namespace msa
