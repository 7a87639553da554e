// Workspace layout and launch geometry shared by the host API and the kernels.
//
// The workspace is caller-owned device memory:
//
//   [0, 256)                  Header (fault word, geometry of the last score pass)
//   [256, 256 + P)            prefix: int32 [batch + 1], cumulative pages per request
//   [slots_offset, ...)       slots:  uint64 [capacity][4 heads][kmax] candidate lists
//
// with P = round_up(4 * (batch + 1), 256).  The pages of the whole batch are
// numbered 0..total-1 request after request (page p of the batch is logical
// block p - prefix[b] of the request b with prefix[b] <= p < prefix[b+1]).
// The score kernel cuts that sequence into chunks (see Partition below);
// chunk c contributes one top-kmax list per head for every request it
// touches, stored in slot c + b.  Slot indices are unique because both c and
// b grow along the page sequence.
#pragma once

#include <cstddef>
#include <cstdint>

namespace msa {

constexpr int kHeads = 4;
constexpr int kDim = 128;
constexpr int kPage = 128;
constexpr int kPageBytes = kPage * kDim * 2;  // 32 KiB of bf16
constexpr int kHalfPageBytes = kPageBytes / 2;
constexpr size_t kHeaderBytes = 256;

__host__ __device__ constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline int kmax_for(int k) { return k <= 16 ? 16 : 32; }

__host__ __device__ inline size_t prefix_offset() { return kHeaderBytes; }

__host__ __device__ inline size_t slots_offset(int batch)
{
    return kHeaderBytes + round_up(sizeof(int32_t) * (static_cast<size_t>(batch) + 1), 256);
}

__host__ __device__ inline size_t slot_bytes(int kmax)
{
    return static_cast<size_t>(kHeads) * kmax * sizeof(uint64_t);
}

}  // namespace msa

namespace msa {

// ---------------------------------------------------------------------------
// Partition of the batch's pages into chunks (shared by both kernels and the
// host's workspace sizing).
//
// Automatic mode (split_blocks == 0): with G score CTAs, every CTA has a home
// of H = ceil(total / G) consecutive pages.  A home is cut into 1 + T chunks:
// a "big" chunk of about 3/4 of the home, which the home CTA processes first,
// then T pool chunks of H/8, H/16, ... pages (each >= 1, T <= kMaxLevels).
// Homes under kMinPoolHome pages are short enough that the SMs' differences
// in streaming speed do not add up; they form a single chunk (T = 0).
// Pool chunks are claimed through one atomic counter in level order (every
// home's H/8 piece, then every H/16 piece, ...), so CTAs that stream faster
// take more of the tail and all CTAs finish together.
//
// Forced mode (split_blocks = W > 0): chunk c is pages [cW, cW + W); CTA g
// starts with chunk g and the rest are claimed in order.
//
// Chunks are contiguous page ranges numbered in page order and none inside
// the batch is empty, so the chunks covering a request are consecutive.
// ---------------------------------------------------------------------------
constexpr int kMaxLevels = 6;
constexpr int kMinPoolHome = 64;  // homes shorter than this keep all their pages (no pool)

struct Partition {
    int32_t forced;               // split_blocks > 0
    int32_t grid;                 // G
    int32_t total;                // pages in the batch
    int32_t unit;                 // H (automatic) or W (forced)
    int32_t levels;               // T (automatic), 0 (forced)
    int32_t chunks;               // chunk count covering [0, total)
    int32_t pool;                 // chunks claimed through the counter
    int32_t lo[kMaxLevels + 2];   // chunk r of a home covers [lo[r], lo[r+1]) (automatic)

    __host__ __device__ static Partition make(int total, int grid, int split_blocks)
    {
        Partition p;
        p.grid = grid;
        p.total = total;
        for (int i = 0; i < kMaxLevels + 2; ++i)
            p.lo[i] = 0;
        if (split_blocks > 0) {
            p.forced = 1;
            p.unit = split_blocks;
            p.levels = 0;
            p.chunks = total > 0 ? (total + split_blocks - 1) / split_blocks : 0;
            p.pool = p.chunks > grid ? p.chunks - grid : 0;
            return p;
        }
        p.forced = 0;
        const int H = total > 0 ? (total + grid - 1) / grid : 1;
        p.unit = H;
        int T = 0, pool_pages = 0;
        while (H >= kMinPoolHome && T < kMaxLevels && (H >> (T + 3)) > 0) {
            pool_pages += H >> (T + 3);
            ++T;
        }
        p.levels = T;
        p.lo[0] = 0;
        p.lo[1] = H - pool_pages;  // >= 1: the pool takes at most H/4
        for (int t = 0; t < T; ++t)
            p.lo[t + 2] = p.lo[t + 1] + (H >> (t + 3));
        p.chunks = total > 0 ? p.chunk_of(total - 1) + 1 : 0;
        p.pool = grid * T;
        return p;
    }

    // page range [a, b) of chunk c, clipped to the batch (may be empty)
    __host__ __device__ void range(int c, int &a, int &b) const
    {
        long long s, e;
        if (forced) {
            s = static_cast<long long>(c) * unit;
            e = s + unit;
        } else {
            const int g = c / (1 + levels), r = c % (1 + levels);
            const long long base = static_cast<long long>(g) * unit;
            s = base + lo[r];
            e = base + lo[r + 1];
        }
        if (s > total)
            s = total;
        if (e > total)
            e = total;
        a = static_cast<int>(s);
        b = static_cast<int>(e);
    }

    // chunk holding batch page p (0 <= p < total)
    __host__ __device__ int chunk_of(int p) const
    {
        if (forced)
            return p / unit;
        const int g = p / unit, off = p - g * unit;
        int r = 0;
        while (r < levels && lo[r + 1] <= off)
            ++r;
        return g * (1 + levels) + r;
    }

    // the chunk CTA g starts with (static), or -1
    __host__ __device__ int first_chunk(int g) const
    {
        const int c = forced ? g : g * (1 + levels);
        return c < chunks ? c : -1;
    }

    // the chunk behind pool ticket i, or -1 when the pool is exhausted
    __host__ __device__ int pool_chunk(int i) const
    {
        if (i < 0 || i >= pool)
            return -1;
        const int c = forced ? grid + i : (i % grid) * (1 + levels) + 1 + i / grid;
        return c < chunks ? c : -2;  // -2: a ticket past the batch's end (skip it)
    }
};

// Upper bound on chunks for a grid of `grid` CTAs (automatic) or the forced width.
__host__ __device__ inline long long chunk_capacity(int grid, long long max_pages, int split_blocks)
{
    if (split_blocks > 0)
        return (max_pages + split_blocks - 1) / split_blocks;
    return static_cast<long long>(grid) * (1 + kMaxLevels);
}

}  // namespace msa

namespace msa {

struct WorkspaceHeader {
    uint32_t fault;      // OR of MSA_FAULT_* bits; cleared by msa_indexer_get_error
    uint32_t pool_next;  // pool tickets handed out by the running score pass; 0 between passes
    uint32_t done;       // CTAs of the running pass done claiming; 0 between passes
    int32_t batch;       // batch of the last score pass
    int32_t kmax;        // list length of the last score pass
    uint32_t epoch;      // score passes completed on this workspace (wraps)
    uint32_t aborted;    // 1 + the count at the start of the last pass in which a wait ran out
    int32_t reserved0;
    Partition part;      // chunking of the last score pass (read by the merge)
    uint32_t reserved[(kHeaderBytes - 32 - sizeof(Partition)) / 4];
};
static_assert(sizeof(WorkspaceHeader) == kHeaderBytes, "header must be 256 bytes");

}  // namespace msa
