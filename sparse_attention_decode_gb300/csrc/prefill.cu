// Prefill scoring for the MSA lightning indexer on GB300 (sm_103a).
//
// Every new token of every request scores the blocks of its own causal prefix
// (vLLM PR #57832, reply to "Will this re-run the decode part when in mixed
// batches?": the prefill branch scores the prefill query rows over the block
// table, then takes a per-token top-k over cu_seqlens_q; prefill amortises
// each index-cache read over many query tokens).  Request b has n_b new
// tokens, its last ones: new token t sits at position seq_len_b - n_b + t and
// sees tokens [0, position].
//
// tc_prefill_pair_kernel (persistent, clusters of two CTAs, one CTA per SM):
// the product of the new tokens' query rows (token x head) with the keys is a
// dense contraction, run on the 5th-generation tensor cores, the two SMs of a
// cluster multiplying as one (tcgen05 cta_group::2).  Work unit = (tile of 64
// new tokens of one request, one visible page of that tile); the units of the
// whole batch, in order, are cut into one equal range per pair of CTAs (the
// page counts have a closed form), which balances the causal triangle.  The
// kernel itself is described where it is defined; tc_prefill_fp8_kernel
// (prefill_fp8.cuh) does the same on the E4M3 cache, also on pairs of SMs.
//
// rows_topk_kernel (rows_topk.cuh): one warp per (token, head) row: pins and
// top-k over the row's block scores.

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/msa_indexer.h"
#include "host_util.cuh"
#include "keys.cuh"
#include "layout.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace msa {

constexpr int kTileTokens = 64;  // new tokens per work tile
constexpr int kMRows = 128;      // rows each CTA of a pair multiplies: 32 tokens x 4 heads
static_assert(kTileTokens * kHeads == 2 * kMRows && kPage % kTileTokens == 0,
              "a tile's rows are split between the two CTAs of a pair");

struct TcParams {
    CUtensorMap kmap;  // pool: bf16 [num_pages*128][128] in 64x128 boxes, or E4M3
                       // codes [num_pages*128][128 B] in 128x128 boxes; 128B swizzle
    CUtensorMap qmap;  // q as [total_q*4][128] bf16, 64x128 boxes, 128B swizzle
    const float *kscale;  // E4M3 cache: fp32 [num_pages, 128] per-token scales
    const int32_t *cu_q;
    const int32_t *block_table;
    const int32_t *seq_lens;
    float *scores;  // [total_q, 4, bs_stride]
    uint32_t *fault;
    WorkspaceHeader *hdr;  // fault word, pass count and aborted pass of the workspace
    int64_t bt_stride;
    int64_t bs_stride;
    int64_t num_pages;
    int batch;
    int seq_limit;
    int total_q;
};

// One request as the kernels see it.  ok = false for a request they refuse:
// rows outside [0, total_q) or out of order, a length past the limit or
// negative, or more new tokens than tokens.
struct Req {
    int n, len, c0;
    bool ok;
};

// A request from its row range [c0, c1) and length.
__device__ __forceinline__ Req make_req(int c0, int c1, int len, int total_q, int seq_limit)
{
    Req r;
    r.c0 = c0;
    r.n = c1 - c0;
    r.len = len;
    r.ok = c0 >= 0 && c1 <= total_q && r.n >= 0 && len >= 0 && len <= seq_limit && r.n <= len;
    return r;
}
__device__ __forceinline__ Req req_info(const int32_t *cu_q, const int32_t *seq_lens, int total_q,
                                        int seq_limit, int b)
{
    return make_req(cu_q[b], cu_q[b + 1], seq_lens[b], total_q, seq_limit);
}

__device__ __forceinline__ int tiles_of(const Req &r) { return (r.n + kTileTokens - 1) / kTileTokens; }

// Pages tile t sees: those up to its last token's position.
__device__ __forceinline__ int tile_pages(const Req &r, int t)
{
    const int last = min(r.n, kTileTokens * (t + 1)) - 1;
    return (r.len - r.n + last) / kPage + 1;
}

// Pages of tiles [0, t) for t <= tiles - 1 (all full tiles).  Full tile t'
// ends at position c + T t' (T = kTileTokens, c = len - n + T - 1) and sees
// floor((c + T t') / 128) + 1 pages; writing t' = R m + r with R = 128 / T,
// that is m + floor((c + T r) / 128) + 1, so the tiles of residue r sum in
// closed form.
__device__ __forceinline__ long long pages_before(const Req &r, int t)
{
    constexpr int R = kPage / kTileTokens;
    const long long c = static_cast<long long>(r.len) - r.n + kTileTokens - 1;
    long long sum = t;
#pragma unroll
    for (int res = 0; res < R; ++res) {
        const long long n_r = t > res ? (t - res + R - 1) / R : 0;  // tiles t' < t with t' % R == res
        sum += n_r * ((c + static_cast<long long>(kTileTokens) * res) / kPage) + n_r * (n_r - 1) / 2;
    }
    return sum;
}

__device__ __forceinline__ long long req_units(const Req &r)
{
    if (!r.ok || r.n == 0)
        return 0;
    const int T = tiles_of(r);
    return pages_before(r, T - 1) + tile_pages(r, T - 1);
}

__device__ __forceinline__ long long warp_sum64(long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ long long warp_incl_scan64(long long v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o)
            v += u;
    }
    return v;
}

// Walks a CTA's range of (tile, page) units one segment (the range's pages
// of one tile) at a time, last tile first: the range's last tile begins at
// page 0, so the CTAs that score the tiles of one request step through its
// pages nearly together (two fronts: those still in their last tile and those
// back in the tail of the one before), and each page is read from DRAM about
// twice instead of once per tile.  Pages within a segment go in order.
struct Cursor {
    int b, t, j, je;  // segment: pages [j, je) of tile t of request b
    Req r;
    int fb, ft, fj;   // the range's first unit

    __device__ __forceinline__ void load(const TcParams &p, int b0, int t0, int j0, int b1, int t1, int j1)
    {
        fb = b0;
        ft = t0;
        fj = j0;
        b = b1;
        t = t1;
        r = req_info(p.cu_q, p.seq_lens, p.total_q, p.seq_limit, b);
        je = j1;
        j = (b == fb && t == ft) ? fj : 0;
    }

    // Moves to the segment before; false past the range's first tile.
    __device__ __forceinline__ bool next(const TcParams &p)
    {
        if (b == fb && t == ft)
            return false;
        if (t > 0) {
            --t;
        } else {
            do {
                --b;
                r = req_info(p.cu_q, p.seq_lens, p.total_q, p.seq_limit, b);
            } while (b > fb && !(r.ok && r.n > 0));
            t = tiles_of(r) - 1;
        }
        je = tile_pages(r, t);
        j = (b == fb && t == ft) ? fj : 0;
        return true;
    }
};

// The (request, tile, page) of unit u of the batch's (tile, page) units in
// order (0 <= u < the unit count).  Run by one warp; every lane gets it.
__device__ __forceinline__ void locate_unit(const TcParams &p, long long u, int lane, int &ub, int &ut, int &uj)
{
    int fb = 0;
    long long base = 0, cum = 0;
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
        long long v = 0;
        if (b0 + lane < p.batch)
            v = req_units(req_info(p.cu_q, p.seq_lens, p.total_q, p.seq_limit, b0 + lane));
        const long long incl = warp_incl_scan64(v, lane);
        const long long total = __shfl_sync(0xffffffffu, incl, 31);
        if (cum + total > u) {
            const unsigned m = __ballot_sync(0xffffffffu, cum + incl > u);
            const int l = __ffs(m) - 1;
            fb = b0 + l;
            base = cum + __shfl_sync(0xffffffffu, incl - v, l);
            break;
        }
        cum += total;
    }
    const Req r = req_info(p.cu_q, p.seq_lens, p.total_q, p.seq_limit, fb);
    const long long rel = u - base;
    // the last tile t with pages_before(t) <= rel
    int lo = 0, hi = tiles_of(r) - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pages_before(r, mid) <= rel)
            lo = mid;
        else
            hi = mid - 1;
    }
    ub = fb;
    ut = lo;
    uj = static_cast<int>(rel - pages_before(r, lo));
}

// A range of work units: its first (tile, page) unit, its last + 1 page, and
// its unit count.
struct UnitRange {
    int b0, t0, j0;
    int b1, t1, j1;
    long long units;
};

// The batch's (tile, page) unit count W.  Run by one warp (every lane gets
// it); the first CTA flags the requests the kernels refuse.
__device__ long long batch_units(const TcParams &p, int lane)
{
    long long W = 0;
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
        long long v = 0;
        if (b0 + lane < p.batch) {
            const Req r = req_info(p.cu_q, p.seq_lens, p.total_q, p.seq_limit, b0 + lane);
            if (!r.ok && blockIdx.x == 0)
                atomicOr(p.fault, MSA_FAULT_SEQ_LEN);
            v = req_units(r);
        }
        W += warp_sum64(v);
    }
    return W;
}

// Range g of the batch's W units, in order, cut G ways: [W*g/G, W*(g+1)/G).
// Run by one warp; writes the range's first and last positions and its unit
// count into *ctl (a UnitRange, or a control block with the same fields).
template <class Ctl>
__device__ void plan_range_of(const TcParams &p, Ctl *ctl, int lane, long long W, long long G, long long g)
{
    const long long u0 = W * g / G, u1 = W * (g + 1) / G;
    if (u1 <= u0) {
        if (lane == 0)
            ctl->units = 0;
        return;
    }
    int b0, t0, j0, b1, t1, j1;
    locate_unit(p, u0, lane, b0, t0, j0);
    locate_unit(p, u1 - 1, lane, b1, t1, j1);
    if (lane == 0) {
        ctl->b0 = b0;
        ctl->t0 = t0;
        ctl->j0 = j0;
        ctl->b1 = b1;
        ctl->t1 = t1;
        ctl->j1 = j1 + 1;
        ctl->units = u1 - u0;
    }
}

template <class Ctl>
__device__ void plan_range(const TcParams &p, Ctl *ctl, int lane, long long G, long long g)
{
    plan_range_of(p, ctl, lane, batch_units(p, lane), G, g);
}

template <class Ctl>
__device__ __forceinline__ bool aborted(const Ctl *ctl)
{
    return *reinterpret_cast<const volatile int *>(&ctl->abort) != 0;
}

template <class Ctl>
__device__ __forceinline__ void give_up(const TcParams &p, Ctl *ctl)
{
    atomicOr(p.fault, MSA_FAULT_TIMEOUT);
    *reinterpret_cast<volatile int *>(&ctl->abort) = 1;
}

// Pass bookkeeping in the workspace header, as the decode kernels keep it:
// thread 0 of each CTA reads the pass count once the previous kernel on the
// stream has finished; at its exit a CTA that gave up records that count + 1
// as the aborted pass, and the last CTA to finish bumps the count.  The top-k
// kernel that follows compares the two and writes -1 / -inf to every row of a
// pass that gave up (its block scores are incomplete).
template <class Ctl>
__device__ __forceinline__ void pass_start(const TcParams &p, Ctl *ctl)
{
    ctl->epoch = __ldcg(&p.hdr->epoch);
}

// Thread 0 of each CTA, after a barrier that every thread of the CTA reached
// once all its waits had ended.
template <class Ctl>
__device__ __forceinline__ void pass_end(const TcParams &p, const Ctl *ctl)
{
    if (aborted(ctl))
        atomicExch(&p.hdr->aborted, ctl->epoch + 1u);
    __threadfence();
    if (atomicAdd(&p.hdr->done, 1u) == gridDim.x - 1) {
        atomicExch(&p.hdr->done, 0u);
        atomicAdd(&p.hdr->epoch, 1u);
    }
}

// Bounded waits.  The test copy of the pair kernel (TH = true, which loads
// nothing) polls 2^14 times instead of the normal limit, so that its waits
// run out quickly.
constexpr uint32_t kTestSpinLimit = 1u << 14;
template <bool TH>
constexpr uint32_t kWaitPolls = TH ? kTestSpinLimit : kSpinLimit;

template <bool TH>
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity)
{
    for (uint32_t i = 0; i < kWaitPolls<TH>; ++i)
        if (mbar_try_wait(bar, parity))
            return true;
    return false;
}

// A shared-memory word published by one thread (release) and polled by
// another (acquire), CTA scope.
__device__ __forceinline__ uint32_t ld_acquire_shared_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_shared_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// The issuing thread's wait for its unit of work number need - 1 (a page, or
// a pair of pages): the waiter warp raises `ready` to n once units 0 .. n-1
// have their operands in shared memory and their accumulator buffer free.  An
// mbarrier wait costs the thread that makes it ~250 cycles even when the
// phase has long completed; two a page in the issuing thread cost it ~500 of
// the ~1700 cycles a page took.  This load of a counter that is usually
// already there is cheaper, and the waits happen on another warp.
template <class Ctl>
__device__ __forceinline__ bool wait_ready(Ctl *ctl, uint32_t need, uint32_t limit = kSpinLimit)
{
    const uint32_t addr = smem_addr(&ctl->ready);
    for (uint32_t i = 0; i < limit; ++i) {
        if (ld_acquire_shared_u32(addr) >= need)
            return true;
        if (aborted(ctl))
            return false;
    }
    return false;
}

// ---------------- pairs of SMs, two pages per MMA (bf16 cache) ----------------
// tc_prefill_pair_kernel: the (tile, page) units split over clusters of two
// CTAs that multiply as one (tcgen05 cta_group::2).  A tile's 256 query rows
// are split 128 / 128 between the even and the odd CTA; its pages are taken
// two at a time, the even CTA holding the first page of each pair and the odd
// CTA the second (a segment's odd last page is paired with nothing).  One
// thread of the even CTA issues 8 MMAs of M = 256 rows x N = 256 keys x
// K = 16 per pair of pages; each SM's tensor core computes its own 128 rows x
// 256 keys (128 cycles an MMA), into its own TMEM (two accumulator buffers of
// 256 columns).  A single thread issues a tcgen05.mma in ~70 cycles whatever
// its size, so with M = 128 x N = 128 MMAs (64 cycles of tensor work each)
// the issuing thread, not the tensor pipe, set the pace (~1500 cycles a page
// against 1024); here it issues a pair's 8 MMAs in ~700 cycles against 1024.
// Each SM still reads one page from L2 or DRAM per 256 rows multiplied.
// Per CTA:
//   warp 0     TMA producer: its 128 query rows at each tile (two tiles'
//              rows resident), its page of each pair through a 5-stage ring;
//   warp 1     TMEM allocation (both CTAs, collectively); even CTA: one
//              thread issues the MMAs; odd CTA: one thread tells the even CTA
//              that its query rows and each of its pages have landed;
//   warps 2-9  epilogue: warps 2-5 the pair's first page, 6-9 its second,
//              one TMEM lane quarter each: all 128 columns of the warp's rows
//              into registers, the accumulator buffer handed back to the even
//              CTA at once, then the masked block max (reducing before the
//              hand-back left the issuing thread waiting ~650 cycles a pair);
//   warp 10    even CTA: waits for both pages of a pair and a free
//              accumulator buffer and counts the pairs the issuing thread
//              may multiply.
// Every wait is bounded; a CTA that gives up still meets its partner at the
// final cluster barrier, after which TMEM is freed.
constexpr int kP2Stages = 5;
constexpr int kP2QBufs = 2;  // a tile's query rows load while the previous tile is multiplied
constexpr long long kP2SplitUnits = 512;  // units a half-range needs for the two-range walk
constexpr int kP2AccBufs = 2;
constexpr uint32_t kP2TmemCols = kP2AccBufs * 2 * kPage;  // 512
constexpr uint32_t kP2QBytes = kMRows * kDim * 2;          // 32 KiB: 128 query rows
constexpr uint32_t kP2QHalf = kP2QBytes / 2;               // 128 rows x 64 dims
constexpr uint32_t kP2Idesc = umma_idesc_bf16_f32(2 * kMRows, 2 * kPage);
constexpr int kP2EpiWarps = 8;
constexpr int kP2WaiterWarp = 2 + kP2EpiWarps;
constexpr int kP2Threads = 32 * (3 + kP2EpiWarps);
static_assert(kP2TmemCols <= 512, "TMEM columns");

struct P2Smem {
    uint64_t k_full[kP2Stages];
    uint64_t k_peer[kP2Stages];  // even CTA: the odd CTA's page of the stage has landed
    uint64_t k_empty[kP2Stages];
    uint64_t q_full[kP2QBufs];
    uint64_t q_peer[kP2QBufs];   // even CTA: the odd CTA's query rows have landed
    uint64_t q_empty[kP2QBufs];
    uint64_t acc_full[kP2AccBufs];
    uint64_t acc_empty[kP2AccBufs];  // even CTA: both CTAs' epilogue warps
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t ready;  // even CTA: pairs of pages the issuing thread may multiply
    uint32_t epoch;  // the workspace's pass count when this pass started
    int abort;
    UnitRange rng[2];  // the pair's two ranges of units, walked one after the other
};

constexpr size_t kP2SmemBytes = 1024 + kP2QBufs * kP2QBytes + static_cast<size_t>(kP2Stages) * kPageBytes + sizeof(P2Smem);
static_assert(kP2SmemBytes <= 227 * 1024, "shared memory per CTA");

__device__ __forceinline__ int pairs_of(int j, int je) { return (je - j + 1) / 2; }

// The segments of a pair's two ranges in walking order: each range from its
// last tile back to its first, pages in order within a tile (as Cursor walks
// one range); every role of the kernel walks the same ones.  The current
// range's first unit stays in shared memory, which keeps the epilogue (a
// row's 128 accumulators in registers) within its register budget.
struct SegWalk {
    int b, t, j, je;  // segment: pages [j, je) of tile t of request b
    Req r;
    long long left;   // units of the current range from this segment on
    int k;            // the current range

    __device__ __forceinline__ bool next_range(const TcParams &p, const UnitRange *rng)
    {
        while (++k < 2) {
            const UnitRange &R = rng[k];
            if (R.units > 0) {
                b = R.b1;
                t = R.t1;
                r = req_info(p.cu_q, p.seq_lens, p.total_q, p.seq_limit, b);
                je = R.j1;
                j = (b == R.b0 && t == R.t0) ? R.j0 : 0;
                left = R.units;
                return true;
            }
        }
        return false;
    }
    __device__ __forceinline__ bool start(const TcParams &p, const UnitRange *rng)
    {
        k = -1;
        return next_range(p, rng);
    }
    // After the current segment: the next one; false when both ranges are done.
    __device__ __forceinline__ bool next(const TcParams &p, const UnitRange *rng)
    {
        left -= je - j;
        if (left <= 0)
            return next_range(p, rng);
        const UnitRange &R = rng[k];
        if (b == R.b0 && t == R.t0)
            return false;  // past the range's first tile (not reached: left counts its units)
        if (t > 0) {
            --t;
        } else {
            do {
                --b;
                r = req_info(p.cu_q, p.seq_lens, p.total_q, p.seq_limit, b);
            } while (b > R.b0 && !(r.ok && r.n > 0));
            t = tiles_of(r) - 1;
        }
        je = tile_pages(r, t);
        j = (b == R.b0 && t == R.t0) ? R.j0 : 0;
        return true;
    }
};

template <bool TH>
__global__ void __launch_bounds__(kP2Threads, 1) tc_prefill_pair_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t q_smem = smem_addr(smem);
    const uint32_t k_smem = q_smem + kP2QBufs * kP2QBytes;
    P2Smem *ctl = reinterpret_cast<P2Smem *>(smem + kP2QBufs * kP2QBytes + kP2Stages * kPageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: the CTA that issues the MMAs

    if (threadIdx.x == 0) {
        for (int s = 0; s < kP2Stages; ++s) {
            mbar_init(smem_addr(&ctl->k_full[s]), 1);
            mbar_init(smem_addr(&ctl->k_peer[s]), 1);
            mbar_init(smem_addr(&ctl->k_empty[s]), 1);
        }
        for (int b = 0; b < kP2QBufs; ++b) {
            mbar_init(smem_addr(&ctl->q_full[b]), 1);
            mbar_init(smem_addr(&ctl->q_peer[b]), 1);
            mbar_init(smem_addr(&ctl->q_empty[b]), 1);
        }
        for (int a = 0; a < kP2AccBufs; ++a) {
            mbar_init(smem_addr(&ctl->acc_full[a]), 1);
            mbar_init(smem_addr(&ctl->acc_empty[a]), 2 * kP2EpiWarps);
        }
        mbar_init(smem_addr(&ctl->mma_done), 1);
        ctl->abort = 0;
        ctl->ready = 0;
        fence_barrier_init();
    }
    griddep_wait();
    griddep_launch_dependents();
    if (threadIdx.x == 0)
        pass_start(p, ctl);
    // On a large batch pair g of G takes ranges g and g + G of the units cut
    // 2G ways.  The first ranges of all pairs cover the first half of the
    // batch's units and the second ranges the rest, so at any time the pairs
    // stream each request's pages on the few fronts a single-CTA split has: a
    // pair walking one range of twice the length restarts at page 0
    // mid-range, and on the chunked prefill of 4 x 2048 tokens at 128K each
    // page then left DRAM ~5.6 times instead of about once.  A smaller batch
    // (fewer than kP2SplitUnits units a half-range) takes range g of G: there
    // the extra segments of the two-range walk cost more than L2 reuse gives.
    if (warp == 0) {
        const long long W = batch_units(p, lane);
        const long long G = gridDim.x / 2, g = blockIdx.x / 2;
        if (W >= 2 * G * kP2SplitUnits) {
            plan_range_of(p, &ctl->rng[0], lane, W, 2 * G, g);
            plan_range_of(p, &ctl->rng[1], lane, W, 2 * G, g + G);
        } else {
            plan_range_of(p, &ctl->rng[0], lane, W, G, g);
            if (lane == 0)
                ctl->rng[1].units = 0;
        }
    }
    __syncwarp();
    // both CTAs' barriers are initialised before either arrives on the other's
    cluster_sync_all();
    if (ctl->rng[0].units + ctl->rng[1].units <= 0) {
        if (threadIdx.x == 0)  // the same for both CTAs of the pair: no TMEM taken yet
            pass_end(p, ctl);
        return;
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(&ctl->tmem_base), kP2TmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 0 && TH) {
        // test copy: no query row or page is loaded and no stage is signalled,
        // so every wait on one runs out; no copy is ever in flight
    } else if (warp == 0) {
        // ---------------- producer (both CTAs) ----------------
        SegWalk w;
        bool more = w.start(p, ctl->rng);
        const SegWalk &c = w;
        uint32_t gc = 0, seg = 0;
        bool ok_run = true;
        while (more && ok_run) {
            const int je = c.je;
            if (lane == 0) {
                const int qb = static_cast<int>(seg % kP2QBufs);
                if (seg >= kP2QBufs &&
                    !bar_wait<TH>(smem_addr(&ctl->q_empty[qb]), ((seg / kP2QBufs) - 1) & 1u)) {
                    give_up(p, ctl);
                    ok_run = false;
                } else {
                    const uint32_t qf = smem_addr(&ctl->q_full[qb]);
                    const uint32_t qdst = q_smem + static_cast<uint32_t>(qb) * kP2QBytes;
                    const int row0 = (c.r.c0 + kTileTokens * c.t) * kHeads + kMRows * static_cast<int>(rank);
                    mbar_arrive_expect_tx(qf, kP2QBytes);
                    tma_load_2d(qdst, &p.qmap, 0, row0, qf);
                    tma_load_2d(qdst + kP2QHalf, &p.qmap, 64, row0, qf);
                }
            }
            ok_run = __shfl_sync(0xffffffffu, ok_run ? 1 : 0, 0) != 0;
            const int ng = pairs_of(c.j, je);
            for (int gb = 0; gb < ng && ok_run; gb += 32) {
                const int gl = gb + lane;
                const int jl = c.j + 2 * gl + static_cast<int>(rank);  // this CTA's page of pair gl
                int page = 0, ok = 0;
                if (gl < ng && jl < je) {
                    page = p.block_table[static_cast<int64_t>(c.b) * p.bt_stride + jl];
                    ok = (page >= 0 && page < p.num_pages) ? 1 : 0;
                    if (!ok)
                        atomicOr(p.fault, MSA_FAULT_PAGE_ID);
                }
                const int cnt = min(32, ng - gb);
                for (int i = 0; i < cnt; ++i) {
                    const int pg = __shfl_sync(0xffffffffu, page, i);
                    const int pok = __shfl_sync(0xffffffffu, ok, i);
                    int good = 1;
                    if (lane == 0) {
                        const int s = static_cast<int>(gc % kP2Stages);
                        const uint32_t full = smem_addr(&ctl->k_full[s]);
                        if (aborted(ctl) ||
                            (gc >= kP2Stages &&
                             !bar_wait<TH>(smem_addr(&ctl->k_empty[s]), ((gc / kP2Stages) - 1) & 1u))) {
                            give_up(p, ctl);
                            good = 0;
                        } else if (pok) {
                            const uint32_t dst = k_smem + s * kPageBytes;
                            mbar_arrive_expect_tx(full, kPageBytes);
                            tma_load_2d(dst, &p.kmap, 0, pg * kPage, full);
                            tma_load_2d(dst + kHalfPageBytes, &p.kmap, 64, pg * kPage, full);
                        } else {
                            mbar_arrive(full);  // no page here (odd tail or bad id): nothing to load
                        }
                    }
                    if (__shfl_sync(0xffffffffu, good, 0) == 0) {
                        ok_run = false;
                        break;
                    }
                    ++gc;
                }
            }
            ++seg;
            more = w.next(p, ctl->rng);
        }
        if (lane == 0) {  // drain: no copy may land after the CTA exits
            for (uint32_t i = gc > kP2Stages ? gc - kP2Stages : 0; i < gc; ++i)
                if (!bar_wait<TH>(smem_addr(&ctl->k_full[i % kP2Stages]), (i / kP2Stages) & 1u))
                    give_up(p, ctl);
            for (uint32_t i = seg > kP2QBufs ? seg - kP2QBufs : 0; i < seg; ++i)
                if (!bar_wait<TH>(smem_addr(&ctl->q_full[i % kP2QBufs]), (i / kP2QBufs) & 1u))
                    give_up(p, ctl);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            SegWalk w;
            bool more = w.start(p, ctl->rng);
            const SegWalk &c = w;
            uint32_t gc = 0, seg = 0;
            bool ok_run = true;
            if (rank == 0) {
                // ---------------- MMA issue for the pair ----------------
                while (more && ok_run) {
                    const int je = c.je;
                    const int qb = static_cast<int>(seg % kP2QBufs);
                    const uint32_t qph = (seg / kP2QBufs) & 1u;
                    if (!bar_wait<TH>(smem_addr(&ctl->q_full[qb]), qph) || !bar_wait<TH>(smem_addr(&ctl->q_peer[qb]), qph)) {
                        give_up(p, ctl);
                        break;
                    }
                    const uint32_t a_lo = umma_desc_lo(q_smem + static_cast<uint32_t>(qb) * kP2QBytes);
                    const int ng = pairs_of(c.j, je);
                    for (int g = 0; g < ng; ++g) {
                        const int s = static_cast<int>(gc % kP2Stages);
                        const int a = static_cast<int>(gc % kP2AccBufs);
                        if (!wait_ready(ctl, gc + 1, kWaitPolls<TH>)) {
                            give_up(p, ctl);
                            ok_run = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t b_lo = umma_desc_lo(k_smem + s * kPageBytes);
                        const uint32_t d = tmem + static_cast<uint32_t>(a * 2 * kPage);
#pragma unroll
                        for (int ks = 0; ks < kDim / 16; ++ks) {
                            const uint32_t qo = ((ks >> 2) * kP2QHalf + (ks & 3) * 32) >> 4;
                            const uint32_t ko = ((ks >> 2) * kHalfPageBytes + (ks & 3) * 32) >> 4;
                            if (ks == 0)
                                umma_pair_f16<false>(d, a_lo + qo, b_lo + ko, kP2Idesc);
                            else
                                umma_pair_f16<true>(d, a_lo + qo, b_lo + ko, kP2Idesc);
                        }
                        umma_commit_pair(smem_addr(&ctl->k_empty[s]));
                        umma_commit_pair(smem_addr(&ctl->acc_full[a]));
                        ++gc;
                    }
                    umma_commit_pair(smem_addr(&ctl->q_empty[qb]));
                    ++seg;
                    more = w.next(p, ctl->rng);
                }
                // every MMA issued has completed before TMEM is freed or either CTA exits
                umma_commit_pair(smem_addr(&ctl->mma_done));
            } else {
                // ---------------- odd CTA: its query rows and pages have landed ----------------
                while (more && ok_run) {
                    const int je = c.je;
                    const int qb = static_cast<int>(seg % kP2QBufs);
                    if (!bar_wait<TH>(smem_addr(&ctl->q_full[qb]), (seg / kP2QBufs) & 1u)) {
                        give_up(p, ctl);
                        break;
                    }
                    mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->q_peer[qb]), 0));
                    const int ng = pairs_of(c.j, je);
                    for (int g = 0; g < ng; ++g) {
                        const int s = static_cast<int>(gc % kP2Stages);
                        if (aborted(ctl) || !bar_wait<TH>(smem_addr(&ctl->k_full[s]), (gc / kP2Stages) & 1u)) {
                            give_up(p, ctl);
                            ok_run = false;
                            break;
                        }
                        mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->k_peer[s]), 0));
                        ++gc;
                    }
                    ++seg;
                    more = w.next(p, ctl->rng);
                }
            }
            if (!bar_wait<TH>(smem_addr(&ctl->mma_done), 0))
                give_up(p, ctl);
        }
        __syncwarp();
    } else if (warp == kP2WaiterWarp) {
        // ---------------- even CTA: pair gc may be multiplied ----------------
        if (rank == 0 && lane == 0) {
            const uint32_t addr = smem_addr(&ctl->ready);
            SegWalk w;
            bool more = w.start(p, ctl->rng);
            const SegWalk &c = w;
            uint32_t gc = 0;
            bool ok_run = true;
            while (more && ok_run) {
                const int je = c.je;
                const int ng = pairs_of(c.j, je);
                for (int g = 0; g < ng; ++g) {
                    const int s = static_cast<int>(gc % kP2Stages);
                    const int a = static_cast<int>(gc % kP2AccBufs);
                    if (aborted(ctl) || !bar_wait<TH>(smem_addr(&ctl->k_full[s]), (gc / kP2Stages) & 1u) ||
                        !bar_wait<TH>(smem_addr(&ctl->k_peer[s]), (gc / kP2Stages) & 1u) ||
                        (gc >= kP2AccBufs &&
                         !bar_wait<TH>(smem_addr(&ctl->acc_empty[a]), ((gc / kP2AccBufs) - 1) & 1u))) {
                        give_up(p, ctl);
                        ok_run = false;
                        break;
                    }
                    st_release_shared_u32(addr, gc + 1);
                    ++gc;
                }
                more = w.next(p, ctl->rng);
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: TMEM -> block scores ----------------
        const int h = (warp - 2) >> 2;  // 0: the pair's first page, 1: its second
        const int quarter = warp & 3;
        const int row_in_tile = kMRows * static_cast<int>(rank) + 32 * quarter + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + static_cast<uint32_t>(h * kPage);
        const float neg_inf = -__int_as_float(0x7f800000);
        SegWalk w;
        bool more = w.start(p, ctl->rng);
        const SegWalk &c = w;
        uint32_t gc = 0;
        bool ok_run = true;
        while (more && ok_run) {
            const int je = c.je;
            const int tl = kTileTokens * c.t + (row_in_tile >> 2);
            const int head = row_in_tile & 3;
            const bool live = tl < c.r.n;
            const int pos = c.r.len - c.r.n + tl;
            float *out = p.scores + (static_cast<int64_t>(c.r.c0 + tl) * kHeads + head) * p.bs_stride;
            const int32_t *bt_row = p.block_table + static_cast<int64_t>(c.b) * p.bt_stride;
            const int ng = pairs_of(c.j, je);
            // this warp's page of each pair, its block-table entry read a pair ahead
            int page_next = c.j + h < je ? bt_row[c.j + h] : 0;
            for (int g = 0; g < ng; ++g, ++gc) {
                const int a = static_cast<int>(gc % kP2AccBufs);
                const int j = c.j + 2 * g + h;
                const int page = page_next;
                if (j + 2 < je)
                    page_next = bt_row[j + 2];
                bool ready = !aborted(ctl) && bar_wait<TH>(smem_addr(&ctl->acc_full[a]), (gc / kP2AccBufs) & 1u);
                ready = __all_sync(0xffffffffu, ready);
                if (!ready) {
                    if (lane == 0)
                        give_up(p, ctl);
                    ok_run = false;
                    break;
                }
                tc_fence_after_sync();
                const bool page_ok = page >= 0 && page < p.num_pages;
                const int first_key = j * kPage;
                const bool want = j < je && live && first_key <= pos;
                const bool math = j < je && page_ok && __any_sync(0xffffffffu, want);
                // all 128 columns into registers, the buffer handed back at once,
                // then the masked max
                uint32_t r0[32], r1[32], r2[32], r3[32];
                if (math) {
                    const uint32_t col = lane_addr + static_cast<uint32_t>(a * 2 * kPage);
                    tmem_ld32(col, r0);
                    tmem_ld32(col + 32, r1);
                    tmem_ld32(col + 64, r2);
                    tmem_ld32(col + 96, r3);
                    tmem_wait_ld(r0);
                    tmem_regs_ready(r1);
                    tmem_regs_ready(r2);
                    tmem_regs_ready(r3);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->acc_empty[a]), 0));
                if (math) {
                    const int lim = pos - first_key;  // keys i <= lim of the page are visible
                    float mx = neg_inf;
                    if (lim >= kPage - 1) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            mx = fmaxf(fmaxf(mx, __uint_as_float(r0[i])),
                                       fmaxf(__uint_as_float(r1[i]), fmaxf(__uint_as_float(r2[i]), __uint_as_float(r3[i]))));
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            mx = fmaxf(mx, i <= lim ? __uint_as_float(r0[i]) : neg_inf);
                            mx = fmaxf(mx, i + 32 <= lim ? __uint_as_float(r1[i]) : neg_inf);
                            mx = fmaxf(mx, i + 64 <= lim ? __uint_as_float(r2[i]) : neg_inf);
                            mx = fmaxf(mx, i + 96 <= lim ? __uint_as_float(r3[i]) : neg_inf);
                        }
                    }
                    if (want)
                        out[j] = mx;
                } else if (j < je && !page_ok && want) {
                    out[j] = neg_inf;
                }
            }
            more = w.next(p, ctl->rng);
        }
    }

    // all of both CTAs' work is done (the issuing thread has seen its last MMA
    // complete) before either frees TMEM or exits
    tc_fence_before_sync();
    __syncwarp();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, kP2TmemCols);
    }
    if (threadIdx.x == 0)
        pass_end(p, ctl);
}

}  // namespace msa

#include "prefill_fp8.cuh"
#include "rows_topk.cuh"

namespace msa {

bool test_withhold_pages();  // msa_indexer.cu: the bounded-wait test hook is set

// 2-D tensor map over the E4M3 codes: [num_pages*128 rows][128 B], one
// 128x128-byte box per page, 128-byte swizzle.
static bool make_codes_map(CUtensorMap *map, const void *base, int64_t rows)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDim)};
    const cuuint32_t box[2] = {128u, 128u};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor map over `rows` rows of 128 elements (256 B), 64x128 boxes,
// 128-byte swizzle: two boxes fill one 128x128 operand tile.
static bool make_rows_map(CUtensorMap *map, const void *base, int64_t rows)
{
    EncodeTiledFn enc = encode_tiled();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDim) * 2};
    const cuuint32_t box[2] = {64u, 128u};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of two the pair kernels run: one per two SMs, fewer if the GPU
// cannot hold that many at once (queried once per device, on the bf16
// kernel; the E4M3 one also holds one CTA an SM).
static int pair_clusters(int dev, int sms)
{
    static std::atomic<int> cache[kMaxDevices];
    int v = (dev >= 0 && dev < kMaxDevices) ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (v > 0)
        return v;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(sms / 2 * 2));
    cfg.blockDim = dim3(kP2Threads);
    cfg.dynamicSmemBytes = kP2SmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_prefill_pair_kernel<false>, &cfg) != cudaSuccess || n <= 0)
        n = sms / 2;
    v = n < sms / 2 ? n : sms / 2;
    if (v < 1)
        v = 1;
    if (dev >= 0 && dev < kMaxDevices)
        cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

}  // namespace msa

using namespace msa;

extern "C" size_t msa_indexer_prefill_workspace_bytes(int max_total_q, int max_model_len)
{
    if (max_total_q < 0 || max_model_len < 1)
        return 0;
    return kHeaderBytes + static_cast<size_t>(max_total_q) * kHeads *
                              static_cast<size_t>(blocks_for(max_model_len)) * sizeof(float);
}

// Checks the arguments and launches the score kernel; fills *pp (the block
// score buffer it writes: the caller's, else the workspace's).
static msa_status prefill_score_launch(const void *q, const int32_t *cu_seqlens_q, int total_q,
                                       const void *kcache_pool, const float *kscale,
                                       int64_t num_pages, const int32_t *block_table,
                                       int64_t bt_stride, const int32_t *seq_lens, int batch,
                                       int max_model_len, float *out_block_scores, void *workspace,
                                       size_t workspace_bytes, cudaStream_t st, TcParams *pp,
                                       bool fp8)
{
    if ((!q && total_q > 0) || !cu_seqlens_q || !kcache_pool || !block_table || !seq_lens ||
        !workspace)
        return MSA_ERR_INVALID_ARG;
    if (fp8 && (!kscale || (reinterpret_cast<uintptr_t>(kscale) & 15)))
        return MSA_ERR_INVALID_ARG;
    if (total_q < 0 || batch < 1 || max_model_len < 1 || num_pages < 1 || bt_stride < 1)
        return MSA_ERR_INVALID_ARG;
    if (batch > MSA_MAX_BATCH || num_pages > (int64_t{1} << 24) || total_q > (1 << 28))
        return MSA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(kcache_pool) & 15) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255))
        return MSA_ERR_INVALID_ARG;
    const int64_t bs_stride = blocks_for(max_model_len);
    const size_t scores_bytes = static_cast<size_t>(total_q) * kHeads * bs_stride * sizeof(float);
    const size_t need = kHeaderBytes + (out_block_scores ? 0 : scores_bytes);
    if (workspace_bytes < need)
        return MSA_ERR_WORKSPACE_TOO_SMALL;
    TcParams &p = *pp;
    std::memset(&p, 0, sizeof p);
    p.cu_q = cu_seqlens_q;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.scores = out_block_scores ? out_block_scores
                                : reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + kHeaderBytes);
    p.hdr = static_cast<WorkspaceHeader *>(workspace);
    p.fault = &p.hdr->fault;
    p.bt_stride = bt_stride;
    p.bs_stride = bs_stride;
    p.num_pages = num_pages;
    p.batch = batch;
    p.seq_limit = static_cast<int>(bt_stride * kPage < max_model_len ? bt_stride * kPage : max_model_len);
    p.total_q = total_q;
    p.kscale = fp8 ? kscale : nullptr;
    if (total_q == 0)
        return MSA_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MSA_ERR_CUDA;
    const int sms = device_sms(dev);
    if (sms <= 0)
        return MSA_ERR_CUDA;
    const bool withhold = test_withhold_pages();
    if (withhold && fp8)
        return MSA_ERR_UNSUPPORTED;
    static std::atomic<bool> attr_done[2][kMaxDevices];
    if (dev >= 0 && dev < kMaxDevices && !attr_done[fp8][dev].load(std::memory_order_acquire)) {
        const cudaError_t e =
            fp8 ? cudaFuncSetAttribute(tc_prefill_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kF8SmemBytes))
                : cudaFuncSetAttribute(tc_prefill_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kP2SmemBytes));
        if (e != cudaSuccess)
            return MSA_ERR_CUDA;
        attr_done[fp8][dev].store(true, std::memory_order_release);
    }
    const bool maps = fp8 ? make_codes_map(&p.kmap, kcache_pool, num_pages * kPage)
                          : make_rows_map(&p.kmap, kcache_pool, num_pages * kPage);
    if (!maps || !make_rows_map(&p.qmap, q, static_cast<int64_t>(total_q) * kHeads))
        return MSA_ERR_CUDA;
    // both kernels: clusters of two CTAs, with programmatic dependent launch
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pair_clusters(dev, sms)));
    cfg.blockDim = dim3(fp8 ? kF8Threads : kP2Threads);
    cfg.dynamicSmemBytes = fp8 ? kF8SmemBytes : kP2SmemBytes;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (fp8)
        return cudaLaunchKernelEx(&cfg, tc_prefill_fp8_kernel, p) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
    if (withhold) {
        if (cudaFuncSetAttribute(tc_prefill_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kP2SmemBytes)) != cudaSuccess)
            return MSA_ERR_CUDA;
        return cudaLaunchKernelEx(&cfg, tc_prefill_pair_kernel<true>, p) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
    }
    return cudaLaunchKernelEx(&cfg, tc_prefill_pair_kernel<false>, p) == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

extern "C" msa_status msa_indexer_prefill_score(const void *q, const int32_t *cu_seqlens_q,
                                                int total_q, const void *kcache_pool,
                                                int64_t num_pages, const int32_t *block_table,
                                                int64_t bt_stride, const int32_t *seq_lens,
                                                int batch, int max_model_len,
                                                float *out_block_scores, void *workspace,
                                                size_t workspace_bytes, void *stream)
{
    if (!out_block_scores)
        return MSA_ERR_INVALID_ARG;
    TcParams p;
    return prefill_score_launch(q, cu_seqlens_q, total_q, kcache_pool, nullptr, num_pages,
                                block_table, bt_stride, seq_lens, batch, max_model_len,
                                out_block_scores, workspace, workspace_bytes,
                                static_cast<cudaStream_t>(stream), &p, false);
}

static msa_status prefill_entry(const void *q, const int32_t *cu_seqlens_q, int total_q,
                                const void *kcache_pool, const float *kscale, int64_t num_pages,
                                const int32_t *block_table, int64_t bt_stride,
                                const int32_t *seq_lens, int batch, int max_model_len, int k,
                                int n_sink, int n_window, int32_t *out_ids, float *out_scores,
                                float *out_block_scores, void *workspace, size_t workspace_bytes,
                                void *stream, bool fp8)
{
    if (!out_ids || !out_scores)
        return MSA_ERR_INVALID_ARG;
    if (k < 1 || n_sink < 0 || n_window < 0)
        return MSA_ERR_INVALID_ARG;
    if (k > MSA_MAX_TOPK)
        return MSA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(n_sink) + n_window > k)
        return MSA_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    TcParams p;
    const msa_status s = prefill_score_launch(q, cu_seqlens_q, total_q, kcache_pool, kscale,
                                              num_pages, block_table, bt_stride, seq_lens, batch,
                                              max_model_len, out_block_scores, workspace,
                                              workspace_bytes, st, &p, fp8);
    if (s != MSA_OK || total_q == 0)
        return s;
    const int64_t rows = static_cast<int64_t>(total_q) * kHeads;
    const bool k16 = kmax_for(k) == 16;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MSA_ERR_CUDA;
    static std::atomic<bool> topk_attr_done[kMaxDevices];
    if (dev >= 0 && dev < kMaxDevices && !topk_attr_done[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(rows_topk_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kTopkSmemBytes)) != cudaSuccess ||
            cudaFuncSetAttribute(rows_topk_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kTopkSmemBytes)) != cudaSuccess)
            return MSA_ERR_CUDA;
        topk_attr_done[dev].store(true, std::memory_order_release);
    }
    // persistent: every warp walks rows a grid's worth of warps apart
    const int64_t ctas = (rows + kTopkRowsPerCta - 1) / kTopkRowsPerCta;
    const int sms = device_sms(dev);
    if (sms <= 0)
        return MSA_ERR_CUDA;
    const int64_t resident = static_cast<int64_t>(sms) * kTopkCtasPerSm;
    cudaLaunchAttribute attr2[1];
    cudaLaunchConfig_t cfg2 = pdl_config(dim3(static_cast<unsigned>(ctas < resident ? ctas : resident)),
                                         dim3(32 * kTopkRowsPerCta), kTopkSmemBytes, st, attr2);
    cudaError_t e = k16 ? cudaLaunchKernelEx(&cfg2, rows_topk_kernel<16>, static_cast<const float *>(p.scores),
                                             p.bs_stride, cu_seqlens_q, seq_lens, batch, total_q,
                                             p.seq_limit, k, n_sink, n_window, out_ids, out_scores,
                                             static_cast<const WorkspaceHeader *>(p.hdr))
                        : cudaLaunchKernelEx(&cfg2, rows_topk_kernel<32>, static_cast<const float *>(p.scores),
                                             p.bs_stride, cu_seqlens_q, seq_lens, batch, total_q,
                                             p.seq_limit, k, n_sink, n_window, out_ids, out_scores,
                                             static_cast<const WorkspaceHeader *>(p.hdr));
    return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

extern "C" msa_status msa_indexer_prefill(const void *q, const int32_t *cu_seqlens_q, int total_q,
                                          const void *kcache_pool, int64_t num_pages,
                                          const int32_t *block_table, int64_t bt_stride,
                                          const int32_t *seq_lens, int batch, int max_model_len,
                                          int k, int n_sink, int n_window, int32_t *out_ids,
                                          float *out_scores, float *out_block_scores,
                                          void *workspace, size_t workspace_bytes, void *stream)
{
    return prefill_entry(q, cu_seqlens_q, total_q, kcache_pool, nullptr, num_pages, block_table,
                         bt_stride, seq_lens, batch, max_model_len, k, n_sink, n_window, out_ids,
                         out_scores, out_block_scores, workspace, workspace_bytes, stream, false);
}

extern "C" msa_status msa_indexer_prefill_fp8(const void *q, const int32_t *cu_seqlens_q,
                                              int total_q, const void *kcache_fp8,
                                              const float *kscale, int64_t num_pages,
                                              const int32_t *block_table, int64_t bt_stride,
                                              const int32_t *seq_lens, int batch,
                                              int max_model_len, int k, int n_sink, int n_window,
                                              int32_t *out_ids, float *out_scores,
                                              float *out_block_scores, void *workspace,
                                              size_t workspace_bytes, void *stream)
{
    return prefill_entry(q, cu_seqlens_q, total_q, kcache_fp8, kscale, num_pages, block_table,
                         bt_stride, seq_lens, batch, max_model_len, k, n_sink, n_window, out_ids,
                         out_scores, out_block_scores, workspace, workspace_bytes, stream, true);
}

extern "C" msa_status msa_indexer_prefill_score_fp8(const void *q, const int32_t *cu_seqlens_q,
                                                    int total_q, const void *kcache_fp8,
                                                    const float *kscale, int64_t num_pages,
                                                    const int32_t *block_table, int64_t bt_stride,
                                                    const int32_t *seq_lens, int batch,
                                                    int max_model_len, float *out_block_scores,
                                                    void *workspace, size_t workspace_bytes,
                                                    void *stream)
{
    if (!out_block_scores)
        return MSA_ERR_INVALID_ARG;
    TcParams p;
    return prefill_score_launch(q, cu_seqlens_q, total_q, kcache_fp8, kscale, num_pages,
                                block_table, bt_stride, seq_lens, batch, max_model_len,
                                out_block_scores, workspace, workspace_bytes,
                                static_cast<cudaStream_t>(stream), &p, true);
}
