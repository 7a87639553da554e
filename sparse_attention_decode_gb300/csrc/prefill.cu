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
// tc_prefill_score_kernel (persistent, one CTA per SM): the product of the
// new tokens' query rows (token x head) with the keys is a dense contraction,
// run on the 5th-generation tensor cores.  Work unit = (tile of 64 new tokens
// of one request, one visible page of that tile); the units of the whole
// batch, in order, are cut into one equal range per CTA (the page counts
// have a closed form), which balances the causal triangle.  Per CTA:
//   warp 0     TMA producer: the tile's 256 query rows (64 KiB, 128B swizzle)
//              and the pages (32 KiB each) through a 4-stage ring;
//   warp 1     owns the TMEM allocation; one thread issues tcgen05.mma
//              (M = 128 rows, N = 128 keys, K = 16) for both 128-row halves
//              of the tile against each page, fp32 accumulators in TMEM,
//              double-buffered across pages (2 x 2 x 128 = 512 columns);
//              (tiles of 32 tokens would allow four buffers but load every
//              page for half as many rows: 1.3x slower when measured)
//   warps 2-9  read their rows' 128 accumulators per page from TMEM and
//              write the masked block max (keys <= the row's position);
//   warp 10    waits, page by page, for the stage to be full and the
//              accumulator buffer to be free, and counts the pages that may
//              be multiplied in a shared word the issuing thread polls.
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

constexpr int kTileTokens = 64;                       // new tokens per work tile
constexpr int kMRows = 128;                           // rows per MMA: 32 tokens x 4 heads
constexpr int kMTiles = kTileTokens * kHeads / kMRows;  // 2
constexpr int kTcStages = 4;
constexpr int kEpiWarps = 4 * kMTiles;                // one per (TMEM lane quarter, M tile)
constexpr int kWaiterWarp = 2 + kEpiWarps;
constexpr int kTcThreads = 32 * (3 + kEpiWarps);
constexpr uint32_t kTmemCols = 512;                   // the whole tensor memory
constexpr int kAccBufs = kTmemCols / (kMTiles * kPage);  // accumulator buffers (pages in flight)
static_assert(kPage % kTileTokens == 0 && kAccBufs >= 2, "tile geometry");
constexpr int kQTileBytes = kMRows * kDim * 2;        // 32 KiB per M tile
constexpr uint32_t kQBytes = kMTiles * kQTileBytes;
constexpr uint32_t kIdesc = umma_idesc_bf16_f32(kMRows, kPage);

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
    int64_t bt_stride;
    int64_t bs_stride;
    int64_t num_pages;
    int batch;
    int seq_limit;
    int total_q;
};

struct TcSmem {
    uint64_t k_full[kTcStages];
    uint64_t k_empty[kTcStages];
    uint64_t q_full;
    uint64_t q_empty;
    uint64_t acc_full[kAccBufs];
    uint64_t acc_empty[kAccBufs];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t ready;  // pages whose operands and accumulator buffer the issuing thread may use
    int abort;
    int b0, t0, j0;  // the range's first unit
    int b1, t1, j1;  // its last unit + 1 page
    long long units;
};

constexpr size_t kTcSmemBytes = 1024 /* alignment slack */ + kQBytes +
                                static_cast<size_t>(kTcStages) * kPageBytes + sizeof(TcSmem);

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

// This CTA's range of work units: [W*g/G, W*(g+1)/G) of the batch's
// (tile, page) units in order.  Run by one warp; writes its first and last
// positions and its unit count.
template <class Ctl>
__device__ void plan_range(const TcParams &p, Ctl *ctl, int lane)
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
    const long long G = gridDim.x, g = blockIdx.x;
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

// The issuing thread's wait for page `need - 1` of its range: the waiter
// warp raises `ready` to n once pages 0 .. n-1 have their stage full and
// their accumulator buffer free.  Two mbarrier waits per page in the issuing
// thread cost it ~500 of the ~1700 cycles a page took; one acquire load of a
// counter that is usually already there leaves it free to issue.
template <class Ctl>
__device__ __forceinline__ bool wait_ready(Ctl *ctl, uint32_t need)
{
    const uint32_t addr = smem_addr(&ctl->ready);
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (ld_acquire_shared_u32(addr) >= need)
            return true;
        if (aborted(ctl))
            return false;
    }
    return false;
}

// The MMAs of pages [j0, je) of one segment, by the issuing thread: per page,
// NMT M tiles of 8 tcgen05.mma each.  NMT = 1 for a tile whose second M tile
// holds no new token (its epilogue writes nothing); the choice is made once
// per segment so the per-page issue path carries no branch.  Returns false
// when a wait ran out.
template <int NMT>
__device__ __forceinline__ bool mma_pages(const TcParams &p, TcSmem *ctl, uint32_t tmem,
                                          uint32_t q_smem, uint32_t k_smem, int j0, int je,
                                          uint32_t &kc, uint32_t &ac)
{
    for (int j = j0; j < je; ++j) {
        const int s = static_cast<int>(kc % kTcStages);
        const int a = static_cast<int>(ac % kAccBufs);
        if (!wait_ready(ctl, kc + 1)) {
            give_up(p, ctl);
            return false;
        }
        tc_fence_after_sync();
        // descriptors as base low words plus byte offsets >> 4: one integer add
        // per operand keeps the single issuing thread ahead of the tensor pipe
        const uint32_t a_lo = umma_desc_lo(q_smem);
        const uint32_t b_lo = umma_desc_lo(k_smem + s * kPageBytes);
        const uint32_t d0 = tmem + static_cast<uint32_t>(a * kMTiles * kPage);
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
#pragma unroll
            for (int ks = 0; ks < kDim / 16; ++ks) {
                const uint32_t off = ((ks >> 2) * kHalfPageBytes + (ks & 3) * 32) >> 4;
                const uint32_t qo = (mt * kQTileBytes) >> 4;
                if (ks == 0)
                    umma_f16<false>(d0 + mt * kPage, a_lo + qo + off, b_lo + off, kIdesc);
                else
                    umma_f16<true>(d0 + mt * kPage, a_lo + qo + off, b_lo + off, kIdesc);
            }
        }
        umma_commit(smem_addr(&ctl->k_empty[s]));
        umma_commit(smem_addr(&ctl->acc_full[a]));
        ++kc;
        ++ac;
    }
    return true;
}

__global__ void __launch_bounds__(kTcThreads, 1) tc_prefill_score_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t q_smem = smem_addr(smem);
    const uint32_t k_smem = q_smem + kQBytes;
    TcSmem *ctl = reinterpret_cast<TcSmem *>(smem + kQBytes + kTcStages * kPageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(smem_addr(&ctl->k_full[s]), 1);
            mbar_init(smem_addr(&ctl->k_empty[s]), 1);
        }
        mbar_init(smem_addr(&ctl->q_full), 1);
        mbar_init(smem_addr(&ctl->q_empty), 1);
        for (int a = 0; a < kAccBufs; ++a) {
            mbar_init(smem_addr(&ctl->acc_full[a]), 1);
            mbar_init(smem_addr(&ctl->acc_empty[a]), kEpiWarps);
        }
        mbar_init(smem_addr(&ctl->mma_done), 1);
        ctl->abort = 0;
        ctl->ready = 0;
        fence_barrier_init();
    }
    griddep_wait();
    griddep_launch_dependents();
    if (warp == 0)
        plan_range(p, ctl, lane);
    __syncthreads();
    const long long units = ctl->units;
    if (units <= 0)
        return;  // uniform: no TMEM taken yet
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl->tmem_base), kTmemCols);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;
    const int sb = ctl->b0, st = ctl->t0, sj = ctl->j0;
    const int eb = ctl->b1, et = ctl->t1, ej = ctl->j1;

    if (warp == 0) {
        // ---------------- producer ----------------
        Cursor c;
        c.load(p, sb, st, sj, eb, et, ej);
        long long left = units;
        uint32_t kc = 0, seg = 0;
        bool ok_run = true;
        while (left > 0 && ok_run) {
            const int je = c.je;
            if (lane == 0) {
                if (seg > 0 && !mbar_wait(smem_addr(&ctl->q_empty), (seg - 1) & 1u)) {
                    give_up(p, ctl);
                    ok_run = false;
                } else {
                    const uint32_t qf = smem_addr(&ctl->q_full);
                    const int row0 = (c.r.c0 + kTileTokens * c.t) * kHeads;
                    mbar_arrive_expect_tx(qf, kQBytes);
#pragma unroll
                    for (int mt = 0; mt < kMTiles; ++mt)
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            tma_load_2d(q_smem + mt * kQTileBytes + h * kHalfPageBytes, &p.qmap, 64 * h,
                                        row0 + mt * kMRows, qf);
                }
            }
            ok_run = __shfl_sync(0xffffffffu, ok_run ? 1 : 0, 0) != 0;
            for (int jb = c.j; jb < je && ok_run; jb += 32) {
                const int jl = jb + lane;
                int page = 0, ok = 0;
                if (jl < je) {
                    page = p.block_table[static_cast<int64_t>(c.b) * p.bt_stride + jl];
                    ok = (page >= 0 && page < p.num_pages) ? 1 : 0;
                    if (!ok)
                        atomicOr(p.fault, MSA_FAULT_PAGE_ID);
                }
                const int cnt = min(32, je - jb);
                for (int i = 0; i < cnt; ++i) {
                    const int pg = __shfl_sync(0xffffffffu, page, i);
                    const int pok = __shfl_sync(0xffffffffu, ok, i);
                    int good = 1;
                    if (lane == 0) {
                        const int s = static_cast<int>(kc % kTcStages);
                        const uint32_t full = smem_addr(&ctl->k_full[s]);
                        if (aborted(ctl) ||
                            (kc >= kTcStages &&
                             !mbar_wait(smem_addr(&ctl->k_empty[s]), ((kc / kTcStages) - 1) & 1u))) {
                            give_up(p, ctl);
                            good = 0;
                        } else if (pok) {
                            const uint32_t dst = k_smem + s * kPageBytes;
                            mbar_arrive_expect_tx(full, kPageBytes);
                            tma_load_2d(dst, &p.kmap, 0, pg * kPage, full);
                            tma_load_2d(dst + kHalfPageBytes, &p.kmap, 64, pg * kPage, full);
                        } else {
                            mbar_arrive(full);  // nothing to load; the epilogue writes -inf
                        }
                    }
                    if (__shfl_sync(0xffffffffu, good, 0) == 0) {
                        ok_run = false;
                        break;
                    }
                    ++kc;
                }
            }
            ++seg;
            left -= je - c.j;
            if (left > 0 && !c.next(p))
                break;
        }
        if (lane == 0) {  // drain: no copy may land after the CTA exits
            for (uint32_t i = kc > kTcStages ? kc - kTcStages : 0; i < kc; ++i)
                if (!mbar_wait(smem_addr(&ctl->k_full[i % kTcStages]), (i / kTcStages) & 1u))
                    give_up(p, ctl);
            if (seg > 0 && !mbar_wait(smem_addr(&ctl->q_full), (seg - 1) & 1u))
                give_up(p, ctl);
        }
    } else if (warp == 1) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            Cursor c;
            c.load(p, sb, st, sj, eb, et, ej);
            long long left = units;
            uint32_t kc = 0, ac = 0, seg = 0;
            bool ok_run = true;
            while (left > 0 && ok_run) {
                const int je = c.je;
                if (!mbar_wait(smem_addr(&ctl->q_full), seg & 1u)) {
                    give_up(p, ctl);
                    break;
                }
                tc_fence_after_sync();
                // M tiles holding at least one of the tile's new tokens
                const int live_tokens = min(kTileTokens, c.r.n - kTileTokens * c.t);
                const int live_mtiles = (live_tokens * kHeads + kMRows - 1) / kMRows;
                ok_run = live_mtiles == kMTiles
                             ? mma_pages<kMTiles>(p, ctl, tmem, q_smem, k_smem, c.j, je, kc, ac)
                             : mma_pages<1>(p, ctl, tmem, q_smem, k_smem, c.j, je, kc, ac);
                umma_commit(smem_addr(&ctl->q_empty));
                ++seg;
                left -= je - c.j;
                if (left > 0 && !c.next(p))
                    break;
            }
            // every MMA issued has completed before TMEM is freed
            umma_commit(smem_addr(&ctl->mma_done));
            if (!mbar_wait(smem_addr(&ctl->mma_done), 0))
                give_up(p, ctl);
        }
        __syncwarp();
    } else if (warp == kWaiterWarp) {
        // ---------------- waiter: page kc may be multiplied ----------------
        // (pages are issued in order; page kc uses stage kc mod S and
        // accumulator buffer kc mod A)
        if (lane == 0) {
            const uint32_t addr = smem_addr(&ctl->ready);
            for (uint32_t kc = 0; kc < static_cast<uint32_t>(units); ++kc) {
                const int s = static_cast<int>(kc % kTcStages);
                const int a = static_cast<int>(kc % kAccBufs);
                if (aborted(ctl) || !mbar_wait(smem_addr(&ctl->k_full[s]), (kc / kTcStages) & 1u) ||
                    (kc >= kAccBufs && !mbar_wait(smem_addr(&ctl->acc_empty[a]), ((kc / kAccBufs) - 1) & 1u))) {
                    give_up(p, ctl);
                    break;
                }
                st_release_shared_u32(addr, kc + 1);
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: TMEM -> block scores ----------------
        const int e = warp - 2;
        const int quarter = warp & 3;        // TMEM lanes this warp may read
        const int mt = e >> 2;               // M tile of this warp
        const int row_in_tile = mt * kMRows + 32 * quarter + lane;  // 0..255
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quarter) << 16) +
                                   static_cast<uint32_t>(mt * kPage);
        const float neg_inf = -__int_as_float(0x7f800000);
        Cursor c;
        c.load(p, sb, st, sj, eb, et, ej);
        long long left = units;
        uint32_t ac = 0;
        bool ok_run = true;
        while (left > 0 && ok_run) {
            const int je = c.je;
            const int tl = kTileTokens * c.t + (row_in_tile >> 2);  // token within the request's new ones
            const int head = row_in_tile & 3;
            const bool live = tl < c.r.n;
            const int pos = c.r.len - c.r.n + tl;
            float *out = p.scores + (static_cast<int64_t>(c.r.c0 + tl) * kHeads + head) * p.bs_stride;
            for (int j = c.j; j < je; ++j) {
                const int a = static_cast<int>(ac % kAccBufs);
                bool ready = !aborted(ctl) && mbar_wait(smem_addr(&ctl->acc_full[a]), (ac / kAccBufs) & 1u);
                ready = __all_sync(0xffffffffu, ready);
                if (!ready) {
                    if (lane == 0)
                        give_up(p, ctl);
                    ok_run = false;
                    break;
                }
                tc_fence_after_sync();
                const int page = p.block_table[static_cast<int64_t>(c.b) * p.bt_stride + j];
                const bool page_ok = page >= 0 && page < p.num_pages;
                const int first_key = j * kPage;
                const bool want = live && first_key <= pos;
                if (page_ok && __any_sync(0xffffffffu, want)) {
                    float mx = neg_inf;
#pragma unroll
                    for (int q4 = 0; q4 < kPage / 32; ++q4) {
                        uint32_t r[32];
                        tmem_ld32(lane_addr + static_cast<uint32_t>(a * kMTiles * kPage + 32 * q4), r);
                        tmem_wait_ld(r);
                        const int lim = pos - (first_key + 32 * q4);  // keys i <= lim are visible
                        if (lim >= 31) {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                mx = fmaxf(mx, __uint_as_float(r[i]));
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                mx = fmaxf(mx, i <= lim ? __uint_as_float(r[i]) : neg_inf);
                        }
                    }
                    if (want)
                        out[j] = mx;
                } else if (!page_ok && want) {
                    out[j] = neg_inf;
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_addr(&ctl->acc_empty[a]));
                ++ac;
            }
            left -= je - c.j;
            if (left > 0 && !c.next(p))
                break;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace msa

#include "prefill_fp8.cuh"
#include "rows_topk.cuh"

namespace msa {

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
    p.fault = &static_cast<WorkspaceHeader *>(workspace)->fault;
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
    static std::atomic<bool> attr_done[2][kMaxDevices];
    if (dev >= 0 && dev < kMaxDevices && !attr_done[fp8][dev].load(std::memory_order_acquire)) {
        const cudaError_t e =
            fp8 ? cudaFuncSetAttribute(tc_prefill_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kF8SmemBytes))
                : cudaFuncSetAttribute(tc_prefill_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kTcSmemBytes));
        if (e != cudaSuccess)
            return MSA_ERR_CUDA;
        attr_done[fp8][dev].store(true, std::memory_order_release);
    }
    const bool maps = fp8 ? make_codes_map(&p.kmap, kcache_pool, num_pages * kPage)
                          : make_rows_map(&p.kmap, kcache_pool, num_pages * kPage);
    if (!maps || !make_rows_map(&p.qmap, q, static_cast<int64_t>(total_q) * kHeads))
        return MSA_ERR_CUDA;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(static_cast<unsigned>(sms)),
                                        dim3(fp8 ? kF8Threads : kTcThreads),
                                        fp8 ? kF8SmemBytes : kTcSmemBytes, st, attr);
    const cudaError_t e = fp8 ? cudaLaunchKernelEx(&cfg, tc_prefill_fp8_kernel, p)
                              : cudaLaunchKernelEx(&cfg, tc_prefill_score_kernel, p);
    return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
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
                                             p.seq_limit, k, n_sink, n_window, out_ids, out_scores)
                        : cudaLaunchKernelEx(&cfg2, rows_topk_kernel<32>, static_cast<const float *>(p.scores),
                                             p.bs_stride, cu_seqlens_q, seq_lens, batch, total_q,
                                             p.seq_limit, k, n_sink, n_window, out_ids, out_scores);
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
