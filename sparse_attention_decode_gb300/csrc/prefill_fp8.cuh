// Prefill scoring on the E4M3 index-K cache (tcgen05, included by prefill.cu).
//
// One tcgen05.mma multiplies operands of one type, so neither the bf16
// query nor the E4M3 keys can enter it as they are.  Both become f16, exactly:
//  * an E4M3 code is exactly an f16 value (cvt.rn.f16x2.e4m3x2);
//  * a query row is scaled by a power of two so its largest |q| lands in
//    [2^13, 2^14) and rounded to f16 (exact for values within 2^-14..2^14 of
//    that maximum: the same treatment as the fp8 decode path).
// Products of f16 values are exact in the fp32 accumulators.  The per-token
// scale multiplies each key's column of the accumulators before the masked
// max, and the row's power of two is undone after it.
//
// Per CTA (persistent, one per SM; the same (tile, page) work split as the
// bf16 kernel):
//   warp 0       TMA producer: the tile's 256 bf16 query rows, and each page's
//                16 KiB of codes (one 128x128-byte box) + 512 B of scales
//                (one bulk copy) into a 3-stage raw ring;
//   warp 2       one thread issues tcgen05.mma (f16, M = 128, N = 128, K = 16)
//                for both M tiles against each converted page (its SM
//                sub-partition holds no converter warp, which would slow the
//                issue);
//   warps 1, 3-5 converters: one key row per thread, E4M3 -> f16 into a
//                3-stage operand ring (the 128-byte swizzle layout of a bf16
//                TMA page), scales into an 8-slot ring;
//   warps 6-21   epilogue, four per TMEM lane quarter (2 M tiles x 2 halves of
//                the quarter's 32 rows): first its 16 query rows to f16 in
//                place (per segment), then per page their scaled, masked
//                block max (sixteen warps of 16 rows: half the per-page
//                work of each, against eight of 32);
//   warp 22      waiter: per page, the converted stage full and the
//                accumulator buffer free, counted in a shared word that the
//                issuing thread polls (as in the bf16 kernel).
// (23 warps: up to six on one SM sub-partition, whose 16K-register file then
// allows 80 registers a thread; the register cap keeps the kernel there.)
#pragma once

namespace msa {

constexpr int kF8RawStages = 3;
constexpr int kF8OpStages = 3;
constexpr int kF8Ring = 8;                   // scale slots, one page each
constexpr int kF8ConvWarps = 4;              // one key row per thread, one warp per SM sub-partition
constexpr int kF8FirstEpiWarp = 2 + kF8ConvWarps;
constexpr int kF8EpiWarps = 16;             // four per TMEM lane quarter: 2 M tiles x 2 row halves
static_assert(kF8EpiWarps == 4 * 2 * kMTiles && kMTiles == 2,
              "the epilogue maps warp e to M tile e / 8 and row half (e / 4) % 2");
constexpr int kF8WaiterWarp = kF8FirstEpiWarp + kF8EpiWarps;
constexpr int kF8Threads = 32 * (kF8WaiterWarp + 1);
constexpr uint32_t kF8RawBytes = kPage * kDim;  // 16 KiB of codes
constexpr uint32_t kF8ScaleBytes = kPage * 4;   // 512 B
constexpr uint32_t kIdescF16 = umma_idesc_f16_f32(kMRows, kPage);

struct F8Smem {
    uint64_t raw_full[kF8RawStages];   // codes + scales landed (TMA bytes)
    uint64_t raw_empty[kF8RawStages];  // converted (converter warps)
    uint64_t op_full[kF8OpStages];     // f16 page written (converter warps)
    uint64_t op_empty[kF8OpStages];    // multiplied (MMA commit)
    uint64_t sc_full[kF8Ring];         // scales copied (converter warps)
    uint64_t sc_empty[kF8Ring];        // scales used (epilogue warps)
    uint64_t q_full;                   // bf16 query tile landed (TMA bytes)
    uint64_t q_conv;                   // query tile converted (epilogue warps)
    uint64_t q_empty;                  // multiplied (MMA commit)
    uint64_t acc_full[kAccBufs];
    uint64_t acc_empty[kAccBufs];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t ready;  // pages the issuing thread may multiply (the waiter warp's count)
    uint32_t epoch;  // the workspace's pass count when this pass started
    int abort;
    int b0, t0, j0;  // the range's first unit
    int b1, t1, j1;  // its last unit + 1 page
    long long units;
};

// Shared memory: query tile | operand ring | raw ring | raw scales | scale ring | control.
constexpr uint32_t kF8OpOff = kQBytes;
constexpr uint32_t kF8RawOff = kF8OpOff + kF8OpStages * kPageBytes;
constexpr uint32_t kF8RawScOff = kF8RawOff + kF8RawStages * kF8RawBytes;
constexpr uint32_t kF8RingOff = kF8RawScOff + kF8RawStages * kF8ScaleBytes;
constexpr uint32_t kF8CtlOff = kF8RingOff + kF8Ring * kF8ScaleBytes;
constexpr size_t kF8SmemBytes = 1024 /* alignment slack */ + kF8CtlOff + sizeof(F8Smem);
static_assert(kF8OpOff % 1024 == 0 && kF8RawOff % 1024 == 0, "swizzled tiles need 1 KiB alignment");

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Four E4M3 codes (byte i -> element i) -> two f16x2 words, exactly.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    lo = e4m3x2_to_f16x2(static_cast<uint16_t>(w & 0xffffu));
    hi = e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16));
}

// Two fp32 products in one instruction (packed f32x2 multiply, sm_100+).
__device__ __forceinline__ void mul2(float a0, float a1, float b0, float b1, float &d0, float &d1)
{
    uint64_t a, b, d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}

// Scaled maximum over one 16x256b.x4 TMEM load (tmem_ld16x256b_x4): r holds
// rows g and g + 8 of a 16-row block at the 8 columns 8 i + 2 c + {0, 1} of a
// 32-column chunk (g = lane / 4, c = lane % 4); sc points at the chunk's
// per-key scales as pairs.  Folds the products of row g into ma and of row
// g + 8 into mb; with MASK, column kbase + k counts for row g only if
// kbase + k <= lim_a (row g + 8: lim_b), the causal edge.
template <bool MASK>
__device__ __forceinline__ void scaled_max_frag(const uint32_t (&r)[16], const float2 *sc, int c, int kbase,
                                                int lim_a, int lim_b, float &ma, float &mb)
{
    const float neg_inf = -__int_as_float(0x7f800000);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 si = sc[4 * i + c];
        float v0, v1, v2, v3;
        mul2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]), si.x, si.y, v0, v1);
        mul2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]), si.x, si.y, v2, v3);
        if (MASK) {
            const int k0 = kbase + 8 * i + 2 * c;
            v0 = k0 <= lim_a ? v0 : neg_inf;
            v1 = k0 + 1 <= lim_a ? v1 : neg_inf;
            v2 = k0 <= lim_b ? v2 : neg_inf;
            v3 = k0 + 1 <= lim_b ? v3 : neg_inf;
        }
        ma = fmaxf(ma, fmaxf(v0, v1));
        mb = fmaxf(mb, fmaxf(v2, v3));
    }
}

// bf16 pair -> f32 pair.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 23 warps leave six on three SM sub-partitions, whose 16K registers then
// hold 80 a thread (a multiple of 8); the cap keeps the launch inside that.
constexpr int kF8MaxRegs = (16384 / (32 * ((kF8Threads / 32 + 3) / 4))) & ~7;
static_assert(kF8MaxRegs >= 64, "too many warps for the register file");

__global__ void __maxnreg__(kF8MaxRegs) tc_prefill_fp8_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t q_smem = smem_addr(smem);
    const uint32_t op_smem = q_smem + kF8OpOff;
    const uint32_t raw_smem = q_smem + kF8RawOff;
    const uint32_t rawsc_smem = q_smem + kF8RawScOff;
    float *ring = reinterpret_cast<float *>(smem + kF8RingOff);
    F8Smem *ctl = reinterpret_cast<F8Smem *>(smem + kF8CtlOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kF8RawStages; ++s) {
            mbar_init(smem_addr(&ctl->raw_full[s]), 1);
            mbar_init(smem_addr(&ctl->raw_empty[s]), kF8ConvWarps);
        }
        for (int s = 0; s < kF8OpStages; ++s) {
            mbar_init(smem_addr(&ctl->op_full[s]), kF8ConvWarps);
            mbar_init(smem_addr(&ctl->op_empty[s]), 1);
        }
        for (int s = 0; s < kF8Ring; ++s) {
            mbar_init(smem_addr(&ctl->sc_full[s]), kF8ConvWarps);
            mbar_init(smem_addr(&ctl->sc_empty[s]), kF8EpiWarps);
        }
        mbar_init(smem_addr(&ctl->q_full), 1);
        mbar_init(smem_addr(&ctl->q_conv), kF8EpiWarps);
        mbar_init(smem_addr(&ctl->q_empty), 1);
        for (int a = 0; a < kAccBufs; ++a) {
            mbar_init(smem_addr(&ctl->acc_full[a]), 1);
            mbar_init(smem_addr(&ctl->acc_empty[a]), kF8EpiWarps);
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
    if (warp == 0)
        plan_range(p, ctl, lane, gridDim.x, blockIdx.x);
    __syncthreads();
    const long long units = ctl->units;
    if (units <= 0) {
        if (threadIdx.x == 0)  // uniform: no TMEM taken yet
            pass_end(p, ctl);
        return;
    }
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
        // ---------------- producer: query tiles and raw pages ----------------
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
                        const int s = static_cast<int>(kc % kF8RawStages);
                        const uint32_t full = smem_addr(&ctl->raw_full[s]);
                        if (aborted(ctl) ||
                            (kc >= kF8RawStages &&
                             !mbar_wait(smem_addr(&ctl->raw_empty[s]), ((kc / kF8RawStages) - 1) & 1u))) {
                            give_up(p, ctl);
                            good = 0;
                        } else if (pok) {
                            mbar_arrive_expect_tx(full, kF8RawBytes + kF8ScaleBytes);
                            tma_load_2d(raw_smem + s * kF8RawBytes, &p.kmap, 0, pg * kPage, full);
                            bulk_load_hint(rawsc_smem + s * kF8ScaleBytes,
                                           p.kscale + static_cast<size_t>(pg) * kPage, kF8ScaleBytes,
                                           full, l2_evict_first_policy());
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
            for (uint32_t i = kc > kF8RawStages ? kc - kF8RawStages : 0; i < kc; ++i)
                if (!mbar_wait(smem_addr(&ctl->raw_full[i % kF8RawStages]), (i / kF8RawStages) & 1u))
                    give_up(p, ctl);
            if (seg > 0 && !mbar_wait(smem_addr(&ctl->q_full), (seg - 1) & 1u))
                give_up(p, ctl);
        }
    } else if (warp == 2) {
        // ---------------- MMA issue (one thread) ----------------
        if (lane == 0) {
            Cursor c;
            c.load(p, sb, st, sj, eb, et, ej);
            long long left = units;
            uint32_t kc = 0, ac = 0, seg = 0;
            bool ok_run = true;
            while (left > 0 && ok_run) {
                const int je = c.je;
                if (!mbar_wait(smem_addr(&ctl->q_conv), seg & 1u)) {
                    give_up(p, ctl);
                    break;
                }
                tc_fence_after_sync();
                const int live_tokens = min(kTileTokens, c.r.n - kTileTokens * c.t);
                const int nmt = (live_tokens * kHeads + kMRows - 1) / kMRows;
                for (int j = c.j; j < je; ++j) {
                    const int s = static_cast<int>(kc % kF8OpStages);
                    const int a = static_cast<int>(ac % kAccBufs);
                    if (!wait_ready(ctl, kc + 1)) {
                        give_up(p, ctl);
                        ok_run = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t a_lo = umma_desc_lo(q_smem);
                    const uint32_t b_lo = umma_desc_lo(op_smem + s * kPageBytes);
                    const uint32_t d0 = tmem + static_cast<uint32_t>(a * kMTiles * kPage);
#pragma unroll
                    for (int mt = 0; mt < kMTiles; ++mt) {
                        if (mt < nmt) {
#pragma unroll
                            for (int ks = 0; ks < kDim / 16; ++ks) {
                                const uint32_t off = ((ks >> 2) * kHalfPageBytes + (ks & 3) * 32) >> 4;
                                const uint32_t qo = (mt * kQTileBytes) >> 4;
                                if (ks == 0)
                                    umma_f16<false>(d0 + mt * kPage, a_lo + qo + off, b_lo + off, kIdescF16);
                                else
                                    umma_f16<true>(d0 + mt * kPage, a_lo + qo + off, b_lo + off, kIdescF16);
                            }
                        }
                    }
                    umma_commit(smem_addr(&ctl->op_empty[s]));
                    umma_commit(smem_addr(&ctl->acc_full[a]));
                    ++kc;
                    ++ac;
                }
                umma_commit(smem_addr(&ctl->q_empty));
                ++seg;
                left -= je - c.j;
                if (left > 0 && !c.next(p))
                    break;
            }
            umma_commit(smem_addr(&ctl->mma_done));
            if (!mbar_wait(smem_addr(&ctl->mma_done), 0))
                give_up(p, ctl);
        }
        __syncwarp();
    } else if (warp < kF8FirstEpiWarp) {
        // ---------------- converters: E4M3 page -> f16 operand ----------------
        const int kr0 = 32 * (warp == 1 ? 0 : warp - 2) + lane;  // this thread's key row
        for (long long pc = 0; pc < units; ++pc) {
            const uint32_t u = static_cast<uint32_t>(pc);
            const int rs = static_cast<int>(u % kF8RawStages);
            const int os = static_cast<int>(u % kF8OpStages);
            const int slot = static_cast<int>(u % kF8Ring);
            bool ready = !aborted(ctl) && mbar_wait(smem_addr(&ctl->raw_full[rs]), (u / kF8RawStages) & 1u);
            ready = ready && (u < kF8OpStages ||
                              mbar_wait(smem_addr(&ctl->op_empty[os]), ((u / kF8OpStages) - 1) & 1u));
            ready = ready && (u < kF8Ring ||
                              mbar_wait(smem_addr(&ctl->sc_empty[slot]), ((u / kF8Ring) - 1) & 1u));
            ready = __all_sync(0xffffffffu, ready);
            if (!ready) {
                if (lane == 0)
                    give_up(p, ctl);
                break;
            }
            {
                const int kr = kr0;
                const uint32_t swz = static_cast<uint32_t>(kr & 7);
                const uint32_t src = raw_smem + rs * kF8RawBytes + static_cast<uint32_t>(kr) * 128;
                const uint32_t dst = op_smem + os * kPageBytes + static_cast<uint32_t>(kr) * 128;
#pragma unroll
                for (int cch = 0; cch < 8; ++cch) {
                    // codes of dims 16 cch .. 16 cch + 15 -> f16 chunks 2 cch, 2 cch + 1
                    // (dims 16 cch + 8 i .. + 7) of half cch / 4
                    const uint4 v = lds128(src + ((static_cast<uint32_t>(cch) ^ swz) << 4));
                    uint4 f0, f1;
                    e4m3x4_to_f16(v.x, f0.x, f0.y);
                    e4m3x4_to_f16(v.y, f0.z, f0.w);
                    e4m3x4_to_f16(v.z, f1.x, f1.y);
                    e4m3x4_to_f16(v.w, f1.z, f1.w);
                    const uint32_t half = static_cast<uint32_t>(cch >> 2) * kHalfPageBytes;
                    const uint32_t c0 = static_cast<uint32_t>((cch & 3) * 2);
                    sts128(dst + half + ((c0 ^ swz) << 4), f0);
                    sts128(dst + half + (((c0 + 1) ^ swz) << 4), f1);
                }
                ring[slot * kPage + kr] = reinterpret_cast<const float *>(smem + kF8RawScOff)[rs * kPage + kr];
            }
            fence_proxy_async_smem();  // the f16 page is read by the tensor cores
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_addr(&ctl->op_full[os]));
                mbar_arrive(smem_addr(&ctl->raw_empty[rs]));
                mbar_arrive(smem_addr(&ctl->sc_full[slot]));
            }
        }
    } else if (warp == kF8WaiterWarp) {
        // ---------------- waiter: page kc may be multiplied ----------------
        if (lane == 0) {
            const uint32_t addr = smem_addr(&ctl->ready);
            for (uint32_t kc = 0; kc < static_cast<uint32_t>(units); ++kc) {
                const int s = static_cast<int>(kc % kF8OpStages);
                const int a = static_cast<int>(kc % kAccBufs);
                if (aborted(ctl) || !mbar_wait(smem_addr(&ctl->op_full[s]), (kc / kF8OpStages) & 1u) ||
                    (kc >= kAccBufs && !mbar_wait(smem_addr(&ctl->acc_empty[a]), ((kc / kAccBufs) - 1) & 1u))) {
                    give_up(p, ctl);
                    break;
                }
                st_release_shared_u32(addr, kc + 1);
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: query row to f16, then block scores ----------------
        const int e = warp - kF8FirstEpiWarp;
        const int quarter = warp & 3;  // TMEM lanes this warp may read
        const int mt = e >> 3;         // M tile of this warp
        const int hh = (e >> 2) & 1;   // its 16 of the quarter's 32 rows
        const int row0 = 32 * quarter + 16 * hh;  // first of those rows within the M tile
        // Query conversion: two lanes per row, each half of the row's 128 dims.
        const int rr = row0 + (lane & 15);
        const uint32_t qrow = q_smem + static_cast<uint32_t>(mt) * kQTileBytes + static_cast<uint32_t>(rr) * 128 +
                              static_cast<uint32_t>(lane >> 4) * kHalfPageBytes;
        const uint32_t qswz = static_cast<uint32_t>(rr & 7);
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(row0) << 16) + static_cast<uint32_t>(mt * kPage);
        const float neg_inf = -__int_as_float(0x7f800000);
        Cursor c;
        c.load(p, sb, st, sj, eb, et, ej);
        long long left = units;
        uint32_t ac = 0, seg = 0;
        bool ok_run = true;
        while (left > 0 && ok_run) {
            const int je = c.je;
            // this row of the segment's query tile to f16, scaled by 2^sh
            bool qready = !aborted(ctl) && mbar_wait(smem_addr(&ctl->q_full), seg & 1u);
            qready = __all_sync(0xffffffffu, qready);
            if (!qready) {
                if (lane == 0)
                    give_up(p, ctl);
                break;
            }
            float amax = 0.0f;  // pass 1: the row's largest |q| (this lane's half, then both)
#pragma unroll 4
            for (int i = 0; i < 8; ++i) {
                const uint4 v = lds128(qrow + ((static_cast<uint32_t>(i) ^ qswz) << 4));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[t])), fabsf(bf16_hi(w[t]))));
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
            int ex = 0;
            if (amax > 0.0f)
                frexpf(amax, &ex);  // amax = m * 2^ex, m in [0.5, 1)
            const int sh = max(-100, min(100, 14 - ex));
            const float up = __int_as_float((127 + sh) << 23);
            const float inv_row = __int_as_float((127 - sh) << 23);
#pragma unroll 4
            for (int i = 0; i < 8; ++i) {  // pass 2: scale, round to f16, write back in place
                const uint32_t addr = qrow + ((static_cast<uint32_t>(i) ^ qswz) << 4);
                const uint4 v = lds128(addr);
                uint4 o;
                o.x = f32x2_to_f16x2(bf16_lo(v.x) * up, bf16_hi(v.x) * up);
                o.y = f32x2_to_f16x2(bf16_lo(v.y) * up, bf16_hi(v.y) * up);
                o.z = f32x2_to_f16x2(bf16_lo(v.z) * up, bf16_hi(v.z) * up);
                o.w = f32x2_to_f16x2(bf16_lo(v.w) * up, bf16_hi(v.w) * up);
                sts128(addr, o);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&ctl->q_conv));

            // Per page the accumulator is read in the mma-fragment layout: lane
            // (g, cq) = (lane / 4, lane % 4) holds rows g and g + 8 of the warp's
            // 16 at the 32 key columns 8 i + 2 cq + {0, 1}, so it needs only
            // those columns' scales.  After the quad's max, lane (g, 0) writes
            // row g and lane (g, 1) row g + 8.
            const int g = lane >> 2, cq = lane & 3;
            const int my_local = g + 8 * (cq & 1);  // the row this lane writes, of the warp's 16
            const float my_inv = __shfl_sync(0xffffffffu, inv_row, my_local);
            const int my_rr = row0 + my_local;
            const int tl = kTileTokens * c.t + ((mt * kMRows + my_rr) >> 2);  // token within the new ones
            const bool live = cq < 2 && tl < c.r.n;
            const int pos = c.r.len - c.r.n + tl;
            float *out =
                p.scores + (static_cast<int64_t>(c.r.c0 + tl) * kHeads + (my_rr & 3)) * p.bs_stride;
            const int pos_lo = c.r.len - c.r.n + kTileTokens * c.t + (mt * kMRows + row0) / 4;
            const int pos_q = pos_lo + (g >> 2);  // rows g and g + 8 are the tokens at pos_q, pos_q + 2
            // the block-table entry of the next page is fetched while this one is
            // reduced: a global load on each page's critical path otherwise
            const int32_t *bt_row = p.block_table + static_cast<int64_t>(c.b) * p.bt_stride;
            int page_next = c.j < je ? __ldg(bt_row + c.j) : 0;
            for (int j = c.j; j < je; ++j) {
                const int page = page_next;
                if (j + 1 < je)
                    page_next = __ldg(bt_row + j + 1);
                const int a = static_cast<int>(ac % kAccBufs);
                const int slot = static_cast<int>(ac % kF8Ring);
                bool ready = !aborted(ctl) &&
                             mbar_wait(smem_addr(&ctl->acc_full[a]), (ac / kAccBufs) & 1u) &&
                             mbar_wait(smem_addr(&ctl->sc_full[slot]), (ac / kF8Ring) & 1u);
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
                const bool want = live && first_key <= pos;
                if (page_ok && __any_sync(0xffffffffu, want)) {
                    const float2 *sc2 = reinterpret_cast<const float2 *>(ring + slot * kPage);
                    const uint32_t acc = lane_addr + static_cast<uint32_t>(a * kMTiles * kPage);
                    // the page fully visible to every row of the warp, or its causal edge
                    const bool full = pos_lo >= first_key + kPage - 1;
                    const int l0 = pos_q - first_key;
                    float ma = neg_inf, mb = neg_inf;
                    // 4 loads of 16 rows x 32 columns, two in flight
                    uint32_t ra[16], rb[16];
                    tmem_ld16x256b_x4(acc, ra);
                    tmem_ld16x256b_x4(acc + 32, rb);
#pragma unroll
                    for (int cp = 0; cp < kPage / 64; ++cp) {
                        tmem_wait_ld(ra);
                        tmem_regs_ready(rb);
                        const int c0 = 64 * cp;
                        if (full)
                            scaled_max_frag<false>(ra, sc2 + c0 / 2, cq, c0, 0, 0, ma, mb);
                        else
                            scaled_max_frag<true>(ra, sc2 + c0 / 2, cq, c0, l0, l0 + 2, ma, mb);
                        if (cp + 1 < kPage / 64)
                            tmem_ld16x256b_x4(acc + c0 + 64, ra);
                        if (full)
                            scaled_max_frag<false>(rb, sc2 + c0 / 2 + 16, cq, c0 + 32, 0, 0, ma, mb);
                        else
                            scaled_max_frag<true>(rb, sc2 + c0 / 2 + 16, cq, c0 + 32, l0, l0 + 2, ma, mb);
                        if (cp + 1 < kPage / 64)
                            tmem_ld16x256b_x4(acc + c0 + 96, rb);
                    }
                    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
                    ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
                    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
                    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
                    const float mx = (cq & 1) ? mb : ma;
                    if (want)
                        out[j] = mx * my_inv;
                } else if (!page_ok && want) {
                    out[j] = neg_inf;
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_addr(&ctl->acc_empty[a]));
                    mbar_arrive(smem_addr(&ctl->sc_empty[slot]));
                }
                ++ac;
            }
            ++seg;
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
    if (threadIdx.x == 0)
        pass_end(p, ctl);
}

}  // namespace msa
