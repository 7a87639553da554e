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
// The bf16 kernel's pairing (tc_prefill_pair_kernel): clusters of two CTAs
// multiplying as one (cta_group::2), a tile's 256 query rows split 128 / 128,
// its pages taken two at a time (the even CTA holds the first page of each
// pair, the odd CTA the second), one thread of the even CTA issuing 8 MMAs of
// M = 256 x N = 256 x K = 16 per pair into each CTA's TMEM (two accumulator
// buffers of 256 columns).  Per CTA, 23 warps:
//   warp 0       TMA producer: its 128 bf16 query rows at each tile (two
//                tiles' rows resident), and per pair of pages its page's
//                16 KiB of codes (one 128x128-byte box) plus both pages' 512 B
//                of scales into a 3-stage raw ring;
//   warp 1       TMEM allocation (both CTAs, collectively); even CTA: the
//                issuing thread; odd CTA: a thread that tells the even CTA
//                its query rows and each converted page are ready;
//   warp 2       even CTA: the waiter (both CTAs' converted pages and a free
//                accumulator buffer, counted in a shared word that the issuing
//                thread polls);
//   warps 3-6    converters, a row a lane: at each tile the query rows to f16
//                in place (a power of two per row), per pair the page to f16
//                in the operand layout (the 128-byte swizzle layout of a bf16
//                TMA page, 3 stages) and both pages' scales into an 8-slot
//                ring;
//   warps 7-22   epilogue, four per TMEM lane quarter (the pair's first or
//                second page x the quarter's first or second 16 rows): per
//                pair its 16 rows x 128 columns in the mma-fragment layout
//                (tcgen05.ld 16x256b), each lane scaling its 32 key columns,
//                the masked max and the row's power of two undone.
// (23 warps: up to six on one SM sub-partition, whose 16K-register file then
// allows 80 registers a thread; the register cap keeps the kernel there.  At
// 80 registers the epilogue cannot hold a row's 128 accumulators, so it hands
// the buffer back after its max, unlike the bf16 kernel.)  Against the
// earlier single-CTA form (M = 128 x N = 128 MMAs, whose issuing thread took
// ~1480 cycles a page for 1024 of tensor work) the pair halves the MMAs per
// unit of work; a non-blocking test before each wait on a phase that has
// most likely completed saves the ~250 cycles a polling wait costs even then.
#pragma once

namespace msa {

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

constexpr int kF8OpStages = 3;                 // f16 operand stages, one page each
constexpr int kF8RawStages = 3;                // raw stages: a page's codes + both pages' scales
constexpr int kF8Ring = 8;                     // scale slots: both pages' 256 scales each
constexpr int kF8QBufs = 2;                    // a tile's query rows load while the previous is used
constexpr int kF8AccBufs = 2;
constexpr uint32_t kF8TmemCols = kF8AccBufs * 2 * kPage;  // 512
constexpr uint32_t kF8QBytes = kMRows * kDim * 2;          // 32 KiB: 128 query rows
constexpr uint32_t kF8QHalf = kF8QBytes / 2;               // 128 rows x 64 dims
constexpr uint32_t kF8RawBytes = kPage * kDim;             // 16 KiB of codes
constexpr uint32_t kF8PairScales = 2 * kPage;              // floats: both pages' scales
constexpr uint32_t kF8Idesc = umma_idesc_f16_f32(2 * kMRows, 2 * kPage);
constexpr int kF8WaiterWarp = 2;
constexpr int kF8FirstConv = 3;
constexpr int kF8ConvWarps = 4;
constexpr int kF8FirstEpi = kF8FirstConv + kF8ConvWarps;  // 7
constexpr int kF8EpiWarps = 16;
constexpr int kF8Threads = 32 * (kF8FirstEpi + kF8EpiWarps);  // 736
// 23 warps leave six on three SM sub-partitions, whose 16K registers then
// hold 80 a thread (a multiple of 8); the cap keeps the launch inside that.
constexpr int kF8MaxRegs = (16384 / (32 * ((kF8Threads / 32 + 3) / 4))) & ~7;
static_assert(kF8MaxRegs >= 64, "too many warps for the register file");
static_assert(kMRows == 32 * kF8ConvWarps && kPage == 32 * kF8ConvWarps, "a row a converter lane");

struct F8Smem {
    uint64_t raw_full[kF8RawStages];
    uint64_t raw_empty[kF8RawStages];
    uint64_t op_full[kF8OpStages];
    uint64_t op_peer[kF8OpStages];
    uint64_t op_empty[kF8OpStages];
    uint64_t sc_full[kF8Ring];
    uint64_t sc_empty[kF8Ring];
    uint64_t q_full[kF8QBufs];
    uint64_t q_conv[kF8QBufs];
    uint64_t q_peer[kF8QBufs];
    uint64_t q_empty[kF8QBufs];
    uint64_t inv_free[kF8QBufs];
    uint64_t acc_full[kF8AccBufs];
    uint64_t acc_empty[kF8AccBufs];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t ready;
    uint32_t epoch;
    int abort;
    float inv_row[kF8QBufs][kMRows];
    UnitRange rng[2];
};

constexpr uint32_t kF8OpOff = kF8QBufs * kF8QBytes;
constexpr uint32_t kF8RawOff = kF8OpOff + kF8OpStages * kPageBytes;
constexpr uint32_t kF8RawScOff = kF8RawOff + kF8RawStages * kF8RawBytes;
constexpr uint32_t kF8RingOff = kF8RawScOff + kF8RawStages * kF8PairScales * 4;
constexpr uint32_t kF8CtlOff = kF8RingOff + kF8Ring * kF8PairScales * 4;
constexpr size_t kF8SmemBytes = 1024 + kF8CtlOff + sizeof(F8Smem);
static_assert(kF8OpOff % 1024 == 0 && kF8RawOff % 1024 == 0, "swizzled tiles need 1 KiB alignment");
static_assert(kF8RawScOff % 16 == 0 && kF8RingOff % 16 == 0 && kF8CtlOff % 16 == 0, "16-byte alignment");
static_assert(kF8SmemBytes <= 227 * 1024, "shared memory per CTA");

// A wait on a phase that has most likely completed already: one
// non-blocking test first, the bounded polling wait only if it has not.
__device__ __forceinline__ bool bar_wait_test(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n"
        "  .reg .pred p;\n"
        "  mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "  selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0 || mbar_wait(bar, parity);
}

__global__ void __maxnreg__(kF8MaxRegs) tc_prefill_fp8_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t q_smem = smem_addr(smem);
    const uint32_t op_smem = q_smem + kF8OpOff;
    const uint32_t raw_smem = q_smem + kF8RawOff;
    const uint32_t rawsc_smem = q_smem + kF8RawScOff;
    const float *rawsc = reinterpret_cast<const float *>(smem + kF8RawScOff);
    float *ring = reinterpret_cast<float *>(smem + kF8RingOff);
    F8Smem *ctl = reinterpret_cast<F8Smem *>(smem + kF8CtlOff);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < kF8RawStages; ++s) {
            mbar_init(smem_addr(&ctl->raw_full[s]), 1);
            mbar_init(smem_addr(&ctl->raw_empty[s]), kF8ConvWarps);
        }
        for (int s = 0; s < kF8OpStages; ++s) {
            mbar_init(smem_addr(&ctl->op_full[s]), kF8ConvWarps);
            mbar_init(smem_addr(&ctl->op_peer[s]), 1);
            mbar_init(smem_addr(&ctl->op_empty[s]), 1);
        }
        for (int s = 0; s < kF8Ring; ++s) {
            mbar_init(smem_addr(&ctl->sc_full[s]), kF8ConvWarps);
            mbar_init(smem_addr(&ctl->sc_empty[s]), kF8EpiWarps);
        }
        for (int b = 0; b < kF8QBufs; ++b) {
            mbar_init(smem_addr(&ctl->q_full[b]), 1);
            mbar_init(smem_addr(&ctl->q_conv[b]), kF8ConvWarps);
            mbar_init(smem_addr(&ctl->q_peer[b]), 1);
            mbar_init(smem_addr(&ctl->q_empty[b]), 1);
            mbar_init(smem_addr(&ctl->inv_free[b]), kF8EpiWarps);
        }
        for (int a = 0; a < kF8AccBufs; ++a) {
            mbar_init(smem_addr(&ctl->acc_full[a]), 1);
            mbar_init(smem_addr(&ctl->acc_empty[a]), 2 * kF8EpiWarps);
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
    cluster_sync_all();
    if (ctl->rng[0].units + ctl->rng[1].units <= 0) {
        if (threadIdx.x == 0)
            pass_end(p, ctl);
        return;
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(&ctl->tmem_base), kF8TmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ctl->tmem_base;

    if (warp == 0) {
        // ---------------- producer (both CTAs) ----------------
        SegWalk w;
        bool more = w.start(p, ctl->rng);
        const SegWalk &c = w;
        uint32_t gc = 0, seg = 0;
        bool ok_run = true;
        while (more && ok_run) {
            const int je = c.je;
            if (lane == 0) {
                const int qb = static_cast<int>(seg % kF8QBufs);
                if (seg >= kF8QBufs &&
                    !mbar_wait(smem_addr(&ctl->q_empty[qb]), ((seg / kF8QBufs) - 1) & 1u)) {
                    give_up(p, ctl);
                    ok_run = false;
                } else {
                    const uint32_t qf = smem_addr(&ctl->q_full[qb]);
                    const uint32_t qdst = q_smem + static_cast<uint32_t>(qb) * kF8QBytes;
                    const int row0 = (c.r.c0 + kTileTokens * c.t) * kHeads + kMRows * static_cast<int>(rank);
                    mbar_arrive_expect_tx(qf, kF8QBytes);
                    tma_load_2d(qdst, &p.qmap, 0, row0, qf);
                    tma_load_2d(qdst + kF8QHalf, &p.qmap, 64, row0, qf);
                }
            }
            ok_run = __shfl_sync(0xffffffffu, ok_run ? 1 : 0, 0) != 0;
            const int ng = pairs_of(c.j, je);
            for (int gb = 0; gb < ng && ok_run; gb += 32) {
                const int gl = gb + lane;
                const int j0 = c.j + 2 * gl;
                int pg0 = 0, ok0 = 0, pg1 = 0, ok1 = 0;
                if (gl < ng) {
                    pg0 = p.block_table[static_cast<int64_t>(c.b) * p.bt_stride + j0];
                    ok0 = (pg0 >= 0 && pg0 < p.num_pages) ? 1 : 0;
                    if (j0 + 1 < je) {
                        pg1 = p.block_table[static_cast<int64_t>(c.b) * p.bt_stride + j0 + 1];
                        ok1 = (pg1 >= 0 && pg1 < p.num_pages) ? 1 : 0;
                    }
                    if ((!ok0 || (j0 + 1 < je && !ok1)) && rank == 0)
                        atomicOr(p.fault, MSA_FAULT_PAGE_ID);
                }
                const int cnt = min(32, ng - gb);
                for (int i = 0; i < cnt; ++i) {
                    const int q0 = __shfl_sync(0xffffffffu, pg0, i);
                    const int k0 = __shfl_sync(0xffffffffu, ok0, i);
                    const int q1 = __shfl_sync(0xffffffffu, pg1, i);
                    const int k1 = __shfl_sync(0xffffffffu, ok1, i);
                    int good = 1;
                    if (lane == 0) {
                        const int s = static_cast<int>(gc % kF8RawStages);
                        const uint32_t full = smem_addr(&ctl->raw_full[s]);
                        if (aborted(ctl) ||
                            (gc >= kF8RawStages &&
                             !mbar_wait(smem_addr(&ctl->raw_empty[s]), ((gc / kF8RawStages) - 1) & 1u))) {
                            give_up(p, ctl);
                            good = 0;
                        } else {
                            const int mine = rank == 0 ? q0 : q1;
                            const int mine_ok = rank == 0 ? k0 : k1;
                            const uint32_t bytes = (mine_ok ? kF8RawBytes : 0u) + (k0 ? kPage * 4u : 0u) +
                                                   (k1 ? kPage * 4u : 0u);
                            if (bytes == 0) {
                                mbar_arrive(full);
                            } else {
                                mbar_arrive_expect_tx(full, bytes);
                                if (mine_ok)
                                    tma_load_2d(raw_smem + s * kF8RawBytes, &p.kmap, 0, mine * kPage, full);
                                const uint32_t scd = rawsc_smem + s * kF8PairScales * 4;
                                if (k0)
                                    bulk_load_hint(scd, p.kscale + static_cast<size_t>(q0) * kPage, kPage * 4,
                                                   full, l2_evict_first_policy());
                                if (k1)
                                    bulk_load_hint(scd + kPage * 4, p.kscale + static_cast<size_t>(q1) * kPage,
                                                   kPage * 4, full, l2_evict_first_policy());
                            }
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
        if (lane == 0) {
            for (uint32_t i = gc > kF8RawStages ? gc - kF8RawStages : 0; i < gc; ++i)
                if (!mbar_wait(smem_addr(&ctl->raw_full[i % kF8RawStages]), (i / kF8RawStages) & 1u))
                    give_up(p, ctl);
            for (uint32_t i = seg > kF8QBufs ? seg - kF8QBufs : 0; i < seg; ++i)
                if (!mbar_wait(smem_addr(&ctl->q_full[i % kF8QBufs]), (i / kF8QBufs) & 1u))
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
                while (more && ok_run) {
                    const int je = c.je;
                    const int qb = static_cast<int>(seg % kF8QBufs);
                    const uint32_t qph = (seg / kF8QBufs) & 1u;
                    if (!mbar_wait(smem_addr(&ctl->q_conv[qb]), qph) || !mbar_wait(smem_addr(&ctl->q_peer[qb]), qph)) {
                        give_up(p, ctl);
                        break;
                    }
                    const uint32_t a_lo = umma_desc_lo(q_smem + static_cast<uint32_t>(qb) * kF8QBytes);
                    const int ng = pairs_of(c.j, je);
                    for (int g = 0; g < ng; ++g) {
                        const int s = static_cast<int>(gc % kF8OpStages);
                        const int a = static_cast<int>(gc % kF8AccBufs);
                        if (!wait_ready(ctl, gc + 1)) {
                            give_up(p, ctl);
                            ok_run = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t b_lo = umma_desc_lo(op_smem + s * kPageBytes);
                        const uint32_t d = tmem + static_cast<uint32_t>(a * 2 * kPage);
#pragma unroll
                        for (int ks = 0; ks < kDim / 16; ++ks) {
                            const uint32_t qo = ((ks >> 2) * kF8QHalf + (ks & 3) * 32) >> 4;
                            const uint32_t ko = ((ks >> 2) * kHalfPageBytes + (ks & 3) * 32) >> 4;
                            if (ks == 0)
                                umma_pair_f16<false>(d, a_lo + qo, b_lo + ko, kF8Idesc);
                            else
                                umma_pair_f16<true>(d, a_lo + qo, b_lo + ko, kF8Idesc);
                        }
                        umma_commit_pair(smem_addr(&ctl->op_empty[s]));
                        umma_commit_pair(smem_addr(&ctl->acc_full[a]));
                        ++gc;
                    }
                    umma_commit_pair(smem_addr(&ctl->q_empty[qb]));
                    ++seg;
                    more = w.next(p, ctl->rng);
                }
                umma_commit_pair(smem_addr(&ctl->mma_done));
            } else {
                while (more && ok_run) {
                    const int je = c.je;
                    const int qb = static_cast<int>(seg % kF8QBufs);
                    if (!mbar_wait(smem_addr(&ctl->q_conv[qb]), (seg / kF8QBufs) & 1u)) {
                        give_up(p, ctl);
                        break;
                    }
                    mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->q_peer[qb]), 0));
                    const int ng = pairs_of(c.j, je);
                    for (int g = 0; g < ng; ++g) {
                        const int s = static_cast<int>(gc % kF8OpStages);
                        if (aborted(ctl) || !mbar_wait(smem_addr(&ctl->op_full[s]), (gc / kF8OpStages) & 1u)) {
                            give_up(p, ctl);
                            ok_run = false;
                            break;
                        }
                        mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->op_peer[s]), 0));
                        ++gc;
                    }
                    ++seg;
                    more = w.next(p, ctl->rng);
                }
            }
            if (!mbar_wait(smem_addr(&ctl->mma_done), 0))
                give_up(p, ctl);
        }
        __syncwarp();
    } else if (warp == kF8WaiterWarp) {
        if (rank == 0 && lane == 0) {
            const uint32_t addr = smem_addr(&ctl->ready);
            SegWalk w;
            bool more = w.start(p, ctl->rng);
            const SegWalk &c = w;
            uint32_t gc = 0;
            bool ok_run = true;
            while (more && ok_run) {
                const int ng = pairs_of(c.j, c.je);
                for (int g = 0; g < ng; ++g) {
                    const int s = static_cast<int>(gc % kF8OpStages);
                    const int a = static_cast<int>(gc % kF8AccBufs);
                    if (aborted(ctl) || !mbar_wait(smem_addr(&ctl->op_full[s]), (gc / kF8OpStages) & 1u) ||
                        !mbar_wait(smem_addr(&ctl->op_peer[s]), (gc / kF8OpStages) & 1u) ||
                        (gc >= kF8AccBufs &&
                         !bar_wait_test(smem_addr(&ctl->acc_empty[a]), ((gc / kF8AccBufs) - 1) & 1u))) {
                        give_up(p, ctl);
                        ok_run = false;
                        break;
                    }
                    st_release_shared_u32(addr, gc + 1);
                    ++gc;
                }
                more = ok_run && w.next(p, ctl->rng);
            }
        }
        __syncwarp();
    } else if (warp < kF8FirstEpi) {
        // ---------------- converters: a query row and a key row a lane ----------------
        const int cw = warp - kF8FirstConv;
        const int rr = 32 * cw + lane;  // this lane's query row and key row
        const uint32_t swz = static_cast<uint32_t>(rr & 7);
        SegWalk w;
        bool more = w.start(p, ctl->rng);
        const SegWalk &c = w;
        uint32_t gc = 0, seg = 0;
        bool ok_run = true;
        while (more && ok_run) {
            const int qb = static_cast<int>(seg % kF8QBufs);
            const uint32_t qph = (seg / kF8QBufs) & 1u;
            bool qready = !aborted(ctl) && mbar_wait(smem_addr(&ctl->q_full[qb]), qph) &&
                          (seg < kF8QBufs || mbar_wait(smem_addr(&ctl->inv_free[qb]), qph ^ 1u));
            qready = __all_sync(0xffffffffu, qready);
            if (!qready) {
                if (lane == 0)
                    give_up(p, ctl);
                break;
            }
            {
                const uint32_t qrow = q_smem + static_cast<uint32_t>(qb) * kF8QBytes + static_cast<uint32_t>(rr) * 128;
                float amax = 0.0f;
#pragma unroll 4
                for (int i = 0; i < 16; ++i) {
                    const uint4 v = lds128(qrow + static_cast<uint32_t>(i >> 3) * kF8QHalf +
                                           ((static_cast<uint32_t>(i & 7) ^ swz) << 4));
                    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(wv[t])), fabsf(bf16_hi(wv[t]))));
                }
                int ex = 0;
                if (amax > 0.0f)
                    frexpf(amax, &ex);
                const int sh = max(-100, min(100, 14 - ex));
                const float up = __int_as_float((127 + sh) << 23);
#pragma unroll 4
                for (int i = 0; i < 16; ++i) {
                    const uint32_t addr = qrow + static_cast<uint32_t>(i >> 3) * kF8QHalf +
                                          ((static_cast<uint32_t>(i & 7) ^ swz) << 4);
                    const uint4 v = lds128(addr);
                    uint4 o;
                    o.x = f32x2_to_f16x2(bf16_lo(v.x) * up, bf16_hi(v.x) * up);
                    o.y = f32x2_to_f16x2(bf16_lo(v.y) * up, bf16_hi(v.y) * up);
                    o.z = f32x2_to_f16x2(bf16_lo(v.z) * up, bf16_hi(v.z) * up);
                    o.w = f32x2_to_f16x2(bf16_lo(v.w) * up, bf16_hi(v.w) * up);
                    sts128(addr, o);
                }
                ctl->inv_row[qb][rr] = __int_as_float((127 - sh) << 23);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&ctl->q_conv[qb]));
            ++seg;

            const int ng = pairs_of(c.j, c.je);
            for (int g = 0; g < ng; ++g, ++gc) {
                const int rs = static_cast<int>(gc % kF8RawStages);
                const int os = static_cast<int>(gc % kF8OpStages);
                const int slot = static_cast<int>(gc % kF8Ring);
                bool ready = !aborted(ctl) && mbar_wait(smem_addr(&ctl->raw_full[rs]), (gc / kF8RawStages) & 1u);
                ready = ready && (gc < kF8OpStages ||
                                  bar_wait_test(smem_addr(&ctl->op_empty[os]), ((gc / kF8OpStages) - 1) & 1u));
                ready = ready && (gc < kF8Ring ||
                                  bar_wait_test(smem_addr(&ctl->sc_empty[slot]), ((gc / kF8Ring) - 1) & 1u));
                ready = __all_sync(0xffffffffu, ready);
                if (!ready) {
                    if (lane == 0)
                        give_up(p, ctl);
                    ok_run = false;
                    break;
                }
                {
                    const uint32_t src = raw_smem + rs * kF8RawBytes + static_cast<uint32_t>(rr) * 128;
                    const uint32_t dst = op_smem + os * kPageBytes + static_cast<uint32_t>(rr) * 128;
#pragma unroll
                    for (int cch = 0; cch < 8; ++cch) {
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
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int e = 64 * cw + lane + 32 * k;
                    ring[slot * kF8PairScales + e] = rawsc[rs * kF8PairScales + e];
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_addr(&ctl->op_full[os]));
                    mbar_arrive(smem_addr(&ctl->raw_empty[rs]));
                    mbar_arrive(smem_addr(&ctl->sc_full[slot]));
                }
            }
            more = ok_run && w.next(p, ctl->rng);
        }
    } else {
        // ---------------- epilogue: 16 rows x one page of the pair a warp ----------------
        const int e = warp - kF8FirstEpi;
        const int quarter = warp & 3;
        const int idx = e >> 2;
        const int h = idx & 1;          // the pair's first or second page
        const int rh = idx >> 1;        // the quarter's first or second 16 rows
        const int row0 = 32 * quarter + 16 * rh;  // first of the warp's rows, of the CTA's 128
        const int g8 = lane >> 2, cq = lane & 3;
        const int my_local = g8 + 8 * (cq & 1);
        const int my_row = row0 + my_local;
        const int my_tile_row = kMRows * static_cast<int>(rank) + my_row;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(row0) << 16) + static_cast<uint32_t>(h * kPage);
        const float neg_inf = -__int_as_float(0x7f800000);
        SegWalk w;
        bool more = w.start(p, ctl->rng);
        const SegWalk &c = w;
        uint32_t gc = 0, seg = 0;
        bool ok_run = true;
        while (more && ok_run) {
            const int je = c.je;
            const int qb = static_cast<int>(seg % kF8QBufs);
            const uint32_t qph = (seg / kF8QBufs) & 1u;
            bool conv = !aborted(ctl) && mbar_wait(smem_addr(&ctl->q_conv[qb]), qph);
            conv = __all_sync(0xffffffffu, conv);
            if (!conv) {
                if (lane == 0)
                    give_up(p, ctl);
                break;
            }
            const float my_inv = ctl->inv_row[qb][my_row];
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_addr(&ctl->inv_free[qb]));

            const int tl = kTileTokens * c.t + (my_tile_row >> 2);
            const bool live = cq < 2 && tl < c.r.n;
            const int pos = c.r.len - c.r.n + tl;
            float *out = p.scores + (static_cast<int64_t>(c.r.c0 + tl) * kHeads + (my_tile_row & 3)) * p.bs_stride;
            // rows g8 and g8 + 8 of the warp: the tokens at pos_q and pos_q + 2
            const int pos_lo = c.r.len - c.r.n + kTileTokens * c.t + ((kMRows * static_cast<int>(rank) + row0) >> 2);
            const int pos_q = pos_lo + (g8 >> 2);
            const int32_t *bt_row = p.block_table + static_cast<int64_t>(c.b) * p.bt_stride;
            const int ng = pairs_of(c.j, je);
            int page_next = c.j + h < je ? __ldg(bt_row + c.j + h) : 0;
            for (int g = 0; g < ng; ++g, ++gc) {
                const int a = static_cast<int>(gc % kF8AccBufs);
                const int slot = static_cast<int>(gc % kF8Ring);
                const int j = c.j + 2 * g + h;
                const int page = page_next;
                if (j + 2 < je)
                    page_next = __ldg(bt_row + j + 2);
                bool ready = !aborted(ctl) && mbar_wait(smem_addr(&ctl->acc_full[a]), (gc / kF8AccBufs) & 1u) &&
                             bar_wait_test(smem_addr(&ctl->sc_full[slot]), (gc / kF8Ring) & 1u);
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
                if (j < je && page_ok && __any_sync(0xffffffffu, want)) {
                    const float2 *sc2 = reinterpret_cast<const float2 *>(ring + slot * kF8PairScales + h * kPage);
                    const uint32_t acc = lane_addr + static_cast<uint32_t>(a * 2 * kPage);
                    const bool full = pos_lo >= first_key + kPage - 1;
                    const int l0 = pos_q - first_key;
                    float ma = neg_inf, mb = neg_inf;
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
                } else if (j < je && !page_ok && want) {
                    out[j] = neg_inf;
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_cluster(mapa_shared(smem_addr(&ctl->acc_empty[a]), 0));
                    mbar_arrive(smem_addr(&ctl->sc_empty[slot]));
                }
            }
            ++seg;
            more = ok_run && w.next(p, ctl->rng);
        }
    }

    tc_fence_before_sync();
    __syncwarp();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, kF8TmemCols);
    }
    if (threadIdx.x == 0)
        pass_end(p, ctl);
}

}  // namespace msa
