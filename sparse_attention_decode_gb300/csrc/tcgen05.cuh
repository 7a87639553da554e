// Inline-PTX wrappers for the 5th-generation tensor cores (tcgen05) on
// sm_100a / sm_103a: tensor-memory (TMEM) allocation, shared-memory matrix
// descriptors, MMA issue and completion, and TMEM loads.
//
// Conventions used by the kernels here: A and B of one type (bf16, or f16 on
// the E4M3 cache) and K-major in shared memory in the 128-byte swizzle layout
// that a TMA load with CU_TENSOR_MAP_SWIZZLE_128B produces (rows of 128 B,
// atoms of 8 rows = 1024 B, every operand tile 1024-byte aligned), D in fp32
// in TMEM.  The E4M3 kernel runs one CTA per SM (cta_group::1); the bf16
// kernel runs pairs of CTAs (cta_group::2, the wrappers at the end).
#pragma once

#include <cstdint>

namespace msa {

// Allocates `ncols` TMEM columns (a power of two, 32..512) and writes the base
// address to the shared-memory word at `dst`.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_alloc_permit()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Frees what tmem_alloc took; the same warp, after every TMEM access is done.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// Orders tcgen05 operations before / after a thread synchronisation
// (barrier, mbarrier wait or arrive).
__device__ __forceinline__ void tc_fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout, as two 32-bit words.  Low word: start address >> 4 (bits
// 0-13) and the leading-dimension offset (bits 16-29; 16 B, not used by
// swizzled K-major operands whose K extent per instruction, 16 elements =
// 32 B, lies inside one 128-byte row).  High word: the stride between 8-row
// atoms (1024 B >> 4), the descriptor version bit of sm_100-class parts and
// the swizzle mode.  Only the start address changes between instructions, so
// an operand one K step (32 B) or one tile further on is the low word plus
// that byte offset >> 4: shared addresses stay below 2^18, so the 14-bit field
// never carries.
__device__ __forceinline__ uint32_t umma_desc_lo(uint32_t saddr)
{
    return ((saddr >> 4) & 0x3FFFu) | (1u << 16);
}
constexpr uint32_t kUmmaDescHi = (1024u >> 4)    // stride byte offset: 8 rows x 128 B
                                 | (1u << 14)   // version (bit 46)
                                 | (2u << 29);  // 128-byte swizzle (bits 61-63)

// Instruction descriptor of kind::f16 with bf16 A and B (both K-major) and an
// fp32 accumulator, shape M x N (K = 16).
__host__ __device__ constexpr uint32_t umma_idesc_bf16_f32(int m, int n)
{
    return (1u << 4)                                   // D: fp32
           | (1u << 7)                                 // A: bf16
           | (1u << 10)                                // B: bf16
           | (static_cast<uint32_t>(n >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(m >> 4) << 24);    // M / 16
}

// Instruction descriptor of kind::f16 with f16 A and B (both K-major) and an
// fp32 accumulator, shape M x N (K = 16).
__host__ __device__ constexpr uint32_t umma_idesc_f16_f32(int m, int n)
{
    return (1u << 4)                                   // D: fp32
           | (static_cast<uint32_t>(n >> 3) << 17)     // N / 8 (A, B: f16 = 0)
           | (static_cast<uint32_t>(m >> 4) << 24);    // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T (kind::f16, cta_group::1), issued by one
// thread; the operands are given by their descriptors' low words
// (umma_desc_lo), ACC = false overwrites D.
template <bool ACC>
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc)
{
    asm volatile(
        "{\n"
        "  .reg .b64 ad, bd;\n"
        "  mov.b64 ad, {%1, %5};\n"
        "  mov.b64 bd, {%2, %5};\n"
        "  tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %3, %4;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(idesc), "n"(ACC ? 1 : 0), "r"(kUmmaDescHi)
        : "memory");
}

// Arrives once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// 32 consecutive fp32 columns of one TMEM lane per thread (shape 32x32b: warp
// w reads lanes 32*(w%4) .. 32*(w%4)+31, lane i of the warp gets lane 32*(w%4)+i).
// The values are valid after tmem_wait_ld(r).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// 16 lanes x 32 fp32 columns in the mma-fragment layout: with g = lane / 4 and
// c = lane % 4, repetition i (0..3) gives r[4i], r[4i+1] = row g, columns
// 8i + 2c, 8i + 2c + 1 and r[4i+2], r[4i+3] = row g + 8, the same columns.
// taddr's lane field is the first of the 16 rows (inside the warp's quarter).
__device__ __forceinline__ void tmem_ld16x256b_x4(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Waits for all of this thread's TMEM loads (r and any other in flight); r
// passes through the asm so that no use of it is scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

// Marks r as written here: placed after a tmem_wait_ld that also covered r's
// load, it keeps r's uses after that wait.
__device__ __forceinline__ void tmem_regs_ready(uint32_t (&r)[16])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

// Marks r as written here (32 registers): placed after a tmem_wait_ld that
// also covered r's load, it keeps r's uses after that wait.
__device__ __forceinline__ void tmem_regs_ready(uint32_t (&r)[32])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]));
}

// Waits for this thread's TMEM loads; the registers pass through the asm so
// that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}


// ---- pairs of CTAs (a cluster of two, cta_group::2) ----
// With cta_group::2 the two CTAs of a cluster act as one MMA unit: one thread
// of the even CTA issues an M = 256 MMA whose A rows 0-127 come from the even
// CTA's shared memory and rows 128-255 from the odd CTA's (the same offset in
// both), whose B rows (the N keys) come half from each CTA (keys 0 .. N/2-1
// from the even CTA, N/2 .. N-1 from the odd one, again the same offset), and
// whose accumulator rows land in each CTA's own TMEM (rows 0-127 in the even
// CTA's lanes, 128-255 in the odd CTA's, the same columns).  Allocation and
// release are collective: one warp of each CTA executes them.  (Checked on
// GB300 with a known-answer product before use: both CTAs receive the same
// TMEM address, and B's rows split between the CTAs as stated.)

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of the variable at local shared address `addr`
// in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrives on an mbarrier of another CTA of the cluster (default semantics:
// release at CTA scope; with .release.cluster here and acquire.cluster on the
// waiting side the pair kernel ran 1.36x slower).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Every thread of both CTAs: all writes before it are visible to all after it.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A * B^T over the pair (kind::f16, cta_group::2), issued by one
// thread of the even CTA.
template <bool ACC>
__device__ __forceinline__ void umma_pair_f16(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc)
{
    asm volatile(
        "{\n"
        "  .reg .b64 ad, bd;\n"
        "  mov.b64 ad, {%1, %5};\n"
        "  mov.b64 bd, {%2, %5};\n"
        "  tcgen05.mma.cta_group::2.kind::f16 [%0], ad, bd, %3, %4;\n"
        "}\n" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(idesc), "n"(ACC ? 1 : 0), "r"(kUmmaDescHi)
        : "memory");
}

// Arrives once on the mbarrier at local offset `bar` in both CTAs of the pair
// when every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(static_cast<uint16_t>(0x3))
        : "memory");
}

}  // namespace msa
