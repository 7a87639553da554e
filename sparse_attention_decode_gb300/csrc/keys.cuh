// Packed 64-bit candidate keys and warp-level top-k on them.
//
// A candidate is one (score, block id) pair packed into a uint64 so that
// "larger key" means "selected earlier" (vLLM PR #57832, "Solution", step 3:
// each candidate packed into one int64 (score, global block id) key; SGLang
// PR #41488, "Modifications": packed score/ID keys).  Layout:
//
//   free block   : bit 63 = 0, bits 62..31 = ord(score), bits 30..0 = 0x7FFFFFFF - id
//   pinned block : bit 63 = 1, bits 62..32 = 0x7FFFFFFF - id, bits 31..0 = fp32 bits of score
//   empty slot   : 0
//
// ord() maps fp32 to uint32 preserving order, so comparing keys as unsigned
// integers orders free blocks by higher score then lower id, and puts every
// pinned block above every free block, pinned ones in increasing id.  -0 is
// folded to +0 before packing so equal scores compare equal.
#pragma once

#include <cstdint>

namespace msa {

__device__ __forceinline__ uint32_t float_order_bits(float s)
{
    uint32_t u = __float_as_uint(s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float float_from_order_bits(uint32_t o)
{
    uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t pack_key(float score, int block, bool pinned)
{
    score = (score == 0.0f) ? 0.0f : score;  // -0 -> +0
    const uint64_t rid = 0x7FFFFFFFu - static_cast<uint32_t>(block);
    if (pinned)
        return (1ull << 63) | (rid << 32) | __float_as_uint(score);
    return (static_cast<uint64_t>(float_order_bits(score)) << 31) | rid;
}

__device__ __forceinline__ void unpack_key(uint64_t key, int &block, float &score)
{
    if (key == 0) {
        block = -1;
        score = -__int_as_float(0x7f800000);
    } else if (key >> 63) {
        block = static_cast<int>(0x7FFFFFFFu - static_cast<uint32_t>((key >> 32) & 0x7FFFFFFFu));
        score = __uint_as_float(static_cast<uint32_t>(key));
    } else {
        block = static_cast<int>(0x7FFFFFFFu - static_cast<uint32_t>(key & 0x7FFFFFFFu));
        score = float_from_order_bits(static_cast<uint32_t>(key >> 31));
    }
}

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// Sorts a bitonic sequence held one element per lane in aligned groups of
// WIDTH lanes into descending order (rank = lane % WIDTH).  All 32 lanes
// must call it.
template <int WIDTH>
__device__ __forceinline__ uint64_t bitonic_to_desc(uint64_t v, int lane)
{
#pragma unroll
    for (int s = WIDTH / 2; s >= 1; s >>= 1) {
        const uint64_t other = __shfl_xor_sync(0xffffffffu, v, s);
        v = (lane & s) ? umin64(v, other) : umax64(v, other);
    }
    return v;
}

// Given two descending lists of length WIDTH (this lane holds a[rank] and
// b[WIDTH-1-rank]), returns this lane's element of the descending top-WIDTH
// of their union.
template <int WIDTH>
__device__ __forceinline__ uint64_t merge_top(uint64_t a_rank, uint64_t b_reversed, int lane)
{
    return bitonic_to_desc<WIDTH>(umax64(a_rank, b_reversed), lane);
}

// Inserts `key` into a descending list held one element per lane in aligned
// groups of WIDTH lanes; the smallest element drops out.  Keys in one list
// are distinct unless zero.
template <int WIDTH>
__device__ __forceinline__ uint64_t insert_desc(uint64_t cur, uint64_t key, int lane)
{
    const uint64_t up = __shfl_up_sync(0xffffffffu, cur, 1, WIDTH);
    const bool first = (lane % WIDTH) == 0;
    if (key > cur)
        return (!first && key > up) ? up : key;
    return cur;
}

}  // namespace msa
