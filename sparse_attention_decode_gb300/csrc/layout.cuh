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
// The score kernel cuts that sequence into chunks of `split` pages; chunk c
// contributes one top-kmax list per head for every request it touches, stored
// in slot c + b.  Slot indices are unique because both c and b grow along
// the page sequence.
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

struct WorkspaceHeader {
    uint32_t fault;   // OR of MSA_FAULT_* bits; cleared by msa_indexer_get_error
    int32_t split;    // pages per chunk used by the last score pass
    int32_t total;    // pages in that batch
    int32_t chunks;   // chunks in that batch
    int32_t batch;    // batch of that pass
    int32_t kmax;     // list length of that pass
    uint32_t reserved[58];
};
static_assert(sizeof(WorkspaceHeader) == kHeaderBytes, "header must be 256 bytes");

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
