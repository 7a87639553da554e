// Host-side helpers shared by the indexer's translation units: launch
// configuration with programmatic dependent launch, the driver's tensor-map
// encoder, and per-device attribute caches.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "layout.cuh"

namespace msa {

// Launch configuration with programmatic dependent launch: the grid may be
// scheduled while the previous kernel on the stream is still running; it
// calls griddep_wait() before touching global memory, so it observes all of
// that kernel's writes (and the previous kernel cannot see any of its own).
static cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                     cudaLaunchAttribute (&attr)[1])
{
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

constexpr int kMaxDevices = 64;

static int device_sms(int dev)
{
    static std::atomic<int> cache[kMaxDevices];
    int v = (dev >= 0 && dev < kMaxDevices) ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (v > 0)
        return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        return 0;
    if (dev >= 0 && dev < kMaxDevices)
        cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

// L2 size of device `dev` in bytes (0 when the query fails).
static int64_t device_l2_bytes(int dev)
{
    static std::atomic<int> cache[kMaxDevices];
    int v = (dev >= 0 && dev < kMaxDevices) ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (v > 0)
        return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess || v <= 0)
        return 0;
    if (dev >= 0 && dev < kMaxDevices)
        cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

static int64_t blocks_for(int max_model_len) { return (static_cast<int64_t>(max_model_len) + kPage - 1) / kPage; }

}  // namespace msa
