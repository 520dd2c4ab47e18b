// launch_cache.h -- host-side caches that keep driver calls off the per-call
// path: the dynamic shared-memory attribute of a kernel is set once per
// device, and TMA descriptors are re-encoded only when their tensor changes.
// A decode step is ~50 us of GPU time, so a few microseconds of host work per
// launch are visible whenever the caller waits for each step.
#pragma once

#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

namespace vtmu {

// cudaFuncSetAttribute(kern, MaxDynamicSharedMemorySize, bytes), skipped when
// this kernel already has that value on the current device.
inline cudaError_t set_smem_once(const void* kern, int bytes) {
    struct Entry {
        const void* kern;
        int dev;
        int bytes;
    };
    static Entry table[128];
    static int used = 0;
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (table[i].kern == kern && table[i].dev == dev && table[i].bytes == bytes) return cudaSuccess;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (used < 128) table[used++] = Entry{kern, dev, bytes};
    return cudaSuccess;
}

// A 2-D f32 tensor map of `base` ([rows, cols], row-major, boxes box_rows x
// box_cols, swizzle kind `swz`), taken from a small per-thread cache when the
// same tensor was encoded before; `encode` fills a map on a miss.
template <class Encode>
bool cached_tensor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_cols, int box_rows,
                       int swz, Encode encode) {
    struct Entry {
        const void* base;
        int64_t rows, cols;
        int box_cols, box_rows, swz;
        bool valid;
        CUtensorMap map;
    };
    constexpr int kEntries = 16;
    thread_local Entry cache[kEntries];
    thread_local int next = 0;
    for (int i = 0; i < kEntries; ++i) {
        const Entry& c = cache[i];
        if (c.valid && c.base == base && c.rows == rows && c.cols == cols && c.box_cols == box_cols &&
            c.box_rows == box_rows && c.swz == swz) {
            std::memcpy(map, &c.map, sizeof(CUtensorMap));
            return true;
        }
    }
    if (!encode(map)) return false;
    Entry& c = cache[next];
    next = (next + 1) % kEntries;
    c = Entry{base, rows, cols, box_cols, box_rows, swz, true, *map};
    return true;
}

}  // namespace vtmu
