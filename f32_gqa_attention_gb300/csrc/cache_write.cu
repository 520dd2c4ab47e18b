// cache_write.cu -- op "cache_write" of the op catalog (vtmu.mpakt.dev/api/ops):
// cache[offset + r, :] = values[r, :] for r < rows, in place.  A bit-exact
// row-block copy: the destination block is contiguous (rows * width floats
// starting at row `offset`), so the kernel is a flat vectorised copy.
#include "kernels.h"

namespace vtmu {
namespace {

__global__ void cache_write_vec4(float4* __restrict__ dst, const float4* __restrict__ src, int64_t n4) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = __ldg(src + i);
}

__global__ void cache_write_scalar(float* __restrict__ dst, const float* __restrict__ src, int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = __ldg(src + i);
}

}  // namespace

cudaError_t launch_cache_write(float* cache, int64_t width, const float* values, int64_t rows,
                               int64_t offset, cudaStream_t stream) {
    float* dst = cache + offset * width;
    const int64_t n = rows * width;
    if (n == 0) return cudaSuccess;
    constexpr int kThreads = 256;
    constexpr int64_t kMaxBlocks = 152 * 8;
    const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(values)) & 15u) == 0 &&
                     (n % 4) == 0;
    if (vec) {
        const int64_t n4 = n / 4;
        int64_t blocks = (n4 + kThreads - 1) / kThreads;
        if (blocks > kMaxBlocks) blocks = kMaxBlocks;
        cache_write_vec4<<<(unsigned)blocks, kThreads, 0, stream>>>(
            reinterpret_cast<float4*>(dst), reinterpret_cast<const float4*>(values), n4);
    } else {
        int64_t blocks = (n + kThreads - 1) / kThreads;
        if (blocks > kMaxBlocks) blocks = kMaxBlocks;
        cache_write_scalar<<<(unsigned)blocks, kThreads, 0, stream>>>(dst, values, n);
    }
    return cudaGetLastError();
}

}  // namespace vtmu
