// rope.cu -- op "rope" of the op catalog (vtmu.mpakt.dev/api/ops): rotary
// position embedding of x [T, heads*headDim], row t at position offset + t.
// Memory-bound and elementwise: one CTA per row at a time; its threads first
// form the row's (cos, sin) table, one entry per pair (the angle in double,
// see rope.cuh), then turn every head's pairs with it.  Each thread reads and
// writes both channels of a pair, so x == out (in place) is safe.
#include "kernels.h"
#include "rope.cuh"

namespace vtmu {
namespace {

__global__ void __launch_bounds__(256) rope_kernel(const float* x, float* out, int64_t T, int H, int D,
                                                   int64_t offset, const RopeDev r) {
    __shared__ float2 cs[kRopeMaxPairs];
    const int half = r.half;
    const int64_t row_len = (int64_t)H * D;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        __syncthreads();  // the previous row's table is no longer read
        for (int j = threadIdx.x; j < half; j += blockDim.x) cs[j] = rope_cos_sin(r, offset + t, j);
        __syncthreads();
        const float* xr = x + t * row_len;
        float* orow = out + t * row_len;
        for (int e = threadIdx.x; e < H * half; e += blockDim.x) {
            const int h = e / half, j = e - h * half;
            const int ia = r.interleaved ? 2 * j : j;
            const int ib = r.interleaved ? 2 * j + 1 : j + half;
            const float a = xr[h * D + ia], b = xr[h * D + ib];
            orow[h * D + ia] = rope_channel(a, b, true, cs[j]);
            orow[h * D + ib] = rope_channel(b, a, false, cs[j]);
        }
        if (out != x) {
            const int pass = D - 2 * half;
            for (int e = threadIdx.x; e < H * pass; e += blockDim.x) {
                const int h = e / pass, d = 2 * half + (e - h * pass);
                orow[h * D + d] = xr[h * D + d];
            }
        }
    }
}

}  // namespace

cudaError_t launch_rope(const float* x, float* out, int64_t T, int H, int D, int64_t offset, const RopeDev& r,
                        cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    constexpr int kThreads = 256;
    constexpr int64_t kMaxBlocks = 152 * 8;
    const int64_t blocks = T < kMaxBlocks ? T : kMaxBlocks;
    rope_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(x, out, T, H, D, offset, r);
    return cudaGetLastError();
}

}  // namespace vtmu
