// softcap_probe.cu -- test-only kernels that evaluate the library's two tanh
// approximations of the softcap (op "attention", param softcap: x ->
// cap * tanh(x / cap)) pointwise, for a dense comparison against tanh:
//   softcap_tanh (attn_common.cuh): the per-score form, and
//   softcap_tile (softcap.cuh): the tile form with its odd series.
// Built by the test that uses it; not part of the library.
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "softcap.cuh"

namespace {

constexpr int kPer = 16;  // values per thread in the tile form

// out_lib[i] = softcap_tanh(y[i]); out_ref[i] = tanhf(y[i]).
__global__ void scalar_kernel(const float* __restrict__ y, float* __restrict__ out_lib,
                              float* __restrict__ out_ref, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        out_lib[i] = vtmu::softcap_tanh(y[i]);
        out_ref[i] = tanhf(y[i]);
    }
}

// Thread t of the grid holds y[t*kPer .. t*kPer+kPer) (n is a multiple of
// 32 * kPer, so every warp is full); out[i] = cap * tanh(y[i] * qk_mul) by
// softcap_tile; series[warp] = 1 when the warp took the odd series.
__global__ void tile_kernel(const float* __restrict__ y, float* __restrict__ out, int* __restrict__ series,
                            float qk_mul, float cap, int n) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int nthreads = n / kPer;
    if (t >= nthreads) return;  // whole warps only: nthreads is a multiple of 32
    float x[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) x[j] = y[t * kPer + j];
    const bool s = vtmu::softcap_tile<kPer>(x, qk_mul, cap);
#pragma unroll
    for (int j = 0; j < kPer; ++j) out[t * kPer + j] = x[j];
    if ((threadIdx.x & 31) == 0) series[t / 32] = s ? 1 : 0;
}

}  // namespace

#define PROBE_API __attribute__((visibility("default")))

extern "C" {

PROBE_API int softcap_probe_values_per_warp() { return 32 * kPer; }

// y, out_lib, out_ref: DEVICE [n] floats.
PROBE_API int softcap_probe_scalar(const float* y, float* out_lib, float* out_ref, int n, cudaStream_t stream) {
    if (n <= 0) return 0;
    scalar_kernel<<<(n + 255) / 256, 256, 0, stream>>>(y, out_lib, out_ref, n);
    return (int)cudaGetLastError();
}

// y, out: DEVICE [n] floats, series: DEVICE [n / (32 * kPer)] ints; n must be
// a multiple of 32 * kPer.
PROBE_API int softcap_probe_tile(const float* y, float* out, int* series, float qk_mul, float cap, int n,
                       cudaStream_t stream) {
    if (n <= 0 || n % (32 * kPer) != 0) return (int)cudaErrorInvalidValue;
    const int nthreads = n / kPer;
    tile_kernel<<<(nthreads + 127) / 128, 128, 0, stream>>>(y, out, series, qk_mul, cap, n);
    return (int)cudaGetLastError();
}

}  // extern "C"
