// softcap.cuh -- the softcap of op "attention" (param softcap; op softcap:
// cap * tanh(x / cap)) over a whole tile of scores, and the packed f32x2
// arithmetic it runs on.  The per-score form, softcap_tanh, is in
// attn_common.cuh.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "attn_common.cuh"

namespace vtmu {

// Packed pairs of f32 (Blackwell's f32x2 add / mul / fma): two lanes of
// arithmetic per instruction for the softmax's elementwise work.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Softcap of a tile's raw scores, in place, by a converged warp: x <- cap *
// tanh(x * qk_mul) (cap and qk_mul in base-2 units).  The odd Taylor series of
// tanh through y^13 (coefficients 1, -1/3, 2/15, -17/315, 62/2835,
// -1382/155925, 21844/6081075) covers |y| < 1/2, where the first dropped term,
// 929569 y^15 / 638512875, is below 5e-8; it needs no MUFU operation.  Typical
// softcap arguments (score / cap) stay below 1/2; if any lane of the warp
// sees a larger one, the whole tile takes softcap_tanh instead.  Returns
// true when the series ran (the kernels ignore it; the tests read it).
template <int N>
__device__ __forceinline__ bool softcap_tile(float (&x)[N], float qk_mul, float cap) {
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i) am = fmaxf(am, fabsf(x[i]));
    if (__any_sync(0xffffffffu, am * fabsf(qk_mul) >= 0.5f)) {
#pragma unroll
        for (int i = 0; i < N; ++i) x[i] = cap * softcap_tanh(x[i] * qk_mul);
        return false;
    }
    {
        const uint64_t q2 = f2_pack(qk_mul, qk_mul), cap2 = f2_pack(cap, cap);
        const uint64_t c13 = f2_pack(21844.f / 6081075.f, 21844.f / 6081075.f),
                       c11 = f2_pack(-1382.f / 155925.f, -1382.f / 155925.f),
                       c9 = f2_pack(62.f / 2835.f, 62.f / 2835.f), c7 = f2_pack(-17.f / 315.f, -17.f / 315.f),
                       c5 = f2_pack(2.f / 15.f, 2.f / 15.f), c3 = f2_pack(-1.f / 3.f, -1.f / 3.f),
                       c1 = f2_pack(1.f, 1.f);
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const uint64_t y = f2_mul(f2_pack(x[i], x[i + 1]), q2), y2 = f2_mul(y, y);
            uint64_t p = f2_fma(y2, c13, c11);
            p = f2_fma(y2, p, c9);
            p = f2_fma(y2, p, c7);
            p = f2_fma(y2, p, c5);
            p = f2_fma(y2, p, c3);
            p = f2_fma(y2, p, c1);
            f2_unpack(f2_mul(cap2, f2_mul(y, p)), x[i], x[i + 1]);
        }
    }
    return true;
}

}  // namespace vtmu
