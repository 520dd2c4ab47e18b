// attn_common.cuh -- device-side pieces shared by the attention kernels:
// the resolved call description and the fused score epilogue.
//
// Op "attention" of the op catalog (vtmu.mpakt.dev/api/ops) scores key s for
// query row t of head h as
//     x = scale * q.k ; x = softcap * tanh(x / softcap) ; x += slope_h * (s - p)
//     x += bias ; masked when s is not visible from p = posOffset + t
// (the cap ahead of masking, the bias an additive term).  The kernels keep
// x in base-2 units (x * log2 e) so that the softmax uses exp2; the factor is
// folded into the constants below, never applied as a separate pass.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "attn_desc.h"

namespace vtmu {

// op "attention", param window: causal keys visible when p - w < s <= p,
// non-causal ones when |p - s| <= w (w == 0: no window).  SINKS: attention
// sinks may be on (keys s < a.sinks escape the window).
template <bool SINKS = true>
__device__ __forceinline__ bool key_visible(const AttnDesc& a, int64_t p, int64_t s) {
    if (s < 0 || s >= a.S) return false;
    if (a.causal && s > p) return false;
    if (a.window > 0) {
        if (SINKS && s < a.sinks) return true;  // attention sinks escape the window
        if (a.causal) return s > p - a.window;
        int64_t d = p > s ? p - s : s - p;
        return d <= a.window;
    }
    return true;
}

// tanh(y) for the softcap, from two identities of the hyperbolic tangent:
// its odd Taylor series y - y^3/3 + 2y^5/15 - 17y^7/315 + 62y^9/2835 for
// |y| < 1/4 (the first dropped term, 1382 y^11 / 155925, is below 3e-9 there)
// and tanh|y| = (1 - e) / (1 + e) with e = exp(-2|y|) = 2^(-2|y| log2 e) on the
// MUFU unit elsewhere.  Absolute error a few 1e-7, the order of tanhf's; both
// tails are exact (e -> 0 gives 1).
__device__ __forceinline__ float softcap_tanh(float y) {
    const float ay = fabsf(y);
    float e;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(e) : "f"(ay * -2.8853900817779268f));
    const float big = __fdividef(1.f - e, 1.f + e);
    const float y2 = y * y;
    float p = fmaf(y2, 62.f / 2835.f, -17.f / 315.f);
    p = fmaf(y2, p, 2.f / 15.f);
    p = fmaf(y2, p, -1.f / 3.f);
    p = fmaf(y2, p, 1.f);
    return ay < 0.25f ? y * p : copysignf(big, y);
}

// The fused epilogue, in base-2 units: scale -> softcap -> ALiBi -> bias.
// `dot` is the raw q.k sum; `rel` = s - p; `bias_val` the bias entry (or 0).
__device__ __forceinline__ float score_log2(const AttnDesc& a, float dot, float slope_log2,
                                            int64_t rel, float bias_val) {
    float x;
    if (a.softcap_on)
        x = a.cap_log2 * softcap_tanh(dot * a.qk_mul);
    else
        x = dot * a.qk_mul;
    if (a.alibi_on) x = fmaf(slope_log2, (float)rel, x);
    if (a.bias_kind) x = fmaf(bias_val, kLog2e, x);
    return x;
}

__device__ __forceinline__ float bias_at(const AttnDesc& a, int h, int64_t t, int64_t s) {
    if (a.bias_kind == 1) return __ldg(a.bias + t * a.S + s);
    return __ldg(a.bias + ((int64_t)h * a.T + t) * a.S + s);
}

// exp2 of a base-2 score difference; -inf maps to 0.
__device__ __forceinline__ float exp2_diff(float x, float m) { return exp2f(x - m); }

// ---- cp.async (LDGSTS) helpers: global -> shared without registers --------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte copy; src_bytes == 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}

// 4-byte copy; src_bytes == 0 zero-fills the destination.
__device__ __forceinline__ void cp_async4(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

}  // namespace vtmu
