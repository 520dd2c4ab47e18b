// rope.cuh -- device helpers of the rotary position embedding (op "rope" of
// the op catalog, vtmu.mpakt.dev/api/ops), shared by the rope kernel and the
// fused decode step so that both turn a channel with the same arithmetic.
#pragma once

#include <cstdint>

#include "attn_desc.h"

namespace vtmu {

// attentionFactor * (cos, sin) of theta = pos * inv_freq[j].  The angle is
// formed in double and reduced to [-pi, pi] in double by Cody and Waite's
// method (2 pi as a double plus the double nearest its remainder, each
// subtracted with a fused multiply-add), so that positions in the tens of
// thousands keep full accuracy; the hardware sine/cosine (__sincosf, absolute
// error below 2^-21 on [-pi, pi]) then works on the reduced f32 angle.
__device__ __forceinline__ float2 rope_cos_sin(const RopeDev& r, int64_t pos, int j) {
    constexpr double kTwoPiHi = 6.283185307179586;       // double nearest 2 pi
    constexpr double kTwoPiLo = 2.4492935982947064e-16;  // 2 pi - kTwoPiHi
    constexpr double kInvTwoPi = 0.15915494309189535;
    const double th = (double)pos * r.inv_freq[j];
    const double n = rint(th * kInvTwoPi);
    const double red = fma(-n, kTwoPiLo, fma(-n, kTwoPiHi, th));
    float s, c;
    __sincosf((float)red, &s, &c);
    return make_float2(c * r.attn, s * r.attn);
}

// Pair index j and partner channel of rotated channel d (d < 2 * half);
// `first` is true for the channel that turns as a cos - b sin.
__device__ __forceinline__ void rope_pair_of(const RopeDev& r, int d, int& j, int& partner, bool& first) {
    if (r.interleaved) {
        j = d >> 1;
        partner = d ^ 1;
        first = (d & 1) == 0;
    } else {
        first = d < r.half;
        j = first ? d : d - r.half;
        partner = first ? d + r.half : d - r.half;
    }
}

// The turned value of a channel whose own value is `own` and whose pair
// partner is `other`: (a, b) -> (a cos - b sin, b cos + a sin).
__device__ __forceinline__ float rope_channel(float own, float other, bool first, float2 cs) {
    return first ? fmaf(own, cs.x, -(other * cs.y)) : fmaf(own, cs.x, other * cs.y);
}

}  // namespace vtmu
