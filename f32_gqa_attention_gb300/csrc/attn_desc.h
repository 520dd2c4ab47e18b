// attn_desc.h -- the resolved description of one attention call, shared by
// the host-side C ABI and the kernels (plain structs, no device code).
#pragma once

#include <cstdint>

namespace vtmu {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxAlibiHeads = 512;

// Everything a kernel needs about one call, resolved on the host.
struct AttnDesc {
    const float* q;
    const float* k;
    const float* v;
    const float* bias;   // nullptr when bias_kind == 0
    float* out;
    int64_t T, S;
    int32_t H, Hk, G, D, Dv;
    int32_t causal;
    int64_t pos_offset;
    int64_t window;      // 0 = off
    int64_t sinks;       // with a window: keys s < sinks stay visible (0 = none)
    int32_t bias_kind;   // 0 none, 1 [T,S], 2 [H,T,S]
    int32_t softcap_on;
    int32_t alibi_on;
    // Score constants.  Without softcap: x2 = dot * qk_mul.  With softcap:
    // x2 = cap_log2 * tanh(dot * qk_mul), qk_mul = scale / softcap.
    float qk_mul;
    float cap_log2;
};

// Per-head ALiBi slopes, pre-multiplied by log2 e (passed by value).
struct AlibiTable {
    float slope_log2[kMaxAlibiHeads];
};

// Rotary position embedding (op "rope"), resolved on the host (passed by
// value).  Pair j < half turns by pos * inv_freq[j]: channels (j, j + half),
// or (2j, 2j + 1) when interleaved; channels at or past 2 * half pass through.
constexpr int kRopeMaxPairs = 128;  // rotaryDim <= 256
struct RopeDev {
    int32_t half;         // rotaryDim / 2 (0: nothing turns)
    int32_t interleaved;
    float attn;           // attentionFactor, multiplies cos and sin
    int32_t pad;
    double inv_freq[kRopeMaxPairs];  // with a linear scaling's factor divided out
};

}  // namespace vtmu
