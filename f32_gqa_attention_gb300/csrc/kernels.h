// kernels.h -- host-side launch interface of the kernels (library-internal).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "attn_desc.h"

namespace vtmu {

// Every workspace starts with this header, which only the decode kernel's
// arrival counters use (one per KV head, zero between calls).  Other
// kernels keep their scratch after it, so the counters survive any mix of
// calls on one workspace.
constexpr size_t kWorkspaceHeader = 64 * 1024;
constexpr int kMaxDecodeKvHeads = (int)(kWorkspaceHeader / 4);

// ---- split-KV decode (T == 1) ---------------------------------------------
struct DecodePlan {
    int64_t s_lo = 0;            // first visible key
    int64_t s_end = 0;           // one past the last visible key
    int64_t rows_per_split = 0;  // multiple of the kernel's stage rows
    int64_t sink_end = 0;        // attention sinks: rows [0, sink_end) stream first
    int32_t sink_splits = 0;     // splits given to them
    int32_t splits = 1;          // per KV head and row group
    // Query rows: gv virtual heads (tc rows x the group's heads, padded to a
    // power of two >= 2) per KV head and row group; n_rg row groups.
    int32_t gv = 2;
    int32_t tc = 1;
    int32_t n_rg = 1;
    size_t workspace_bytes = 0;
};

// A cache_write fused into a decode launch: rows [lo, hi) of the K and V
// caches (row-major [*, kvHeads*headDim]) take k_new / v_new rows 0..hi-lo-1.
struct DecodeCacheWrite {
    float* kc;
    float* vc;
    const float* k_new;
    const float* v_new;
    int64_t lo, hi;
};

// True when the decode kernel's shape table covers this call (1 <= T <=
// kDecodeMaxRows, headDim == vHeadDim in {32, 64, 128}, group size in
// {1, 2, 4, 8}).  Pointer alignment is checked separately at launch.
constexpr int kDecodeMaxRows = 16;
bool decode_supported(const AttnDesc& a);
// Fills `plan` for the call; `forced_splits` > 0 overrides the heuristic.
void decode_plan(const AttnDesc& a, int forced_splits, int num_sms, DecodePlan* plan);
// With `rope`, the query row and the new key rows are turned by the rotary
// embedding first (the cache receives turned keys).
cudaError_t launch_decode(const AttnDesc& a, const AlibiTable& alibi, const DecodePlan& plan,
                          void* workspace, cudaStream_t stream, const DecodeCacheWrite* cw = nullptr,
                          const RopeDev* rope = nullptr);
// Reads and clears the decode kernel's device error flag (synchronous).
unsigned int decode_take_device_error();

// ---- decode of a few query rows, scores on the tensor cores ------------------
// Up to 16 virtual heads (query rows x group heads) per KV head.
constexpr int kDecodeTcHeads = 16;
constexpr int kDecodeTcMaxSplits = 256;
struct DecodeTcPlan {
    int64_t lo = 0, hi = 0;  // the visible range [lo, hi)
    int64_t sink_end = 0;    // attention sinks: rows [0, sink_end) as a range of their own
    int32_t n_sink_tiles = 0, n_tiles = 0;  // 128-row tiles of the two ranges
    int32_t splits = 1, sink_splits = 0;    // per KV head
    size_t workspace_bytes = 0;
};
// True when the kernel covers the call: T * group size <= 16, headDim ==
// vHeadDim == 128, no softcap, ALiBi or bias.  16-byte aligned q, k, v, out
// are checked at launch.
bool decode_tc_supported(const AttnDesc& a);
// `forced_splits` > 0 overrides the split count (at most one split per tile).
void decode_tc_plan(const AttnDesc& a, int forced_splits, int num_sms, DecodeTcPlan* tp);
// Launches the attention (which also writes the new rows of `cw` when given;
// its pointers must be 16-byte aligned) and the split merge.  `rope` (or
// NULL) turns q and the new keys inside the launch; the caches receive
// turned keys.
cudaError_t launch_decode_tc(const AttnDesc& a, const DecodeTcPlan& tp, void* workspace, cudaStream_t stream,
                             const DecodeCacheWrite* cw, const RopeDev* rope);
unsigned int decode_tc_take_device_error();

// ---- tiled prefill on FP32 FMA ----------------------------------------------
bool prefill_ffma_supported(const AttnDesc& a);
cudaError_t launch_prefill_ffma(const AttnDesc& a, const AlibiTable& alibi, cudaStream_t stream);

// ---- tcgen05 3xTF32 prefill ---------------------------------------------------
// headDim == vHeadDim in {32, 64, 96, 128}, q and out 16-byte aligned.
bool prefill_tc_supported(const AttnDesc& a);
// Scratch for the tf32 hi/lo copies of K and of V transposed.
size_t prefill_tc_workspace(const AttnDesc& a);
cudaError_t launch_prefill_tc(const AttnDesc& a, const AlibiTable& alibi, void* workspace, cudaStream_t stream);
unsigned int tc_take_device_error();

// ---- rope -----------------------------------------------------------------------
// out = rope(x) for x [T, H*D], row t at position offset + t; out may equal x.
cudaError_t launch_rope(const float* x, float* out, int64_t T, int H, int D, int64_t offset, const RopeDev& r,
                        cudaStream_t stream);

// ---- cache_write --------------------------------------------------------------
cudaError_t launch_cache_write(float* cache, int64_t width, const float* values, int64_t rows,
                               int64_t offset, cudaStream_t stream);

// ---- absorbed latent attention (mla_attention), decode form ------------------------
// The latent cache row is [latent (kMlaKvRank) | rotary key (kMlaRope)].
constexpr int kMlaKvRank = 512;
constexpr int kMlaRope = 64;
struct MlaDesc {
    const float* q;      // [T, H * (N + kMlaRope)]
    const float* state;  // [S, kMlaKvRank + kMlaRope] (first S rows read)
    const float* k_b;    // [H * N, kMlaKvRank]
    const float* v_b;    // [H * Dv, kMlaKvRank]
    float* out;          // [T, H * Dv]
    int64_t T, S;
    int32_t H, N, Dv;
    int32_t causal;
    int64_t pos_offset, window, sinks;
    float qscale;        // scale * log2 e, folded into the absorbed queries
    int32_t use_tc;      // scores on the tensor cores (mla_tc.cu); 0: CUDA cores only
};
// The new cache rows of a decode step (state_new == nullptr: none), written
// by the first launch: state[offset + r, :] = state_new[r, :].
struct MlaCacheWrite {
    float* state;
    const float* state_new;
    int64_t rows, offset;
};
struct MlaPlan {
    int32_t num_sms = 152;
    int32_t hq = 2;           // head quads per CTA (4 * hq virtual heads)
    int32_t groups = 1;       // CTAs per split (virtual heads / (4 * hq))
    int32_t splits = 1;
    int32_t sink_splits = 0;
    int64_t lo = 0, hi = 0, sink_end = 0, per = 32;
    size_t qabs_off = 0, qlo_off = 0, m_off = 0, l_off = 0, o_off = 0, olat_off = 0, workspace_bytes = 0;
};
// The tensor-core attention's split of the same key ranges into 128-row tiles.
constexpr int kMlaTcMaxSplits = 256;
struct MlaTcPlan {
    int32_t groups = 1;       // CTAs per split (16 virtual heads each)
    int32_t splits = 1;
    int32_t sink_splits = 0;
    int32_t n_sink_tiles = 0, n_tiles = 0;
};
void mla_tc_plan(const MlaDesc& m, const MlaPlan& base, int num_sms, MlaTcPlan* tp);
cudaError_t launch_mla_latent_tc(const MlaDesc& m, const MlaPlan& base, const MlaTcPlan& tp, const float* qhi,
                                 const float* qlo, float* part_m, float* part_l, float* part_o, cudaStream_t stream);
unsigned int mla_tc_take_device_error();
void mla_plan(const MlaDesc& m, int num_sms, MlaPlan* plan);
cudaError_t launch_mla(const MlaDesc& m, const MlaPlan& plan, void* workspace, const MlaCacheWrite& cw,
                       cudaStream_t stream);
unsigned int mla_take_device_error();

}  // namespace vtmu
