// decode.cu -- split-KV flash-decode kernel for one query row (T == 1).
//
// Op "attention" (vtmu.mpakt.dev/api/ops) with a KV cache: the single query
// row sits at position posOffset and the visible keys form one contiguous
// range [s_lo, s_end) of cache rows.  The work is HBM-bound: every K and V
// byte of that range is read once.  Layout of the work:
//
//  * grid (splits, kvHeads): one CTA streams a chunk of the range for one KV
//    head and serves all G = heads/kvHeads query heads of its group, so each
//    K/V byte is read once per group, not once per query head;
//  * K/V rows go global -> shared through a multi-stage cp.async ring (no
//    registers held by loads in flight; ~130-190 KB in flight per SM);
//  * a warp takes R = 32/G rows of a stage: lane l holds the query dims
//    {c*32*VEC + l*VEC + j}, computes R*G = 32 partial dot products, and a
//    5-step butterfly reduce-scatter over the warp leaves the full score of
//    (row l/G, head l%G) in lane l;
//  * fused epilogue (scale, softcap, ALiBi, bias) and online softmax in
//    base 2; the probabilities go through 128 bytes of shared memory to the
//    P.V step, where lane l owns value dims as it owns query dims;
//  * warps merge in shared memory, each CTA writes its (m, l, o) partials,
//    and the last CTA of a KV head (arrival counter, no waiting) merges the
//    splits with the log-sum-exp rule  m* = max m_i, l* = sum l_i 2^(m_i-m*),
//    o* = sum o_i 2^(m_i-m*) / l*  and writes the output row.
#include <cfloat>

#include "attn_common.cuh"
#include "kernels.h"

namespace vtmu {
namespace {

constexpr int kMaxSplits = 256;
constexpr size_t kSmemBudget = 200 * 1024;

struct DecodeArgs {
    AttnDesc a;
    int64_t s_lo;
    int64_t s_end;
    int64_t rows_per_split;
    int32_t splits;
    float* part_m;           // [heads][splits]
    float* part_l;           // [heads][splits]
    float* part_o;           // [heads][splits][Dv]
    unsigned int* counters;  // [kvHeads], zero between calls
};

template <int D, int G>
struct DecCfg {
    static constexpr int R = 32 / G;                   // rows per warp step
    static constexpr int NR = 64;                      // rows per stage
    static constexpr int WARPS = NR / R;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int VEC = (D % 128 == 0) ? 4 : ((D % 64 == 0) ? 2 : 1);
    static constexpr int NCH = D / (32 * VEC);         // chunks per row per lane
    static constexpr int PER_LANE = D / 32;            // dims per lane
    static constexpr int STAGE_FLOATS = 2 * NR * D;    // K and V of one stage
    static constexpr int STAGES_FIT = (int)(kSmemBudget / (STAGE_FLOATS * sizeof(float)));
    static constexpr int STAGES = STAGES_FIT > 4 ? 4 : STAGES_FIT;
    static constexpr size_t SMEM = (size_t)STAGES * STAGE_FLOATS * sizeof(float);
    static_assert(STAGES >= 2, "decode stage does not fit twice in shared memory");
    static_assert(D % 32 == 0 && 32 % G == 0, "unsupported decode shape");
};

template <int VEC>
__device__ __forceinline__ void lds_vec(float* dst, const float* src) {
    if constexpr (VEC == 4) {
        float4 t = *reinterpret_cast<const float4*>(src);
        dst[0] = t.x; dst[1] = t.y; dst[2] = t.z; dst[3] = t.w;
    } else if constexpr (VEC == 2) {
        float2 t = *reinterpret_cast<const float2*>(src);
        dst[0] = t.x; dst[1] = t.y;
    } else {
        dst[0] = *src;
    }
}

// G consecutive shared-memory floats (16-byte aligned when G >= 4).
template <int G>
__device__ __forceinline__ void load_group(float* dst, const float* src) {
    if constexpr (G % 4 == 0) {
#pragma unroll
        for (int i = 0; i < G / 4; ++i) lds_vec<4>(dst + 4 * i, src + 4 * i);
    } else if constexpr (G == 2) {
        lds_vec<2>(dst, src);
    } else {
#pragma unroll
        for (int i = 0; i < G; ++i) dst[i] = src[i];
    }
}

// Lane-owned dim j (0 <= j < D/32) of chunked layout.
template <int VEC>
__device__ __forceinline__ int lane_dim(int lane, int j) {
    return (j / VEC) * 32 * VEC + lane * VEC + (j % VEC);
}

template <int D, int G>
__global__ void __launch_bounds__(DecCfg<D, G>::THREADS, 1)
    decode_splitkv_kernel(const DecodeArgs args, const AlibiTable alibi) {
    using C = DecCfg<D, G>;
    constexpr int R = C::R, NR = C::NR, VEC = C::VEC, PL = C::PER_LANE;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(16) float smem[];
    __shared__ __align__(16) float pbuf[C::WARPS][32];
    __shared__ int s_is_last;

    const AttnDesc& a = args.a;
    const int split = blockIdx.x;
    const int kh = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t p = a.pos_offset;  // position of the single query row
    const int64_t ldk = (int64_t)a.Hk * D;

    const int64_t c_begin = args.s_lo + (int64_t)split * args.rows_per_split;
    int64_t c_end = c_begin + args.rows_per_split;
    if (c_end > args.s_end) c_end = args.s_end;
    const int64_t n_rows = c_end > c_begin ? c_end - c_begin : 0;
    const int n_stages = (int)((n_rows + NR - 1) / NR);

    // Query dims owned by this lane, for every head of the group (the
    // score scale is applied in the epilogue).
    float qv[G][PL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float* qh = a.q + (int64_t)(kh * G + g) * D;
#pragma unroll
        for (int j = 0; j < PL; ++j) qv[g][j] = __ldg(qh + lane_dim<VEC>(lane, j));
    }
    // This lane's score slot: row rr of the warp's rows, head gg of the group.
    const int rr = lane / G;
    const int gg = lane % G;
    const int h_lane = kh * G + gg;
    const float slope_lane = a.alibi_on ? alibi.slope_log2[h_lane] : 0.f;

    float m_run = -INFINITY;  // per head gg (equal across lanes of the head)
    float l_run = 0.f;        // this lane's share of the head's sum
    float o[G][PL];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < PL; ++j) o[g][j] = 0.f;

    // ---- stage loader: NR rows of K then NR rows of V, 16-byte cp.async ----
    auto load_stage = [&](int st) {
        float* sk = smem + (st % C::STAGES) * C::STAGE_FLOATS;
        float* sv = sk + NR * D;
        const int64_t r0 = c_begin + (int64_t)st * NR;
        constexpr int CHUNKS = NR * D / 4;
        for (int c = threadIdx.x; c < CHUNKS; c += C::THREADS) {
            const int row = c / (D / 4);
            const int col = (c % (D / 4)) * 4;
            const int64_t s = r0 + row;
            const bool ok = s < c_end;
            const int64_t off = (ok ? s : c_begin) * ldk + (int64_t)kh * D + col;
            cp_async16(sk + row * D + col, a.k + off, ok ? 16 : 0);
            cp_async16(sv + row * D + col, a.v + off, ok ? 16 : 0);
        }
    };

#pragma unroll
    for (int st = 0; st < C::STAGES - 1; ++st) {
        if (st < n_stages) load_stage(st);
        cp_async_commit();
    }

    for (int st = 0; st < n_stages; ++st) {
        cp_async_wait<C::STAGES - 2>();
        __syncthreads();  // stage st visible to all; stage st-1 fully consumed
        if (st + C::STAGES - 1 < n_stages) load_stage(st + C::STAGES - 1);
        cp_async_commit();

        const float* sk = smem + (st % C::STAGES) * C::STAGE_FLOATS + warp * R * D;
        const float* sv = sk + NR * D;

        // 32 partial dot products: slot r*G + g.
        float part[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) part[i] = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
                float kv[VEC];
                lds_vec<VEC>(kv, sk + r * D + c * 32 * VEC + lane * VEC);
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        part[r * G + g] = fmaf(qv[g][c * VEC + j], kv[j], part[r * G + g]);
            }
        }
        // Butterfly reduce-scatter: after step `o` a lane keeps the half of
        // its slots whose bit `o` matches its own lane bit.
#pragma unroll
        for (int step = 0; step < 5; ++step) {
            const int off = 16 >> step;
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < off; ++i) {
                const float send = upper ? part[i] : part[i + off];
                const float keep = upper ? part[i + off] : part[i];
                part[i] = keep + __shfl_xor_sync(FULL, send, off);
            }
        }

        // Fused epilogue for (row rr, head gg).
        const int64_t s = c_begin + (int64_t)st * NR + warp * R + rr;
        float x = -INFINITY;
        if (s < c_end) {
            const float bv = a.bias_kind ? bias_at(a, h_lane, 0, s) : 0.f;
            x = score_log2(a, part[0], slope_lane, s - p, bv);
        }
        // Online softmax per head: max over the R rows of the head.
        float mt = x;
#pragma unroll
        for (int off = G; off < 32; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, off));
        const float m_new = fmaxf(m_run, mt);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = exp2f(m_run - m_use);
        const float pr = exp2f(x - m_use);
        l_run = fmaf(l_run, alpha, pr);
        m_run = m_new;
        pbuf[warp][lane] = pr;
        __syncwarp();
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float ag = __shfl_sync(FULL, alpha, g);  // lane g serves head g
#pragma unroll
            for (int j = 0; j < PL; ++j) o[g][j] *= ag;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float pw[G];
            load_group<G>(pw, &pbuf[warp][r * G]);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c) {
                float vv[VEC];
                lds_vec<VEC>(vv, sv + r * D + c * 32 * VEC + lane * VEC);
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int j = 0; j < VEC; ++j)
                        o[g][c * VEC + j] = fmaf(pw[g], vv[j], o[g][c * VEC + j]);
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();

    // ---- merge the warps of this CTA -------------------------------------
#pragma unroll
    for (int off = G; off < 32; off <<= 1) l_run += __shfl_xor_sync(FULL, l_run, off);
    __syncthreads();  // every warp is done with the stage buffers
    float* wm = smem;                      // [WARPS][G]
    float* wl = wm + C::WARPS * G;         // [WARPS][G]
    float* wo = wl + C::WARPS * G;         // [WARPS][G][D]
    if (lane < G) {
        wm[warp * G + lane] = m_run;
        wl[warp * G + lane] = l_run;
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < PL; ++j) wo[(warp * G + g) * D + lane_dim<VEC>(lane, j)] = o[g][j];
    __syncthreads();

    const int Hs = args.splits;
    for (int idx = threadIdx.x; idx < G * D; idx += C::THREADS) {
        const int g = idx / D, e = idx % D;
        float M = -INFINITY;
#pragma unroll 4
        for (int w = 0; w < C::WARPS; ++w) M = fmaxf(M, wm[w * G + g]);
        const float mu = (M == -INFINITY) ? 0.f : M;
        float acc = 0.f, L = 0.f;
        for (int w = 0; w < C::WARPS; ++w) {
            const float sc = exp2f(wm[w * G + g] - mu);
            acc = fmaf(wo[(w * G + g) * D + e], sc, acc);
            L = fmaf(wl[w * G + g], sc, L);
        }
        const int h = kh * G + g;
        args.part_o[((int64_t)h * Hs + split) * D + e] = acc;
        if (e == 0) {
            args.part_m[(int64_t)h * Hs + split] = M;
            args.part_l[(int64_t)h * Hs + split] = L;
        }
    }

    // ---- last CTA of this KV head merges the splits ----------------------
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned ticket = atomicAdd(&args.counters[kh], 1u);
        s_is_last = (ticket == (unsigned)(Hs - 1));
    }
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();

    float* sw = smem;            // [G][kMaxSplits] split weights
    float* sinv = sw + G * kMaxSplits;  // [G] 1 / l*
    for (int g = warp; g < G; g += C::WARPS) {
        const int h = kh * G + g;
        float M = -INFINITY;
        for (int i = lane; i < Hs; i += 32) M = fmaxf(M, __ldcg(args.part_m + (int64_t)h * Hs + i));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, off));
        const float mu = (M == -INFINITY) ? 0.f : M;
        float L = 0.f;
        for (int i = lane; i < Hs; i += 32) {
            const float w = exp2f(__ldcg(args.part_m + (int64_t)h * Hs + i) - mu);
            sw[g * kMaxSplits + i] = w;
            L = fmaf(__ldcg(args.part_l + (int64_t)h * Hs + i), w, L);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(FULL, L, off);
        if (lane == 0) sinv[g] = (L > 0.f) ? 1.f / L : 0.f;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * D; idx += C::THREADS) {
        const int g = idx / D, e = idx % D;
        const int h = kh * G + g;
        const float* po = args.part_o + (int64_t)h * Hs * D + e;
        float acc = 0.f;
#pragma unroll 8
        for (int i = 0; i < Hs; ++i) acc = fmaf(__ldcg(po + (int64_t)i * D), sw[g * kMaxSplits + i], acc);
        a.out[(int64_t)h * D + e] = acc * sinv[g];
    }
    if (threadIdx.x == 0) args.counters[kh] = 0u;  // ready for the next call
}

template <int D, int G>
cudaError_t launch_cfg(const DecodeArgs& args, const AlibiTable& alibi, cudaStream_t stream) {
    using C = DecCfg<D, G>;
    auto kern = decode_splitkv_kernel<D, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(args.splits, args.a.Hk);
    kern<<<grid, C::THREADS, C::SMEM, stream>>>(args, alibi);
    return cudaGetLastError();
}

int stage_rows() { return 64; }

}  // namespace

bool decode_supported(const AttnDesc& a) {
    if (a.T != 1 || a.D != a.Dv) return false;
    if (!(a.D == 32 || a.D == 64 || a.D == 128)) return false;
    if (!(a.G == 2 || a.G == 4 || a.G == 8)) return false;
    return true;
}

void decode_plan(const AttnDesc& a, int forced_splits, int num_sms, DecodePlan* plan) {
    // Visible keys of the single row form one range (causal: s <= p; causal
    // window: s > p - w; non-causal window: |p - s| <= w).
    const int64_t p = a.pos_offset;
    int64_t lo = 0, hi = a.S;  // [lo, hi)
    if (a.causal) {
        hi = p + 1 < hi ? p + 1 : hi;
        if (a.window > 0) lo = p - a.window + 1;
    } else if (a.window > 0) {
        lo = p - a.window;
        hi = p + a.window + 1 < hi ? p + a.window + 1 : hi;
    }
    if (lo < 0) lo = 0;
    if (hi < lo) hi = lo;
    const int64_t rows = hi - lo;
    const int nr = stage_rows();
    int splits = forced_splits;
    if (splits <= 0) {
        // One CTA per SM: split each KV head's range into ~num_sms/Hk chunks.
        splits = (num_sms + a.Hk - 1) / a.Hk;
        if (splits < 1) splits = 1;
    }
    if (splits > kMaxSplits) splits = kMaxSplits;
    const int64_t min_rows = nr;
    int64_t per = (rows + splits - 1) / splits;
    if (per < min_rows) per = min_rows;
    per = (per + nr - 1) / nr * nr;
    int64_t n = rows > 0 ? (rows + per - 1) / per : 1;
    plan->s_lo = lo;
    plan->s_end = hi;
    plan->rows_per_split = per;
    plan->splits = (int32_t)n;
    const size_t H = (size_t)a.H, Sp = (size_t)n;
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    // Arrival counters first (fixed place, so they stay zero between calls
    // of any shape), then m, l and o partials.
    plan->workspace_bytes = up((size_t)a.Hk * 4) + up(H * Sp * 4) * 2 + up(H * Sp * (size_t)a.Dv * 4);
}

cudaError_t launch_decode(const AttnDesc& a, const AlibiTable& alibi, const DecodePlan& plan,
                          void* workspace, cudaStream_t stream) {
    DecodeArgs args;
    args.a = a;
    args.s_lo = plan.s_lo;
    args.s_end = plan.s_end;
    args.rows_per_split = plan.rows_per_split;
    args.splits = plan.splits;
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t H = (size_t)a.H, Sp = (size_t)plan.splits;
    char* w = static_cast<char*>(workspace);
    args.counters = reinterpret_cast<unsigned int*>(w);
    w += up((size_t)a.Hk * 4);
    args.part_m = reinterpret_cast<float*>(w);
    args.part_l = reinterpret_cast<float*>(w + up(H * Sp * 4));
    args.part_o = reinterpret_cast<float*>(w + 2 * up(H * Sp * 4));
#define VTMU_DEC(D_, G_) \
    if (a.D == D_ && a.G == G_) return launch_cfg<D_, G_>(args, alibi, stream);
    VTMU_DEC(32, 2) VTMU_DEC(32, 4) VTMU_DEC(32, 8)
    VTMU_DEC(64, 2) VTMU_DEC(64, 4) VTMU_DEC(64, 8)
    VTMU_DEC(128, 2) VTMU_DEC(128, 4) VTMU_DEC(128, 8)
#undef VTMU_DEC
    return cudaErrorInvalidValue;
}

}  // namespace vtmu
