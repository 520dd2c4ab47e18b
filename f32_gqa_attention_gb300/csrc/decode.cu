// decode.cu -- split-KV flash-decode kernel for a few query rows (1 <= T <= 16).
//
// Op "attention" (vtmu.mpakt.dev/api/ops) with a KV cache: query row t sits
// at position posOffset + t and the keys any row sees form one contiguous
// range [s_lo, s_end) of cache rows.  The work is HBM-bound: every K and V
// byte of that range is read once per row group.  Layout of the work:
//
//  * the kernel's G "heads" are virtual heads: the group's query heads times
//    the query rows of a row group (tc rows, G = group size x tc <= 8, padded
//    to 2), so one K/V tile serves every query row and head of its group;
//    each row masks the keys of the range it cannot see.  T = 1 is the
//    common decode step; 1 < T is a speculative or chunked step;
//  * grid (kvHeads, splits, row groups): one CTA streams a chunk of the range
//    for one KV head and serves all virtual heads of its group, so each K/V
//    byte is read once per row group, not once per query head;
//  * a producer warp moves NR-row K and V tiles global -> shared with 2-D TMA
//    (cp.async.bulk.tensor) into a ring of stages guarded by full/empty
//    mbarriers; the consumer warps never issue a load;
//  * a consumer warp takes R = 32/G rows of a stage.  Lane l holds the query
//    dims {c*32*VEC + l*VEC + j}; it computes 32 partial dot products, and a
//    5-step butterfly reduce-scatter over the warp leaves the full score of
//    (row l/G, head l%G) in lane l.  Lane l stores its partials at slot
//    index (logical slot XOR l) -- it reads the K row and the query head that
//    the XOR names -- so every butterfly step is a plain shuffle-and-add with
//    no selects;
//  * fused epilogue (scale, softcap, ALiBi, bias) and online softmax in base
//    2 (rescaling skipped when no running max moved); the probabilities go
//    through 128 bytes of shared memory to the P.V step, where lane l owns
//    value dims as it owns query dims;
//  * warps merge in shared memory, each CTA writes its (m, l, o) partials,
//    and the last CTA of a (KV head, row group) (arrival counter, no waiting) merges the
//    splits with the log-sum-exp rule  m* = max m_i, l* = sum l_i 2^(m_i-m*),
//    o* = sum o_i 2^(m_i-m*) / l*  and writes the output row.
//
// Every mbarrier wait is bounded (see tma_sync.cuh); a wait that gives up
// sets a bit of g_decode_device_error and the kernel unwinds.
#include <cfloat>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_common.cuh"
#include "kernels.h"
#include "launch_cache.h"
#include "rope.cuh"
#include "tma_sync.cuh"

namespace vtmu {

__device__ unsigned int g_decode_device_error;

namespace {

// Stage geometry (compile-time; the defaults are the tuned configuration).
#ifndef VTMU_DEC_NR
#define VTMU_DEC_NR 64  // K/V rows per shared-memory stage
#endif
#ifndef VTMU_DEC_SMEM_KB
#define VTMU_DEC_SMEM_KB 200  // shared-memory budget of one CTA's stage ring
#endif
#ifndef VTMU_DEC_MAX_STAGES
#define VTMU_DEC_MAX_STAGES 4
#endif
#ifndef VTMU_DEC_CTAS_PER_SM
#define VTMU_DEC_CTAS_PER_SM 1  // resident CTAs per SM the split count aims for
#endif
#ifndef VTMU_DEC_KH_FAST
#define VTMU_DEC_KH_FAST 1  // 1: the KV heads of one split are adjacent CTAs
#endif

constexpr int kMaxSplits = 256;
constexpr size_t kSmemBudget = (size_t)VTMU_DEC_SMEM_KB * 1024;

struct DecodeArgs {
    AttnDesc a;
    int64_t s_lo;
    int64_t s_end;
    int64_t rows_per_split;
    int64_t sink_end;        // attention sinks: rows [0, sink_end) are a range of their own
    int32_t sink_splits;     // splits [0, sink_splits) stream the sink range
    int32_t splits;
    float* part_m;           // [heads][splits]
    float* part_l;           // [heads][splits]
    float* part_o;           // [heads][splits][Dv]
    unsigned int* counters;  // [kvHeads], zero between calls
    DecodeCacheWrite cw;     // fused cache_write (cw.k_new == nullptr: none)
    RopeDev rope;            // rotary embedding of q and the new keys (rope.half == 0: none)
    // Query rows: the kernel's G "heads" are virtual heads vh = t_local * gr + g
    // (row t_local of this CTA's row group, query head kh * gr + g), tc query
    // rows per row group, one row group per blockIdx.z.
    int32_t gr;              // heads per KV head (group size)
    int32_t tc;              // query rows per row group
};

// Query row and head of virtual head vh of KV head kh in this CTA's row group;
// `ok` is false for padding (past T, or past the row group).
struct VHead {
    int64_t t;
    int h;
    bool ok;
};
__device__ __forceinline__ VHead vhead(const DecodeArgs& args, int kh, int vh) {
    const int tl = vh / args.gr;
    VHead r;
    r.t = (int64_t)blockIdx.z * args.tc + tl;
    r.h = kh * args.gr + vh % args.gr;
    r.ok = tl < args.tc && r.t < args.a.T;
    return r;
}

// Element d of new key row `pos` (k_new row base `src`), turned by the rotary
// embedding when it is on: the cache stores turned keys.
__device__ __forceinline__ float new_key(const DecodeArgs& args, int64_t src, int d, int64_t pos) {
    const float own = __ldg(args.cw.k_new + src + d);
    if (d >= 2 * args.rope.half) return own;
    int j, partner;
    bool first;
    rope_pair_of(args.rope, d, j, partner, first);
    return rope_channel(own, __ldg(args.cw.k_new + src + partner), first, rope_cos_sin(args.rope, pos, j));
}

template <int D, int G>
struct DecCfg {
    static constexpr int R = 32 / G;                   // rows per warp step
    // Rows per stage: VTMU_DEC_NR, but at most 8 consumer warps' worth (the
    // split size is a multiple of VTMU_DEC_NR, hence of NR).
    static constexpr int NR = VTMU_DEC_NR < 8 * R ? VTMU_DEC_NR : 8 * R;
    static constexpr int WARPS = NR / R;               // consumer warps
    static constexpr int THREADS = (WARPS + 1) * 32;   // + one producer warp
    static constexpr int VEC = (D % 128 == 0) ? 4 : ((D % 64 == 0) ? 2 : 1);
    static constexpr int NCH = D / (32 * VEC);         // chunks per row per lane
    static constexpr int PER_LANE = D / 32;            // dims per lane
    static constexpr int TILE_FLOATS = NR * D;         // one K (or V) tile
    static constexpr int STAGE_FLOATS = 2 * TILE_FLOATS;
    static constexpr uint32_t STAGE_BYTES = STAGE_FLOATS * sizeof(float);
    static constexpr int STAGES_FIT = (int)(kSmemBudget / STAGE_BYTES);
    static constexpr int STAGES = STAGES_FIT > VTMU_DEC_MAX_STAGES ? VTMU_DEC_MAX_STAGES : STAGES_FIT;
    static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES;
    static_assert(STAGES >= 2, "decode stage does not fit twice in shared memory");
    static_assert(NR % R == 0 && NR <= 256, "a stage must hold whole warp steps, <= 256 TMA rows");
    static_assert(D % 32 == 0 && 32 % G == 0 && D <= 256, "unsupported decode shape");
    // The warp merge and the split merge reuse the stage ring.
    static_assert(WARPS * G * (2 + D) <= STAGES * STAGE_FLOATS, "merge area exceeds the stage ring");
    static_assert(G * (kMaxSplits + 1) <= STAGES * STAGE_FLOATS, "split weights exceed the stage ring");
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

// Lane-owned dim j (0 <= j < D/32) of the chunked layout.
template <int VEC>
__device__ __forceinline__ int lane_dim(int lane, int j) {
    return (j / VEC) * 32 * VEC + lane * VEC + (j % VEC);
}

template <int D, int G>
__global__ void __launch_bounds__(DecCfg<D, G>::THREADS, VTMU_DEC_CTAS_PER_SM)
    decode_splitkv_kernel(const DecodeArgs args, const AlibiTable alibi, const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv) {
    using C = DecCfg<D, G>;
    constexpr int R = C::R, NR = C::NR, VEC = C::VEC, PL = C::PER_LANE, STAGES = C::STAGES;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(1024) float smem[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(16) float pbuf[C::WARPS][32];
    __shared__ int s_is_last;
    __shared__ float2 q_cs[D / 2];  // rotary (cos, sin) of the query row, per pair

    const AttnDesc& a = args.a;
    const int split = VTMU_DEC_KH_FAST ? blockIdx.y : blockIdx.x;
    const int kh = VTMU_DEC_KH_FAST ? blockIdx.x : blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t p = a.pos_offset;  // position of query row 0 (row t sits at p + t)

    const bool sink_split = split < args.sink_splits;
    const int64_t c_begin = sink_split ? (int64_t)split * args.rows_per_split
                                       : args.s_lo + (int64_t)(split - args.sink_splits) * args.rows_per_split;
    int64_t c_end = c_begin + args.rows_per_split;
    const int64_t c_cap = sink_split ? args.sink_end : args.s_end;
    if (c_end > c_cap) c_end = c_cap;
    const int n_rows = c_end > c_begin ? (int)(c_end - c_begin) : 0;
    const int n_stages = (n_rows + NR - 1) / NR;

    if (threadIdx.x == 0) {
        for (int b = 0; b < STAGES; ++b) {
            mbar_init(&full_bar[b], 1);
            mbar_init(&empty_bar[b], C::WARPS);
        }
        fence_barrier_init();
    }
    // Fused cache_write, rows no split reads: written by split 0 of each KV
    // head (its own columns).  Rows inside the visible range are written by
    // the consumer warp that owns them, below.
    const int64_t ld = (int64_t)a.Hk * D;
    if (args.cw.k_new && split == 0 && blockIdx.z == 0 && warp == 0) {
        for (int64_t r = args.cw.lo; r < args.cw.hi; ++r) {
            if ((r >= args.s_lo && r < args.s_end) || r < args.sink_end) continue;
            const int64_t src = (r - args.cw.lo) * ld + (int64_t)kh * D, dst = r * ld + (int64_t)kh * D;
            for (int d = lane; d < D; d += 32) {
                args.cw.kc[dst + d] = new_key(args, src, d, r);
                args.cw.vc[dst + d] = __ldg(args.cw.v_new + src + d);
            }
        }
    }
    for (int j = threadIdx.x; j < args.rope.half; j += blockDim.x) q_cs[j] = rope_cos_sin(args.rope, p, j);
    __syncthreads();

    float m_run = -INFINITY;  // running max of head lane%G (base 2)
    float l_run = 0.f;        // this lane's share of that head's sum
    float o[G][PL];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < PL; ++j) o[g][j] = 0.f;

    if (warp == C::WARPS) {
        // ---------------- producer: one thread issues every TMA ------------
        if (lane == 0 && n_stages > 0) {
            prefetch_tensormap(&tmk);
            prefetch_tensormap(&tmv);
            int issued = 0;
            for (int st = 0; st < n_stages; ++st) {
                const int b = st % STAGES;
                if (st >= STAGES && !mbar_wait(&empty_bar[b], ((st / STAGES) - 1) & 1)) {
                    raise_device_error(&g_decode_device_error, kErrDecodeEmptyWait);
                    break;
                }
                float* sk = smem + b * C::STAGE_FLOATS;
                mbar_arrive_expect_tx(&full_bar[b], C::STAGE_BYTES);
                const int row = (int)(c_begin + (int64_t)st * NR);
                tma_load_2d(sk, &tmk, kh * D, row, &full_bar[b]);
                tma_load_2d(sk + C::TILE_FLOATS, &tmv, kh * D, row, &full_bar[b]);
                ++issued;
            }
            // Drain: every copy issued has landed before the ring is reused.
            for (int st = issued > STAGES ? issued - STAGES : 0; st < issued; ++st)
                if (!mbar_wait(&full_bar[st % STAGES], (st / STAGES) & 1)) {
                    raise_device_error(&g_decode_device_error, kErrDecodeDrainWait);
                    break;
                }
        }
    } else {
        // ---------------- consumers ----------------------------------------
        // Query dims owned by this lane.  Slot gi holds head gi ^ (lane % G).
        float qv[G][PL];
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            const VHead vq = vhead(args, kh, gi ^ (lane % G));
            const float* qh = a.q + (vq.t * a.H + vq.h) * D;  // read only when vq.ok
#pragma unroll
            for (int j = 0; j < PL; ++j) {
                const int d = lane_dim<VEC>(lane, j);
                float x = vq.ok ? __ldg(qh + d) : 0.f;
                if (vq.ok && d < 2 * args.rope.half) {
                    int pj, partner;
                    bool first;
                    rope_pair_of(args.rope, d, pj, partner, first);
                    x = rope_channel(x, __ldg(qh + partner), first, q_cs[pj]);
                }
                qv[gi][j] = x;
            }
        }
        const int rr = lane / G;  // logical slot after the butterfly: row rr, virtual head gg
        const int gg = lane % G;
        const VHead vl = vhead(args, kh, gg);
        const float slope_lane = a.alibi_on ? alibi.slope_log2[vl.h] : 0.f;
        const float* bias_row = (a.bias_kind == 0 || !vl.ok) ? nullptr
                                : a.bias_kind == 1          ? a.bias + vl.t * a.S + c_begin
                                                            : a.bias + ((int64_t)vl.h * a.T + vl.t) * a.S + c_begin;
        const int64_t p_lane = p + vl.t;  // position of this lane's query row
        const int64_t rel0 = c_begin - p_lane;
        // With several query rows the key range is their union: each row
        // masks the keys it cannot see.
        const bool multi = a.T > 1;
        const int rowx = lane / G;  // slot ri reads warp row ri ^ rowx

        for (int st = 0; st < n_stages; ++st) {
            const int b = st % STAGES;
            if (!mbar_wait(&full_bar[b], (st / STAGES) & 1)) {
                raise_device_error(&g_decode_device_error, kErrDecodeFullWait);
                break;
            }
            float* skw = smem + b * C::STAGE_FLOATS + warp * R * D;
            if (args.cw.k_new) {
                // Fused cache_write of rows this warp owns: the new values go
                // to the cache and replace the staged (old) rows.
                const int64_t row0 = c_begin + (int64_t)st * NR + warp * R;
                int64_t lo = row0 > args.cw.lo ? row0 : args.cw.lo;
                int64_t hi = row0 + R < args.cw.hi ? row0 + R : args.cw.hi;
                if (hi > c_end) hi = c_end;
                if (lo < hi) {
                    for (int64_t r = lo; r < hi; ++r) {
                        float* skr = skw + (int)(r - row0) * D;
                        float* svr = skr + C::TILE_FLOATS;
                        const int64_t src = (r - args.cw.lo) * ld + (int64_t)kh * D, dst = r * ld + (int64_t)kh * D;
#pragma unroll
                        for (int j = 0; j < PL; ++j) {
                            const int d = lane_dim<VEC>(lane, j);
                            const float kx = new_key(args, src, d, r);
                            const float vx = __ldg(args.cw.v_new + src + d);
                            skr[d] = kx;
                            svr[d] = vx;
                            if (blockIdx.z == 0) {  // one row group writes the cache
                                args.cw.kc[dst + d] = kx;
                                args.cw.vc[dst + d] = vx;
                            }
                        }
                    }
                    // Order these generic-proxy writes before the TMA that
                    // refills the stage later.
                    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                    __syncwarp();
                }
            }
            const float* sk = skw;
            const float* sv = sk + C::TILE_FLOATS;

            // 32 partial dot products; slot ri*G + gi = (row ri^rowx, head gi^(lane%G)).
            float part[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) part[i] = 0.f;
#pragma unroll
            for (int ri = 0; ri < R; ++ri) {
                const float* krow = sk + (ri ^ rowx) * D + lane * VEC;
#pragma unroll
                for (int c = 0; c < C::NCH; ++c) {
                    float kv[VEC];
                    lds_vec<VEC>(kv, krow + c * 32 * VEC);
#pragma unroll
                    for (int gi = 0; gi < G; ++gi)
#pragma unroll
                        for (int j = 0; j < VEC; ++j)
                            part[ri * G + gi] = fmaf(qv[gi][c * VEC + j], kv[j], part[ri * G + gi]);
                }
            }
            // Reduce-scatter: lane L's slot i holds logical slot i ^ L, so each
            // step keeps the low half and adds the partner's high half.
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
                for (int i = 0; i < off; ++i) part[i] += __shfl_xor_sync(FULL, part[i + off], off);

            // Fused epilogue for (row rr, head gg).
            const int row_l = st * NR + warp * R + rr;
            float x = -INFINITY;
            if (row_l < n_rows && vl.ok && (!multi || key_visible(a, p_lane, c_begin + row_l))) {
                const float bv = bias_row ? __ldg(bias_row + row_l) : 0.f;
                x = score_log2(a, part[0], slope_lane, rel0 + row_l, bv);
            }
            // Online softmax per head: max over the R rows of the head.
            float mt = x;
#pragma unroll
            for (int off = G; off < 32; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, off));
            const float m_new = fmaxf(m_run, mt);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = fast_exp2(m_run - m_use);
            const float pr = fast_exp2(x - m_use);
            l_run = fmaf(l_run, alpha, pr);
            m_run = m_new;
            pbuf[warp][lane] = pr;
            if (!__all_sync(FULL, alpha == 1.f)) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float ag = __shfl_sync(FULL, alpha, g);  // lane g serves head g
#pragma unroll
                    for (int j = 0; j < PL; ++j) o[g][j] *= ag;
                }
            }
            __syncwarp();
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
            if (lane == 0) mbar_arrive(&empty_bar[b]);  // this warp is done with stage b
        }
#pragma unroll
        for (int off = G; off < 32; off <<= 1) l_run += __shfl_xor_sync(FULL, l_run, off);
    }

    // ---- merge the warps of this CTA -------------------------------------
    __syncthreads();  // all copies landed (producer drained) and all stages consumed
    float* wm = smem;                      // [WARPS][G]
    float* wl = wm + C::WARPS * G;         // [WARPS][G]
    float* wo = wl + C::WARPS * G;         // [WARPS][G][D]
    if (warp < C::WARPS) {
        if (lane < G) {
            wm[warp * G + lane] = m_run;
            wl[warp * G + lane] = l_run;
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int j = 0; j < PL; ++j) wo[(warp * G + g) * D + lane_dim<VEC>(lane, j)] = o[g][j];
    }
    __syncthreads();

    const int Hs = args.splits;
    const int64_t vbase = ((int64_t)blockIdx.z * a.Hk + kh) * G;  // this CTA's virtual heads in the partials
    for (int idx = threadIdx.x; idx < G * D; idx += C::THREADS) {
        const int g = idx / D, e = idx % D;
        float M = -INFINITY;
        for (int w = 0; w < C::WARPS; ++w) M = fmaxf(M, wm[w * G + g]);
        const float mu = (M == -INFINITY) ? 0.f : M;
        float acc = 0.f, L = 0.f;
        for (int w = 0; w < C::WARPS; ++w) {
            const float sc = fast_exp2(wm[w * G + g] - mu);
            acc = fmaf(wo[(w * G + g) * D + e], sc, acc);
            L = fmaf(wl[w * G + g], sc, L);
        }
        const int64_t h = vbase + g;
        args.part_o[((int64_t)h * Hs + split) * D + e] = acc;
        if (e == 0) {
            args.part_m[(int64_t)h * Hs + split] = M;
            args.part_l[(int64_t)h * Hs + split] = L;
        }
    }

    // ---- last CTA of this KV head merges the splits ----------------------
    // Release: the barrier orders every thread's partial stores before
    // thread 0's ticket, whose gpu-scope release publishes them.
    __syncthreads();
    if (threadIdx.x == 0) {
        // One acquire-release atomic: releases this CTA's partials (ordered
        // before it by the barrier) and, for the last CTA, acquires the other
        // splits' (measured ~0.9 us faster per step than two full fences).
        unsigned ticket;
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;"
                     : "=r"(ticket)
                     : "l"(&args.counters[blockIdx.z * a.Hk + kh])
                     : "memory");
        const bool last = (ticket == (unsigned)(Hs - 1));
        s_is_last = last;
    }
    __syncthreads();
    if (!s_is_last) return;

    // Thread t owns outputs t + k*THREADS (k < NOUT).  It issues the loads of
    // its first CH split partials before the warps turn the virtual heads'
    // split maxima into weights, so both L2 round trips overlap.
    constexpr int NOUT = (G * D + C::THREADS - 1) / C::THREADS;
    constexpr int CH = 64 / NOUT > 32 ? 32 : (64 / NOUT < 8 ? 8 : 64 / NOUT);
    float ov[NOUT][CH];
    auto load_chunk = [&](int i0) {
#pragma unroll
        for (int k = 0; k < NOUT; ++k) {
            const int idx = threadIdx.x + k * C::THREADS;
            const int64_t base = idx < G * D ? ((vbase + idx / D) * Hs) * D + idx % D : 0;
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                const int i = i0 + c;
                ov[k][c] = (idx < G * D && i < Hs) ? __ldcg(args.part_o + base + (int64_t)i * D) : 0.f;
            }
        }
    };
    load_chunk(0);

    float* sw = smem;                   // [G][kMaxSplits] split weights
    float* sinv = sw + G * kMaxSplits;  // [G] 1 / l*
    // Warp w serves virtual heads w, w + warps, ... (one each when G <= warps).
    for (int gw = warp; gw < G; gw += C::THREADS / 32) {
        const int64_t h = vbase + gw;
        constexpr int PER = kMaxSplits / 32;
        float mv[PER], lv[PER];
#pragma unroll
        for (int t = 0; t < PER; ++t) {
            const int i = lane + 32 * t;
            mv[t] = i < Hs ? __ldcg(args.part_m + (int64_t)h * Hs + i) : -INFINITY;
            lv[t] = i < Hs ? __ldcg(args.part_l + (int64_t)h * Hs + i) : 0.f;
        }
        float M = -INFINITY;
#pragma unroll
        for (int t = 0; t < PER; ++t) M = fmaxf(M, mv[t]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, off));
        const float mu = (M == -INFINITY) ? 0.f : M;
        float L = 0.f;
#pragma unroll
        for (int t = 0; t < PER; ++t) {
            const float w = fast_exp2(mv[t] - mu);
            if (lane + 32 * t < Hs) sw[gw * kMaxSplits + lane + 32 * t] = w;
            L = fmaf(lv[t], w, L);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(FULL, L, off);
        if (lane == 0) sinv[gw] = (L > 0.f) ? 1.f / L : 0.f;
    }
    __syncthreads();

    float acc[NOUT];
#pragma unroll
    for (int k = 0; k < NOUT; ++k) acc[k] = 0.f;
    for (int i0 = 0;;) {
#pragma unroll
        for (int k = 0; k < NOUT; ++k) {
            const int idx = threadIdx.x + k * C::THREADS;
            const float* wg = sw + (idx < G * D ? idx / D : 0) * kMaxSplits + i0;
#pragma unroll
            for (int c = 0; c < CH; ++c)
                if (i0 + c < Hs) acc[k] = fmaf(ov[k][c], wg[c], acc[k]);
        }
        i0 += CH;
        if (i0 >= Hs) break;
        load_chunk(i0);
    }
#pragma unroll
    for (int k = 0; k < NOUT; ++k) {
        const int idx = threadIdx.x + k * C::THREADS;
        if (idx < G * D) {
            const VHead vo = vhead(args, kh, idx / D);
            if (vo.ok) a.out[(vo.t * a.H + vo.h) * D + idx % D] = acc[k] * sinv[idx / D];
        }
    }
    if (threadIdx.x == 0) args.counters[blockIdx.z * a.Hk + kh] = 0u;  // ready for the next call
}

// ---- host side ---------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Row-major [rows, cols] f32 matrix, tiles of box_rows x box_cols.
bool encode_rows(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, int box_cols, int box_rows) {
    return cached_tensor_map(map, base, rows, cols, box_cols, box_rows, 0, [&](CUtensorMap* m) {
        auto fn = tensor_map_encoder();
        if (!fn) return false;
        const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)cols * sizeof(float)};
        const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
        const cuuint32_t estr[2] = {1, 1};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    });
}

template <int D, int G>
cudaError_t launch_cfg(const DecodeArgs& args, const AlibiTable& alibi, int n_rg, cudaStream_t stream) {
    using C = DecCfg<D, G>;
    const AttnDesc& a = args.a;
    CUtensorMap tmk, tmv;
    std::memset(&tmk, 0, sizeof(tmk));
    std::memset(&tmv, 0, sizeof(tmv));
    if (a.S > 0) {
        if (!encode_rows(&tmk, a.k, a.S, (int64_t)a.Hk * D, D, C::NR) ||
            !encode_rows(&tmv, a.v, a.S, (int64_t)a.Hk * D, D, C::NR))
            return cudaErrorInvalidValue;
    }
    auto kern = decode_splitkv_kernel<D, G>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), (int)C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid = VTMU_DEC_KH_FAST ? dim3(a.Hk, args.splits, n_rg) : dim3(args.splits, a.Hk, n_rg);
    kern<<<grid, C::THREADS, C::SMEM, stream>>>(args, alibi, tmk, tmv);
    return cudaGetLastError();
}

int stage_rows() { return VTMU_DEC_NR; }

}  // namespace

// Rows per row group: as many of the T query rows as fit 8 virtual heads
// (group size x rows), a power of two; padded to 2 virtual heads at least.
// (16 virtual heads, R = 2 rows per warp step, measured slower than two row
// groups of 8 that read the keys twice: the butterfly reduction then serves
// 2 rows instead of 4 to 16.)
void decode_rows(const AttnDesc& a, int* gv, int* tc, int* n_rg) {
    int t2 = 1;
    while (t2 < a.T) t2 *= 2;
    int c = 8 / a.G;
    if (c > t2) c = t2;
    if (c < 1) c = 1;
    *tc = c;
    *gv = a.G * c < 2 ? 2 : a.G * c;
    *n_rg = (int)((a.T + c - 1) / c);
}

bool decode_supported(const AttnDesc& a) {
    if (a.T < 1 || a.T > kDecodeMaxRows || a.D != a.Dv) return false;
    if (!(a.D == 32 || a.D == 64 || a.D == 128)) return false;
    if (!(a.G == 1 || a.G == 2 || a.G == 4 || a.G == 8)) return false;
    if (a.S >= ((int64_t)1 << 31)) return false;
    int gv, tc, n_rg;
    decode_rows(a, &gv, &tc, &n_rg);
    if ((int64_t)a.Hk * n_rg > kMaxDecodeKvHeads) return false;
    return true;
}

void decode_plan(const AttnDesc& a, int forced_splits, int num_sms, DecodePlan* plan) {
    // The keys any query row sees form one range (causal: s <= p; causal
    // window: s > p - w; non-causal window: |p - s| <= w), for rows at
    // positions p0 .. p1; each row masks the rest of it in the kernel.
    const int64_t p0 = a.pos_offset, p1 = a.pos_offset + (a.T > 0 ? a.T - 1 : 0);
    int64_t lo = 0, hi = a.S;  // [lo, hi)
    if (a.causal) {
        hi = p1 + 1 < hi ? p1 + 1 : hi;
        if (a.window > 0) lo = p0 - a.window + 1;
    } else if (a.window > 0) {
        lo = p0 - a.window;
        hi = p1 + a.window + 1 < hi ? p1 + a.window + 1 : hi;
    }
    int gv, tc, n_rg;
    decode_rows(a, &gv, &tc, &n_rg);
    plan->gv = gv;
    plan->tc = tc;
    plan->n_rg = n_rg;
    if (lo < 0) lo = 0;
    if (hi < lo) hi = lo;
    // Attention sinks: keys [0, sink_end) stay visible (within the causal
    // limit); a range of their own before the window's, or one range with it
    // when the two touch.
    const int64_t sink_cap = a.causal ? hi : a.S;
    int64_t sink_end = a.sinks < sink_cap ? a.sinks : sink_cap;
    if (sink_end > 0 && sink_end >= lo) {
        if (sink_end > hi) hi = sink_end;
        lo = 0;
        sink_end = 0;
    }
    if (sink_end < 0) sink_end = 0;
    const int64_t rows = hi - lo + sink_end;
    const int nr = stage_rows();
    int splits = forced_splits;
    if (splits <= 0) {
        // Fill the SMs once, in one wave: split each (KV head, row group)'s
        // range into floor(num_sms * ctas_per_sm / (Hk * n_rg)) chunks (rounding
        // up would start a few CTAs in a second wave and double the time).
        const int units = a.Hk * n_rg;
        splits = (num_sms * VTMU_DEC_CTAS_PER_SM) / units;
        if (splits < 1) splits = 1;
    }
    if (splits > kMaxSplits) splits = kMaxSplits;
    const int64_t min_rows = nr;
    int64_t per = (rows + splits - 1) / splits;
    if (per < min_rows) per = min_rows;
    per = (per + nr - 1) / nr * nr;
    // Each range takes whole splits: grow the split size until both fit the
    // split count (a sink range of its own needs one split of its own).
    int64_t n_sink = (sink_end + per - 1) / per;
    int64_t n = n_sink + (hi - lo + per - 1) / per;
    while (n > splits && per < rows) {
        per += nr;
        n_sink = (sink_end + per - 1) / per;
        n = n_sink + (hi - lo + per - 1) / per;
    }
    if (n < 1) n = 1;
    plan->s_lo = lo;
    plan->s_end = hi;
    plan->sink_end = sink_end;
    plan->sink_splits = (int32_t)n_sink;
    plan->rows_per_split = per;
    plan->splits = (int32_t)n;
    const size_t H = (size_t)n_rg * a.Hk * gv, Sp = (size_t)n;  // virtual heads
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    // Arrival counters in the workspace header (fixed place, so they stay
    // zero between calls of any shape), then m, l and o partials.
    plan->workspace_bytes = kWorkspaceHeader + up(H * Sp * 4) * 2 + up(H * Sp * (size_t)a.Dv * 4);
}

cudaError_t launch_decode(const AttnDesc& a, const AlibiTable& alibi, const DecodePlan& plan,
                          void* workspace, cudaStream_t stream, const DecodeCacheWrite* cw, const RopeDev* rope) {
    DecodeArgs args;
    std::memset(&args.cw, 0, sizeof(args.cw));
    if (cw) args.cw = *cw;
    std::memset(&args.rope, 0, sizeof(args.rope));
    if (rope) args.rope = *rope;
    args.a = a;
    args.s_lo = plan.s_lo;
    args.s_end = plan.s_end;
    args.rows_per_split = plan.rows_per_split;
    args.sink_end = plan.sink_end;
    args.sink_splits = plan.sink_splits;
    args.splits = plan.splits;
    args.gr = a.G;
    args.tc = plan.tc;
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t H = (size_t)plan.n_rg * a.Hk * plan.gv, Sp = (size_t)plan.splits;
    char* w = static_cast<char*>(workspace);
    args.counters = reinterpret_cast<unsigned int*>(w);
    w += kWorkspaceHeader;
    args.part_m = reinterpret_cast<float*>(w);
    args.part_l = reinterpret_cast<float*>(w + up(H * Sp * 4));
    args.part_o = reinterpret_cast<float*>(w + 2 * up(H * Sp * 4));
#define VTMU_DEC(D_, G_) \
    if (a.D == D_ && plan.gv == G_) return launch_cfg<D_, G_>(args, alibi, plan.n_rg, stream);
    VTMU_DEC(32, 2) VTMU_DEC(32, 4) VTMU_DEC(32, 8)
    VTMU_DEC(64, 2) VTMU_DEC(64, 4) VTMU_DEC(64, 8)
    VTMU_DEC(128, 2) VTMU_DEC(128, 4) VTMU_DEC(128, 8)
#undef VTMU_DEC
    return cudaErrorInvalidValue;
}

unsigned int decode_take_device_error() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_decode_device_error, sizeof(v)) != cudaSuccess) return 0;
    if (v) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_decode_device_error, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace vtmu
