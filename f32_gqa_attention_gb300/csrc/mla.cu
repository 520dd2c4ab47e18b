// mla.cu -- absorbed latent attention (mla_attention of the IR schema page,
// $defs.op_mla_attention), the decode form, f32 in and out.
//
// The latent cache row s is [c_s (kv_rank = 512) | r_s (qk_rope = 64)]; head
// h's key is [k_b_h c_s | r_s] and its value v_b_h c_s (k_b_h, v_b_h: head
// h's rows of the up-projections, stored [out, in]).  Absorbing the
// up-projections into the query and the output turns every head into a
// query against the SAME 576-wide latent row:
//     score(t, h, s) = scale * ( (k_b_h^T q_nope) . c_s + q_rope . r_s )
//     out(t, h)      = v_b_h ( sum_s p(t, h, s) c_s / sum_s p(t, h, s) )
// so the cache is read once for all heads.  Four launches:
//  1. mla_absorb_kernel: q_abs[t, h] = [k_b_h^T q_nope | q_rope] * scale *
//     log2 e (scores come out in base 2), and the new cache rows of a decode
//     step (op cache_write) -- the next launch reads them;
//  2. mla_latent_kernel: split-KV flash decoding over the latent rows.  A CTA
//     serves 4*HQ virtual heads (query row x head) on one chunk of keys; one
//     thread streams 32-row stages of the cache by TMA (nine 64-column boxes
//     per stage) into a three-stage ring, refilling a slot once all eight
//     warps have released it (a warp of its own would cap the registers of
//     every thread below what the consumers hold); warp w takes 4 heads
//     and a slice of each stage's keys.  Lane l holds 18 of the 576 dims of
//     every key (dims 128j + 4l .. +3 of the latent and 2l, 2l+1 of the
//     rotary key) and of its heads' queries, as packed pairs of neighbouring
//     dims (Blackwell's f32x2 FMA: two products per instruction, here and in
//     P.c); per 4 keys it forms 16 partial
//     dot products, a butterfly reduce-scatter leaves the score of (key
//     (l%16)/4, head l%4) in lane l, then an online softmax in base 2 (rescale only
//     when a max grows by more than 2^8) and P.c into 4 x 16 accumulators.
//     The same 16 latent dims serve as key and as value.  Warps holding
//     other key slices of the same heads merge in shared memory; the CTA
//     writes (m, l, o) per virtual head and split;
//  3. mla_merge_kernel: per virtual head the log-sum-exp merge of the splits
//     into the weighted latent; mla_project_kernel: its projection through
//     v_b_h.
// Every mbarrier wait is bounded (tma_sync.cuh); a wait that gives up sets a
// bit of g_mla_device_error and the kernel unwinds.
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_common.cuh"
#include "kernels.h"
#include "launch_cache.h"
#include "pdl.cuh"
#include "softcap.cuh"
#include "tma_sync.cuh"

namespace vtmu {

__device__ unsigned int g_mla_device_error;

namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kR = kMlaKvRank, kP = kMlaRope, kW = kR + kP;
constexpr int kNK = 32;                      // cache rows per stage
constexpr int kStages = 3;
constexpr int kBoxCols = 64;                 // TMA box: 64 columns x 32 rows
constexpr int kBoxes = kW / kBoxCols;        // 9 boxes per stage
constexpr int kBoxFloats = kNK * kBoxCols;   // 2048
constexpr int kStageFloats = kNK * kW;       // 18432 floats = 72 KB
constexpr uint32_t kStageBytes = kStageFloats * sizeof(float);
constexpr int kConsumerWarps = 8;
constexpr int kLatThreads = 32 * kConsumerWarps;  // lane 0 of warp 0 also issues the copies
constexpr size_t kLatSmem = (size_t)kStages * kStageBytes + 1024;
constexpr float kRescaleLog2 = 8.f;
constexpr int kMaxMlaSplits = 256;

enum MlaError : unsigned int {
    kErrMlaFull = 1u << 16,   // a consumer gave up on a loaded stage
    kErrMlaEmpty = 1u << 17,  // the producer gave up on a free stage
    kErrMlaDrain = 1u << 18,  // the producer gave up draining its copies
};

static_assert(kW % kBoxCols == 0 && kR == 512 && kP == 64, "latent row layout");

__device__ __forceinline__ void store_q(float* qabs, float* qlo, int64_t i, float x) {
    if (qlo == nullptr) {
        qabs[i] = x;
    } else {
        const float hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
        qabs[i] = hi;
        qlo[i] = x - hi;
    }
}


// ---- 1. absorb the queries, write the new cache rows ------------------------
// grid (heads, kR / 128, ceil(T / 4)), 256 threads.  Lane l of warp w owns
// latent columns 128 jb + 4 l .. + 3 and the k_b rows i = w, w + 8, ... of
// head h: one 16-byte load per row, all issued before the sums (the read of
// k_b is latency-bound otherwise); the eight warps' sums meet in shared memory.
constexpr int kAbsorbRows = 4;  // query rows per block
// With `qlo`, the result is written split for the tensor cores: qabs = its
// value with the low 13 mantissa bits cleared (a tf32 value), qlo = the rest.
__global__ void __launch_bounds__(256) mla_absorb_kernel(const float* __restrict__ q,
                                                         const float* __restrict__ k_b,
                                                         float* __restrict__ qabs, float* __restrict__ qlo,
                                                         int64_t T, int H, int N, float qscale, MlaCacheWrite cw) {
    extern __shared__ float sh[];
    float* qn = sh;                          // [kAbsorbRows][N]
    float* red = sh + kAbsorbRows * N;       // [8][kAbsorbRows][128]
    const int h = blockIdx.x, jb = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.z * kAbsorbRows;
    const int rows = (int)((T - t0) < kAbsorbRows ? (T - t0) : kAbsorbRows);
    const int Dq = N + kP;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_launch_dependents();  // the attention kernel may start its own prologue
    // The decode step's new cache rows (op cache_write), by one block.
    if (cw.state_new != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
        const int64_t n4 = cw.rows * kW / 4;
        const float4* src = reinterpret_cast<const float4*>(cw.state_new);
        float4* dst = reinterpret_cast<float4*>(cw.state + cw.offset * kW);
        for (int64_t i = tid; i < n4; i += blockDim.x) dst[i] = __ldg(src + i);
    }
    for (int idx = tid; idx < kAbsorbRows * N; idx += blockDim.x) {
        const int t = idx / N, i = idx % N;
        qn[idx] = t < rows ? __ldg(q + (t0 + t) * H * Dq + (int64_t)h * Dq + i) : 0.f;
    }
    __syncthreads();
    float acc[kAbsorbRows][4];
#pragma unroll
    for (int t = 0; t < kAbsorbRows; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    const float* kb = k_b + (int64_t)h * N * kR + jb * 128 + 4 * lane;
#pragma unroll 16
    for (int i = warp; i < N; i += 8) {
        const float4 w = __ldg(reinterpret_cast<const float4*>(kb + (int64_t)i * kR));
#pragma unroll
        for (int t = 0; t < kAbsorbRows; ++t) {
            const float qv = qn[t * N + i];
            acc[t][0] = fmaf(qv, w.x, acc[t][0]);
            acc[t][1] = fmaf(qv, w.y, acc[t][1]);
            acc[t][2] = fmaf(qv, w.z, acc[t][2]);
            acc[t][3] = fmaf(qv, w.w, acc[t][3]);
        }
    }
#pragma unroll
    for (int t = 0; t < kAbsorbRows; ++t)
        *reinterpret_cast<float4*>(red + (warp * kAbsorbRows + t) * 128 + 4 * lane) =
            make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
    __syncthreads();
    for (int idx = tid; idx < rows * 128; idx += blockDim.x) {
        const int t = idx / 128, c = idx % 128;
        float sum = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < 8; ++w8) sum += red[(w8 * kAbsorbRows + t) * 128 + c];
        store_q(qabs, qlo, ((t0 + t) * H + h) * kW + jb * 128 + c, sum * qscale);
    }
    if (jb == 0) {  // the rotary part passes through, scaled
        for (int idx = tid; idx < rows * kP; idx += blockDim.x) {
            const int t = idx / kP, r = idx % kP;
            store_q(qabs, qlo, ((t0 + t) * H + h) * kW + kR + r,
                    __ldg(q + (t0 + t) * H * Dq + (int64_t)h * Dq + N + r) * qscale);
        }
    }
}

// ---- 2. split-KV attention over the latent rows -----------------------------
struct LatArgs {
    AttnDesc a;        // S, T, H, causal, pos_offset, window, sinks (visibility)
    const float* qabs; // [V][kW]
    float* part_m;     // [V][splits]
    float* part_l;
    float* part_o;     // [V][splits][kR]
    int32_t V;         // virtual heads T * H
    int32_t splits;
    int32_t sink_splits;
    int64_t sink_end, lo, hi, per;
    int64_t new_lo, new_hi;  // cache rows the absorb launch writes (new_lo == new_hi: none)
};


// 16 partial sums per lane -> lanes l and l ^ 16 hold the warp-wide sum of
// entry l % 16 (entry 4 k + h: key k, head h of a 4-key batch).  Slot 4 k + h
// of lane l holds the partial of key k ^ ((l >> 2) & 3), head h: with the
// keys permuted by the lane's bits 3..2, the first two butterfly steps need
// no selects (a lane keeps its low slots, whose entries match the partner's
// high slots); the two head steps keep/send by the lane's bit; a last add
// joins the half-warps.
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
    for (int w = 8; w >= 4; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) v[i] += __shfl_xor_sync(FULL, v[i + w], w);
#pragma unroll
    for (int w = 2; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = up ? v[i] : v[i + w];
            const float keep = up ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(FULL, send, w);
        }
    }
    return v[0] + __shfl_xor_sync(FULL, v[0], 16);
}

// Offset (floats) of dims 128 j + 4 lane .. +3 of key row `key` in a stage.
__device__ __forceinline__ int lat_off(int j, int lane, int key) {
    return (2 * j + (lane >> 4)) * kBoxFloats + key * kBoxCols + ((4 * lane) & 63);
}
// Offset of rotary dims 2 lane, 2 lane + 1.
__device__ __forceinline__ int rope_off(int lane, int key) { return 8 * kBoxFloats + key * kBoxCols + 2 * lane; }

template <int HQ>
__global__ void __launch_bounds__(kLatThreads, 1)
    mla_latent_kernel(const __grid_constant__ CUtensorMap tm_state, const LatArgs args) {
    constexpr int KS = kConsumerWarps / HQ;  // key slices per stage
    constexpr int KPW = kNK / KS;            // keys per warp and stage
    constexpr int NB = KPW / 4;              // 4-key batches per warp and stage
    static_assert(NB >= 1, "at least 4 keys per warp and stage");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    float* ring = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.y;
    int64_t k0, k1;
    if (split < args.sink_splits) {
        k0 = (int64_t)split * args.per;
        k1 = k0 + args.per < args.sink_end ? k0 + args.per : args.sink_end;
    } else {
        k0 = args.lo + (int64_t)(split - args.sink_splits) * args.per;
        k1 = k0 + args.per < args.hi ? k0 + args.per : args.hi;
    }
    const int nst = k1 > k0 ? (int)((k1 - k0 + kNK - 1) / kNK) : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // Stage `it` of this split: nine boxes of 64 columns x 32 rows.
    auto issue = [&](int it) {
        const int slot = it % kStages;
        mbar_arrive_expect_tx(&full[slot], kStageBytes);
        float* dst = ring + slot * kStageFloats;
        const int y = (int)(k0 + (int64_t)it * kNK);
#pragma unroll 1
        for (int b = 0; b < kBoxes; ++b) tma_load_2d(dst + b * kBoxFloats, &tm_state, b * kBoxCols, y, &full[slot]);
    };
    const bool producer = threadIdx.x == 0;
    int issued = 0;  // stages issued (producer thread)
    pdl_launch_dependents();
    if (producer) {
        prefetch_tensormap(&tm_state);
        // Rows the absorb launch writes must be in memory before a TMA read
        // of them; other splits stream the cache at once.
        if (args.new_hi > args.new_lo && k0 < args.new_hi && args.new_lo < k0 + (int64_t)nst * kNK) pdl_wait();
        for (; issued < nst && issued < kStages; ++issued) issue(issued);
    }
    pdl_wait();  // the absorbed queries

    // ---- consumers ----
    const int hq = warp % HQ, ks = warp / HQ;
    const int vh0 = blockIdx.x * 4 * HQ + hq * 4;  // this warp's first virtual head
    const int my_h = lane & 3;
    const int my_v = vh0 + my_h;
    const int64_t my_pos = args.a.pos_offset + (my_v < args.V ? my_v / args.a.H : 0);
    // The lane's 18 dims of each of its heads' queries as packed pairs of
    // neighbouring dims (f32x2 registers): latent dims 128 j + 4 lane + (0, 1)
    // and (2, 3), then the rotary pair.
    uint64_t q2[4][9];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const int v = vh0 + h;
        if (v < args.V) {
            const float* qr = args.qabs + (int64_t)v * kW;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const ulonglong2 x = __ldg(reinterpret_cast<const ulonglong2*>(qr + 128 * j + 4 * lane));
                q2[h][2 * j] = x.x;
                q2[h][2 * j + 1] = x.y;
            }
            q2[h][8] = __ldg(reinterpret_cast<const unsigned long long*>(qr + kR + 2 * lane));
        } else {
#pragma unroll
            for (int i = 0; i < 9; ++i) q2[h][i] = 0ull;
        }
    }
    // O's latent dims 128 j + 4 lane + (0, 1) and (2, 3) of each head, packed.
    uint64_t o2[4][8];
#pragma unroll
    for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int i = 0; i < 8; ++i) o2[h][i] = 0ull;
    // The lane's head (lane % 4): its reference max (base 2, lazily raised)
    // and its running sum, the same in every lane of that head.
    float m_my = -INFINITY, l_my = 0.f;
    __shared__ __align__(16) float2 pbuf[kConsumerWarps][16];  // a batch's probabilities (p, p), per warp
    const int kx = (lane >> 2) & 3;  // key permutation of the score slots
    bool ok = true;
    for (int it = 0; it < nst; ++it) {
        const int slot = it % kStages;
        if (!__all_sync(FULL, mbar_wait(&full[slot], (uint32_t)((it / kStages) & 1)))) {
            raise_device_error(&g_mla_device_error, kErrMlaFull);
            ok = false;
            break;
        }
        const float* st = ring + slot * kStageFloats;
        const int64_t stage_key0 = k0 + (int64_t)it * kNK;
#pragma unroll 1
        for (int b = 0; b < NB; ++b) {
            const int kb = ks * KPW + b * 4;  // first stage-local key of the batch
            // This lane's latent dims of the batch's first key; key k and
            // latent block j sit at the constant offset k * 64 + 2 j * 2048.
            const float* lp = st + lat_off(0, lane, kb);
            const float* rp = st + rope_off(lane, kb);
            float part[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int kk = k ^ kx;  // this lane's key for slot group k
                uint64_t kv[9];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const ulonglong2 x = *reinterpret_cast<const ulonglong2*>(lp + kk * kBoxCols + 2 * j * kBoxFloats);
                    kv[2 * j] = x.x;
                    kv[2 * j + 1] = x.y;
                }
                kv[8] = *reinterpret_cast<const unsigned long long*>(rp + kk * kBoxCols);
#pragma unroll
                for (int h = 0; h < 4; ++h) {  // even and odd dims in the two halves of a pair
                    uint64_t s2 = f2_mul(q2[h][0], kv[0]);
#pragma unroll
                    for (int i = 1; i < 9; ++i) s2 = f2_fma(q2[h][i], kv[i], s2);
                    float se, so;
                    f2_unpack(s2, se, so);
                    part[4 * k + h] = se + so;
                }
            }
            // Lanes l and l ^ 16: the score of key kb + (l % 16) / 4 for head
            // l % 4 (base 2).
            float x = reduce_scatter16(part, lane);
            const int64_t s_key = stage_key0 + kb + ((lane & 15) >> 2);
            const bool vis = my_v < args.V && s_key < k1 && key_visible<true>(args.a, my_pos, s_key);
            if (!vis) x = -INFINITY;
            float mt = x;  // the batch's max for the lane's head (both half-warps agree)
            mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 4));
            mt = fmaxf(mt, __shfl_xor_sync(FULL, mt, 8));
            // Lazy rescale: only when some head's max beats its reference by > 2^8.
            const bool raise = mt > m_my + kRescaleLog2;
            if (__any_sync(FULL, raise)) {
                // 0 when nothing was visible before; 1 for the heads not raised
                // (also those that have seen nothing: -inf - -inf is no number).
                const float a_my = raise ? fast_exp2(m_my - mt) : 1.f;
                if (raise) m_my = mt;
                l_my *= a_my;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float ah = __shfl_sync(FULL, a_my, h);
                    const uint64_t ah2 = f2_pack(ah, ah);
#pragma unroll
                    for (int i = 0; i < 8; ++i) o2[h][i] = f2_mul(o2[h][i], ah2);
                }
            }
            const float pv = fast_exp2(x - (m_my == -INFINITY ? 0.f : m_my));
            float ps = pv;  // the batch's sum for the lane's head, within a half-warp
            ps += __shfl_xor_sync(FULL, ps, 4);
            ps += __shfl_xor_sync(FULL, ps, 8);
            l_my += ps;
            // O += P c: the latent dims of each key serve as its value.  The
            // batch's 16 probabilities go through shared memory to every lane
            // as (p, p) pairs (eight broadcast loads), then one 16-byte load
            // of a key's block feeds 8 packed FMAs (16 products).
            if (lane < 16) pbuf[warp][lane] = make_float2(pv, pv);
            __syncwarp();
            uint64_t pk2[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const ulonglong2 p2 = *reinterpret_cast<const ulonglong2*>(&pbuf[warp][2 * i]);
                pk2[2 * i] = p2.x;
                pk2[2 * i + 1] = p2.y;
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const ulonglong2 c = *reinterpret_cast<const ulonglong2*>(lp + k * kBoxCols + 2 * j * kBoxFloats);
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        o2[h][2 * j] = f2_fma(pk2[4 * k + h], c.x, o2[h][2 * j]);
                        o2[h][2 * j + 1] = f2_fma(pk2[4 * k + h], c.y, o2[h][2 * j + 1]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        // Refill the slot with stage it + kStages once every warp released it.
        if (producer && issued < nst) {
            if (mbar_wait(&empty[slot], (uint32_t)((it / kStages) & 1))) {
                issue(issued);
                ++issued;
            } else {
                raise_device_error(&g_mla_device_error, kErrMlaEmpty);
                issued = nst + 1;  // stop issuing
            }
        }
    }
    // No copy may be in flight when the CTA exits (a loop that stopped early
    // can leave some).
    if (producer) {
        const int last = issued > nst ? nst : issued;
        for (int it = last - kStages < 0 ? 0 : last - kStages; it < last; ++it)
            if (!mbar_wait(&full[it % kStages], (uint32_t)((it / kStages) & 1)))
                raise_device_error(&g_mla_device_error, kErrMlaDrain);
    }
    float o[4][16];
#pragma unroll
    for (int h = 0; h < 4; ++h)
#pragma unroll
        for (int i = 0; i < 8; ++i) f2_unpack(o2[h][i], o[h][2 * i], o[h][2 * i + 1]);
    // Every head's reference max and sum, in every lane.
    float m_ref[4], l_sum[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        m_ref[h] = __shfl_sync(FULL, m_my, h);
        l_sum[h] = __shfl_sync(FULL, l_my, h);
    }

    // ---- merge the key slices of each head, write the split's partials ----
    const int splits = args.splits;
    if constexpr (KS > 1) {
        // Every consumer warp is done with the ring (each waited for every
        // stage), so its first 64 KB become the merge scratch.
        asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kConsumerWarps) : "memory");
        float* sc_o = ring;                                  // [warp][4][kR]
        float* sc_ml = ring + kConsumerWarps * 4 * kR;       // [warp][4][2]
#pragma unroll
        for (int h = 0; h < 4; ++h) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<float4*>(sc_o + (warp * 4 + h) * kR + 128 * j + 4 * lane) =
                    make_float4(o[h][4 * j], o[h][4 * j + 1], o[h][4 * j + 2], o[h][4 * j + 3]);
        }
        if (lane < 4) {
            const float mm = lane == 0 ? m_ref[0] : lane == 1 ? m_ref[1] : lane == 2 ? m_ref[2] : m_ref[3];
            const float ll = lane == 0 ? l_sum[0] : lane == 1 ? l_sum[1] : lane == 2 ? l_sum[2] : l_sum[3];
            sc_ml[(warp * 4 + lane) * 2] = mm;
            sc_ml[(warp * 4 + lane) * 2 + 1] = ll;
        }
        asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kConsumerWarps) : "memory");
        if (ks != 0) return;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            float M = -INFINITY;
#pragma unroll
            for (int k2 = 0; k2 < KS; ++k2) M = fmaxf(M, sc_ml[((k2 * HQ + hq) * 4 + h) * 2]);
            const float mu = M == -INFINITY ? 0.f : M;
            float L = 0.f;
            float acc[16];
#pragma unroll
            for (int d = 0; d < 16; ++d) acc[d] = 0.f;
#pragma unroll
            for (int k2 = 0; k2 < KS; ++k2) {
                const int wsrc = k2 * HQ + hq;
                const float wgt = fast_exp2(sc_ml[(wsrc * 4 + h) * 2] - mu);
                L = fmaf(sc_ml[(wsrc * 4 + h) * 2 + 1], wgt, L);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 x = *reinterpret_cast<const float4*>(sc_o + (wsrc * 4 + h) * kR + 128 * j + 4 * lane);
                    acc[4 * j] = fmaf(x.x, wgt, acc[4 * j]);
                    acc[4 * j + 1] = fmaf(x.y, wgt, acc[4 * j + 1]);
                    acc[4 * j + 2] = fmaf(x.z, wgt, acc[4 * j + 2]);
                    acc[4 * j + 3] = fmaf(x.w, wgt, acc[4 * j + 3]);
                }
            }
            m_ref[h] = M;
            l_sum[h] = L;
#pragma unroll
            for (int d = 0; d < 16; ++d) o[h][d] = acc[d];
        }
    }
    if (!ok) return;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const int v = vh0 + h;
        if (v >= args.V) continue;
        const int64_t idx = (int64_t)v * splits + split;
        if (lane == 0) {
            args.part_m[idx] = m_ref[h];
            args.part_l[idx] = l_sum[h];
        }
        float* po = args.part_o + idx * kR;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            *reinterpret_cast<float4*>(po + 128 * j + 4 * lane) =
                make_float4(o[h][4 * j], o[h][4 * j + 1], o[h][4 * j + 2], o[h][4 * j + 3]);
    }
}

// ---- 3. merge the splits, then project through v_b ----------------------------
// Merge: grid (V, kR / 32), 256 threads.  Warp w takes splits w, w + 8, ...
// of its 32 latent dims (lane = dim), eight loads in flight per lane; the
// log-sum-exp weights come from one pass over the split maxima.  olat[v] =
// sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i (zeros when nothing was
// visible).
__global__ void __launch_bounds__(256) mla_merge_kernel(const float* __restrict__ part_m,
                                                        const float* __restrict__ part_l,
                                                        const float* __restrict__ part_o, float* __restrict__ olat,
                                                        int splits) {
    __shared__ float wsp[kMaxMlaSplits];
    __shared__ float red[8][32];
    __shared__ float inv_l;
    pdl_launch_dependents();
    pdl_wait();  // the attention kernel's partials
    const int v = blockIdx.x, d = blockIdx.y * 32 + (threadIdx.x & 31);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (warp == 0) {
        float M = -INFINITY;
        for (int i = lane; i < splits; i += 32) M = fmaxf(M, __ldcg(part_m + (int64_t)v * splits + i));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, off));
        const float mu = M == -INFINITY ? 0.f : M;
        float L = 0.f;
        for (int i = lane; i < splits; i += 32) {
            const float w = fast_exp2(__ldcg(part_m + (int64_t)v * splits + i) - mu);
            wsp[i] = w;
            L = fmaf(__ldcg(part_l + (int64_t)v * splits + i), w, L);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(FULL, L, off);
        if (lane == 0) inv_l = L > 0.f ? 1.f / L : 0.f;
    }
    __syncthreads();
    const float* po = part_o + (int64_t)v * splits * kR + d;
    float acc = 0.f;
#pragma unroll 8
    for (int i = warp; i < splits; i += 8) acc = fmaf(__ldcg(po + (int64_t)i * kR), wsp[i], acc);
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) sum += red[w][lane];
        olat[(int64_t)v * kR + d] = sum * inv_l;
    }
}

// Project: grid (V, ceil(Dv / 32)), 256 threads; warp w computes outputs
// e0 + 4 w .. + 3, each the dot product of v_b's row with olat[v] (512 long).
__global__ void __launch_bounds__(256) mla_project_kernel(const float* __restrict__ olat,
                                                          const float* __restrict__ v_b, float* __restrict__ out,
                                                          int H, int Dv) {
    pdl_wait();  // the merged latent
    const int v = blockIdx.x;
    const int64_t t = v / H;
    const int h = v % H;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float4 c[kR / 128];
#pragma unroll
    for (int j = 0; j < kR / 128; ++j) c[j] = __ldcg(reinterpret_cast<const float4*>(olat + (int64_t)v * kR + 128 * j + 4 * lane));
    const int e0 = blockIdx.y * 32 + warp * 4;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int e = e0 + u;
        if (e < Dv) {
            const float* row = v_b + ((int64_t)h * Dv + e) * kR;
#pragma unroll
            for (int j = 0; j < kR / 128; ++j) {
                const float4 w = __ldg(reinterpret_cast<const float4*>(row + 128 * j + 4 * lane));
                acc[u] = fmaf(w.x, c[j].x, fmaf(w.y, c[j].y, fmaf(w.z, c[j].z, fmaf(w.w, c[j].w, acc[u]))));
            }
        }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[u] += __shfl_xor_sync(FULL, acc[u], off);
        if (lane == 0 && e0 + u < Dv) out[(t * H + h) * Dv + e0 + u] = acc[u];
    }
}

// ---- host side ------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 mla_encoder() {
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

bool encode_state(CUtensorMap* map, const float* state, int64_t rows) {
    return cached_tensor_map(map, state, rows, kW, kBoxCols, kNK, 0, [&](CUtensorMap* m) {
        auto fn = mla_encoder();
        if (!fn) return false;
        const cuuint64_t dims[2] = {(cuuint64_t)kW, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)kW * sizeof(float)};
        const cuuint32_t box[2] = {(cuuint32_t)kBoxCols, (cuuint32_t)kNK};
        const cuuint32_t estr[2] = {1, 1};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(state), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    });
}

template <int HQ>
cudaError_t launch_latent(const CUtensorMap& tm, const LatArgs& args, int groups, cudaStream_t stream) {
    auto kern = mla_latent_kernel<HQ>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), (int)kLatSmem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(groups, args.splits), dim3(kLatThreads), kLatSmem, stream, tm, args);
}

size_t up256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace

void mla_layout(MlaPlan* plan, int64_t V, int n);

void mla_plan(const MlaDesc& m, int num_sms, MlaPlan* plan) {
    const int64_t V = m.T * m.H;
    plan->hq = V <= 8 ? 2 : (V <= 16 ? 4 : 8);
    plan->groups = V > 0 ? (int)((V + 4 * plan->hq - 1) / (4 * plan->hq)) : 1;
    // The keys any query row sees: one range [lo, hi), and with a window the
    // sink range [0, sink_end) before it (joined when they touch).
    const int64_t p0 = m.pos_offset, p1 = m.pos_offset + (m.T > 0 ? m.T - 1 : 0);
    int64_t lo = 0, hi = m.S;
    if (m.causal) {
        if (p1 + 1 < hi) hi = p1 + 1;
        if (m.window > 0) lo = p0 - m.window + 1;
    } else if (m.window > 0) {
        lo = p0 - m.window;
        if (p1 + m.window + 1 < hi) hi = p1 + m.window + 1;
    }
    if (lo < 0) lo = 0;
    if (hi < lo) hi = lo;
    int64_t sink_end = m.window > 0 ? m.sinks : 0;
    const int64_t sink_cap = m.causal ? hi : m.S;
    if (sink_end > sink_cap) sink_end = sink_cap;
    if (sink_end > 0 && sink_end >= lo) {
        if (sink_end > hi) hi = sink_end;
        lo = 0;
        sink_end = 0;
    }
    if (sink_end < 0) sink_end = 0;
    const int64_t rows = hi - lo + sink_end;
    int splits = num_sms / plan->groups;
    if (splits < 1) splits = 1;
    if (splits > kMaxMlaSplits) splits = kMaxMlaSplits;
    int64_t per = (rows + splits - 1) / splits;
    per = (per + kNK - 1) / kNK * kNK;
    if (per < kNK) per = kNK;
    int64_t n_sink = (sink_end + per - 1) / per, n = n_sink + (hi - lo + per - 1) / per;
    while (n > kMaxMlaSplits) {
        per += kNK;
        n_sink = (sink_end + per - 1) / per;
        n = n_sink + (hi - lo + per - 1) / per;
    }
    if (n < 1) n = 1;
    plan->lo = lo;
    plan->hi = hi;
    plan->sink_end = sink_end;
    plan->per = per;
    plan->sink_splits = (int)n_sink;
    plan->splits = (int)n;
    plan->num_sms = num_sms;
    mla_layout(plan, V, (int)n);
}

// Workspace: the decode counters' header, q_abs (and its tf32 remainder),
// then the m, l and o partials of n splits, then the merged latents.
void mla_layout(MlaPlan* plan, int64_t V, int n) {
    plan->qabs_off = kWorkspaceHeader;
    plan->qlo_off = plan->qabs_off + up256((size_t)V * kW * 4);
    plan->m_off = plan->qlo_off + up256((size_t)V * kW * 4);
    plan->l_off = plan->m_off + up256((size_t)V * n * 4);
    plan->o_off = plan->l_off + up256((size_t)V * n * 4);
    plan->olat_off = plan->o_off + up256((size_t)V * n * kR * 4);
    plan->workspace_bytes = plan->olat_off + up256((size_t)V * kR * 4);
}

cudaError_t launch_mla(const MlaDesc& m, const MlaPlan& base, void* workspace, const MlaCacheWrite& cw,
                       cudaStream_t stream) {
    if (m.T == 0) return cudaSuccess;
    MlaPlan plan = base;
    MlaTcPlan tp;
    if (m.use_tc) {
        mla_tc_plan(m, base, base.num_sms, &tp);
        mla_layout(&plan, m.T * m.H, tp.splits);
    }
    char* w = static_cast<char*>(workspace);
    float* qabs = reinterpret_cast<float*>(w + plan.qabs_off);
    float* qlo = m.use_tc ? reinterpret_cast<float*>(w + plan.qlo_off) : nullptr;
    const int64_t tblocks = (m.T + kAbsorbRows - 1) / kAbsorbRows;
    const size_t absorb_smem = (size_t)(kAbsorbRows * m.N + 8 * kAbsorbRows * 128) * sizeof(float);
    if (absorb_smem > 48 * 1024) {
        cudaError_t e = set_smem_once(reinterpret_cast<const void*>(mla_absorb_kernel), (int)absorb_smem);
        if (e != cudaSuccess) return e;
    }
    mla_absorb_kernel<<<dim3(m.H, kR / 128, (unsigned)tblocks), 256, absorb_smem, stream>>>(
        m.q, m.k_b, qabs, qlo, m.T, m.H, m.N, m.qscale, cw);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (m.S == 0)  // no cache row: every output row is zero
        return cudaMemsetAsync(m.out, 0, (size_t)m.T * m.H * m.Dv * sizeof(float), stream);
    float* part_m = reinterpret_cast<float*>(w + plan.m_off);
    float* part_l = reinterpret_cast<float*>(w + plan.l_off);
    float* part_o = reinterpret_cast<float*>(w + plan.o_off);
    int splits = plan.splits;
    if (m.use_tc) {
        e = launch_mla_latent_tc(m, plan, tp, qabs, qlo, part_m, part_l, part_o, stream);
        splits = tp.splits;
    } else {
        CUtensorMap tm;
        std::memset(&tm, 0, sizeof(tm));
        if (!encode_state(&tm, m.state, m.S)) return cudaErrorInvalidValue;
        LatArgs args;
        std::memset(&args, 0, sizeof(args));
        args.a.S = m.S;
        args.a.T = m.T;
        args.a.H = m.H;
        args.a.causal = m.causal;
        args.a.pos_offset = m.pos_offset;
        args.a.window = m.window;
        args.a.sinks = m.window > 0 ? m.sinks : 0;
        args.qabs = qabs;
        args.part_m = part_m;
        args.part_l = part_l;
        args.part_o = part_o;
        args.V = (int32_t)(m.T * m.H);
        args.splits = plan.splits;
        args.sink_splits = plan.sink_splits;
        args.sink_end = plan.sink_end;
        args.lo = plan.lo;
        args.hi = plan.hi;
        args.per = plan.per;
        args.new_lo = cw.state_new != nullptr ? cw.offset : 0;
        args.new_hi = cw.state_new != nullptr ? cw.offset + cw.rows : 0;
        switch (plan.hq) {
            case 2: e = launch_latent<2>(tm, args, plan.groups, stream); break;
            case 4: e = launch_latent<4>(tm, args, plan.groups, stream); break;
            default: e = launch_latent<8>(tm, args, plan.groups, stream); break;
        }
    }
    if (e != cudaSuccess) return e;
    const unsigned V = (unsigned)(m.T * m.H);
    float* olat = reinterpret_cast<float*>(w + plan.olat_off);
    e = launch_pdl(mla_merge_kernel, dim3(V, kR / 32), dim3(256), 0, stream, (const float*)part_m,
                   (const float*)part_l, (const float*)part_o, olat, splits);
    if (e != cudaSuccess) return e;
    return launch_pdl(mla_project_kernel, dim3(V, (unsigned)((m.Dv + 31) / 32)), dim3(256), 0, stream,
                      (const float*)olat, m.v_b, m.out, m.H, m.Dv);
}

unsigned int mla_take_device_error() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_mla_device_error, sizeof(v)) != cudaSuccess) return 0;
    if (v) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_mla_device_error, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace vtmu
