// decode_tc.cu -- split-KV decode of a few query rows (a speculative or
// chunked step: T rows at positions posOffset .. posOffset + T - 1 against a
// KV cache, headDim 128) with both contractions on the tcgen05 tensor cores
// in 3xTF32.
//
// Op "attention" (vtmu.mpakt.dev/api/ops) with GQA: query head h reads KV
// head h / G.  For one KV head the T rows x G heads form up to 16 virtual
// heads v = t G + g, and all of them meet the same K and V rows.  The roles
// of the MMAs are swapped with respect to a prefill: the 16 virtual heads are
// the N side of both products,
//     S^T[key, v] = sum_d K[key, d] q[v, d] scale log2 e     (M = 128 keys)
//     O^T[d, v]   = sum_key V^T[d, key] P^T[key, v]          (M = 128 dims)
// each as hi.hi + hi.lo + lo.hi (3xTF32), so one M = 128, N = 16 MMA does
// 2048 (key, head) or (dim, head) pairs.  K and Q are K-major in shared
// memory as the score MMA reads them; the values' contraction index (the
// cache row) is not contiguous in the cache, so V goes to TMEM transposed
// (dims as lanes, rows as columns) through registers and serves as the TMEM
// operand A, with P^T (heads x rows, rows contiguous) from shared memory.
// Each K and V byte of the visible range is read from HBM once for all T
// rows.
//
// One launch, decode_tc_kernel, grid (kv heads, splits):
//  1. one CTA streams a run of
//     128-row tiles of its KV head's range (the attention sinks' tiles
//     first, as splits of their own).  In a decode step, the CTA whose
//     tile shows a new cache row writes that row (its KV head's columns)
//     before its first TMA read; rows no tile shows go to split 0.  Warps:
//       0      the new K rows, then lane 0 streams the score ring (K blocks
//              of [128 rows x 32 dims] by TMA, 128-byte swizzle);
//       1      lane 0 issues the score MMAs into S buffer (tile & 1); warp 1
//              owns TMEM (S 2 x 16 columns, O 2 x 16, K_lo 6 x 32, V^T hi
//              and lo 128 each);
//       2      the new V rows, then lane 0 streams the value ring (V blocks
//              of [128 rows x 32 dims]);
//       3      lane 0 issues the P.V MMAs of a tile into O buffer (tile & 1)
//              once its P^T and V^T are in place;
//       4 .. 7 split each K block in place into K_hi (low 13 mantissa bits
//              cleared) and K_lo = K - K_hi, which goes to TMEM (thread =
//              row = lane) as the operand A of the K_lo.Q_hi product;
//       8 .. 15 first the query tiles: q scaled by scale log2 e, split into
//              Q_hi (tf32, rounded to nearest) and Q_lo = q - Q_hi in the
//              K-major blocks the score MMA reads (zero rows past T G); then
//              two softmax groups: warps 8 .. 11 take the even tiles of
//              the run, 12 .. 15 the odd ones, so two tiles are in flight;
//              each group has its own S buffer, P^T buffer and O buffer and
//              its own running (m, l, o).  Thread = a row of the tile, all 16
//              heads: read S^T from TMEM, mask, reduce max and sum over the
//              rows (a reduce-scatter over the warp, then the group's four
//              warps through shared memory), online softmax in base 2 with
//              a lazy reference max (rescale only when a max grows by more
//              than 2^8), P^T hi and lo to shared memory; then the group
//              folds its previous tile's O into registers, o = o alpha + O
//              (a fresh accumulator per tile, so no sum runs long inside the
//              tensor pipe), and warp q of the group moves the next tile's V
//              block q (dims 32 q ..) into TMEM lanes 32 q .. as V^T hi and
//              lo once this tile's P.V MMAs are done with V^T (group 1 moves
//              the first tile's at the start);
//     then the two groups' (m, l, o) are combined (rescaled to the larger
//     reference) and written as the split's partial;
//  2. the last CTA of a KV head to finish (an arrival counter in the
//     workspace header, no waiting) merges, per virtual head, the splits'
//     partials by the log-sum-exp rule, m* = max m_i, l* = sum l_i 2^(m_i - m*),
//     o* = sum o_i 2^(m_i - m*) / l*, written to the output row (zeros when
//     no key is visible).
// Every ring item is waited for and released by every role that reads it,
// so no role is ever two phases behind a slot (an mbarrier wait only checks
// a phase's parity); a value block always lands in the slots of the one
// warp that reads it.  Every wait is bounded; a wait that gives up sets a
// bit of g_decode_tc_device_error and the kernel unwinds.
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_common.cuh"
#include "kernels.h"
#include "launch_cache.h"
#include "rope.cuh"
#include "tcgen05_ops.cuh"
#include "tma_sync.cuh"

namespace vtmu {

__device__ unsigned int g_decode_tc_device_error;

namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kNV = kDecodeTcHeads;   // virtual heads per KV head (MMA N)
constexpr int kD = 128;               // head dim (the P.V MMA's M)
constexpr int kKT = 128;              // cache rows per tile (the score MMA's M)
constexpr int kC = kD / 32;           // 32-dim blocks per tile
constexpr int kNK = 6;                // score ring slots (1.5 tiles)
constexpr int kNVR = 4;               // value ring slots (one tile; eight, with three K slots, measured slower)
constexpr uint32_t kBlockBytes = kKT * 32 * 4;  // one [128 rows x 32 dims] block, 16 KB
constexpr uint32_t kKSlot = kBlockBytes;        // a K block (K_hi after the split; K_lo goes to TMEM)
constexpr uint32_t kQChunk = kNV * 32 * 4;      // [16 heads x 32 dims or rows], 2 KB
constexpr uint32_t kQBytes = 2u * kC * kQChunk;   // Q_hi chunks, then Q_lo chunks
constexpr uint32_t kPTBytes = 2u * (kKT / 32) * kQChunk;  // per group: P^T hi blocks, then lo blocks
constexpr int kThreads = 16 * 32;
constexpr size_t kSmem = 1024 + (size_t)kNK * kKSlot + (size_t)kNVR * kBlockBytes + kQBytes + 2 * kPTBytes;
constexpr float kRescaleLog2 = 8.f;
// TMEM columns: S (2 buffers x 16), O (2 buffers x 16), K_lo (one 32-column block per score ring
// slot), V^T hi and lo (128 each).
constexpr uint32_t kColS = 0, kColO = 32, kColKlo = 64, kColVhi = 256, kColVlo = 384, kTmemCols = 512;
static_assert(kColKlo + 32 * kNK <= kColVhi && kColVlo + 128 <= kTmemCols, "TMEM budget");
constexpr uint32_t kKReleases = 4 + 1;  // splitter warps, the score issuer's commit
static_assert(kSmem + 2048 <= 232448, "shared memory budget");
static_assert(kNV * kRopeMaxPairs * (int)sizeof(float2) <= kPTBytes, "the query's rotary table fits a P^T buffer");
static_assert(kC == 4 && kNVR % kC == 0, "slot (t % 2) * 4 + q holds value block q of tile t");

enum : unsigned int {
    kErrDtFull = 1u << 26,    // a consumer gave up on an arriving ring item or the query tiles
    kErrDtEmpty = 1u << 27,   // a producer gave up on a free slot
    kErrDtSplit = 1u << 28,   // an issuer gave up on a split item
    kErrDtS = 1u << 29,       // a softmax warp gave up on a score tile
    kErrDtFree = 1u << 30,    // an issuer gave up on a free score buffer
    kErrDtDrain = 1u << 31,   // a producer gave up draining its copies
    kErrDtPV = kErrDtS,       // a P.V or fold wait gave up (reported with the score-tile bit)
    kErrDtV = kErrDtFull,     // a value block or free V^T wait gave up
};

struct DtArgs {
    AttnDesc a;        // S, T, H, G, causal, pos_offset, window, sinks (visibility)
    float* part_m;     // [Hk][16][splits] (both softmax groups combined)
    float* part_l;
    float* part_o;     // [Hk][16][splits][D]
    unsigned int* counters;  // [Hk] arrival counters (workspace header), zero between calls
    int32_t nv;        // virtual heads in use: T * G
    int32_t sink_lim;  // with a window: rows below this are attention sinks (0: none)
    DecodeCacheWrite cw;  // the step's new rows (cw.hi == cw.lo: none); 16-byte aligned
    int32_t splits;
    int32_t sink_splits;
    int32_t n_sink_tiles, n_tiles;  // tiles of the sink range and of the main range
    int64_t lo;        // first row of the main range (the sink range starts at 0)
    int64_t sink_end, hi;
    RopeDev rope;      // rotary embedding of q and the new keys (rope.half == 0: none)
};

// Tiles [t0, t1) of this split in the concatenated (sink, main) tile list.
__device__ __forceinline__ void split_tiles(const DtArgs& g, int split, int& t0, int& t1) {
    if (split < g.sink_splits) {
        t0 = (int)((int64_t)g.n_sink_tiles * split / g.sink_splits);
        t1 = (int)((int64_t)g.n_sink_tiles * (split + 1) / g.sink_splits);
    } else {
        const int ms = g.splits - g.sink_splits, i = split - g.sink_splits;
        t0 = g.n_sink_tiles + (int)((int64_t)g.n_tiles * i / ms);
        t1 = g.n_sink_tiles + (int)((int64_t)g.n_tiles * (i + 1) / ms);
    }
}
// First cache row of tile `t` of the concatenated list, and its range end.
__device__ __forceinline__ void tile_rows(const DtArgs& g, int t, int64_t& r0, int64_t& rend) {
    if (t < g.n_sink_tiles) {
        r0 = (int64_t)t * kKT;
        rend = g.sink_end;
    } else {
        r0 = g.lo + (int64_t)(t - g.n_sink_tiles) * kKT;
        rend = g.hi;
    }
}

// Barrier over the eight softmax warps (named barrier 3, 256 threads);
// returns the AND of `v` over them.
__device__ __forceinline__ bool softmax_sync_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 3, 256, q;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Barrier over one softmax group's four warps (named barrier ID, 128
// threads); returns the AND of `v` over them.
template <int ID>
__device__ __forceinline__ bool group_sync_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, %2, 128, q;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(ID)
        : "memory");
    return r != 0;
}

// True when new cache row r belongs to this CTA: a row of one of its tiles'
// visible ranges, or, for a row that no tile shows, split 0.
__device__ __forceinline__ bool owns_row(const DtArgs& g, int split, int t0, int t1, int64_t r) {
    int64_t ti = -1;
    if (r < g.sink_end)
        ti = r / kKT;
    else if (r >= g.lo && r < g.hi)
        ti = g.n_sink_tiles + (r - g.lo) / kKT;
    return ti >= 0 ? (ti >= t0 && ti < t1) : split == 0;
}

// The new cache rows this CTA owns, its KV head's columns (128 floats = 32
// float4 per row, one per lane), into `cache` before any TMA read of them:
// each lane's generic writes are fenced against the async proxy.  With
// `turn` (the keys under a rotary embedding) channel d < rotary_dim of row r
// is turned at position r with its pair partner, as op "rope" turns it.
__device__ __forceinline__ void write_new_rows(const DtArgs& g, int split, int t0, int t1, int hk, int lane,
                                               float* cache, const float* rows, bool turn) {
    const int64_t width4 = (int64_t)g.a.Hk * (kD / 4);
    for (int64_t r = g.cw.lo; r < g.cw.hi; ++r) {
        if (!owns_row(g, split, t0, t1, r)) continue;
        const int64_t src4 = (r - g.cw.lo) * width4 + hk * (kD / 4);
        float4 x = reinterpret_cast<const float4*>(rows)[src4 + lane];
        if (turn) {
            float* e = reinterpret_cast<float*>(&x);
            const float* src = rows + src4 * 4;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int d = 4 * lane + c;
                if (d >= 2 * g.rope.half) continue;
                int j, partner;
                bool first;
                rope_pair_of(g.rope, d, j, partner, first);
                e[c] = rope_channel(e[c], __ldg(src + partner), first, rope_cos_sin(g.rope, r, j));
            }
        }
        reinterpret_cast<float4*>(cache)[r * width4 + hk * (kD / 4) + lane] = x;
    }
    asm volatile("fence.proxy.async.global;\n" ::: "memory");
    __syncwarp();
}

// The last CTA of a KV head to arrive merges the splits' partials:
// m* = max m_i, weights 2^(m_i - m*) (kept in shared memory, in the score
// ring, idle by now), l* = sum l_i 2^(m_i - m*); warp v serves virtual head
// v; then output (v, d) = sum_i w_i o_i[d] / l*.
__device__ __noinline__ void merge_splits(const DtArgs& g, unsigned char* smem_raw, float* sinv, int* s_is_last) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, hk = blockIdx.x;
    if (threadIdx.x == 0) {
        unsigned ticket;
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(&g.counters[hk]) : "memory");
        *s_is_last = ticket == (unsigned)(g.splits - 1);
    }
    __syncthreads();
    if (!*s_is_last) return;
    const int nsub = g.splits;
    float* sw = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // Thread t: virtual head t / 32, dims 4 (t % 32) .. + 3.  Its first 16
    // partial outputs are loaded before the weights are worked out, so the
    // two round trips to L2 overlap.
    static_assert(kNV * kD / 4 == kThreads, "one output quad per thread");
    constexpr int kCh = 16;
    const int v = threadIdx.x / (kD / 4), d4 = threadIdx.x % (kD / 4);
    const float4* po = reinterpret_cast<const float4*>(g.part_o) + ((int64_t)hk * kNV + v) * nsub * (kD / 4) + d4;
    float4 ov[kCh];
    auto load_chunk = [&](int i0) {
#pragma unroll
        for (int c = 0; c < kCh; ++c)
            ov[c] = (v < g.nv && i0 + c < nsub) ? __ldcg(po + (int64_t)(i0 + c) * (kD / 4))
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    load_chunk(0);
    // Warp w, virtual head w: m* = max m_i, weights 2^(m_i - m*) into shared
    // memory (the score ring, idle by now), l* = sum l_i 2^(m_i - m*).
    if (warp < g.nv) {
        const int64_t row = (int64_t)hk * kNV + warp;
        constexpr int kPer = kDecodeTcMaxSplits / 32;
        float mv[kPer], lv[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = lane + 32 * k;
            mv[k] = i < nsub ? __ldcg(g.part_m + row * nsub + i) : -INFINITY;
            lv[k] = i < nsub ? __ldcg(g.part_l + row * nsub + i) : 0.f;
        }
        float m = -INFINITY;
#pragma unroll
        for (int k = 0; k < kPer; ++k) m = fmaxf(m, mv[k]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, off));
        float l = 0.f;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = lane + 32 * k;
            const float w = m == -INFINITY ? 0.f : fast_exp2(mv[k] - m);  // 0 for a split that saw nothing
            if (i < nsub) sw[warp * nsub + i] = w;
            l = fmaf(lv[k], w, l);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(FULL, l, off);
        if (lane == 0) sinv[warp] = l > 0.f ? 1.f / l : 0.f;
    }
    __syncthreads();
    if (v < g.nv) {
        const float* wv = sw + v * nsub;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i0 = 0;;) {
#pragma unroll
            for (int c = 0; c < kCh; ++c) {
                const float w = i0 + c < nsub ? wv[i0 + c] : 0.f;
                acc.x = fmaf(w, ov[c].x, acc.x);
                acc.y = fmaf(w, ov[c].y, acc.y);
                acc.z = fmaf(w, ov[c].z, acc.z);
                acc.w = fmaf(w, ov[c].w, acc.w);
            }
            i0 += kCh;
            if (i0 >= nsub) break;
            load_chunk(i0);
        }
        const float si = sinv[v];
        const int t = v / g.a.G, h = hk * g.a.G + v % g.a.G;
        reinterpret_cast<float4*>(g.a.out + ((int64_t)t * g.a.H + h) * kD)[d4] =
            make_float4(acc.x * si, acc.y * si, acc.z * si, acc.w * si);
    }
    if (threadIdx.x == 0) g.counters[hk] = 0u;  // ready for the next call
}

// ---- 2: the split-KV attention ----------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const DtArgs g) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~uintptr_t(1023));
    unsigned char* kring = base;                              // kNK slots
    unsigned char* vring = kring + kNK * kKSlot;              // kNVR slots
    unsigned char* qsm = vring + kNVR * kBlockBytes;          // Q_hi chunks, Q_lo chunks
    unsigned char* pt = qsm + kQBytes;                        // per group: P^T hi blocks, then lo blocks
    __shared__ __align__(8) uint64_t kfull[kNK], kempty[kNK], split_done[kNK], vfull[kNVR], vempty[kNVR],
        s_full[2], s_free[2], q_full, p_full[2], p_free[2], vt_full, vt_free[2], o_full[2], o_free[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ __align__(16) float red_max[2][4][kNV], red_sum[2][4][kNV];  // [group][warp][head]
    __shared__ __align__(16) float alpha_s[2][2][kNV];  // [group][its tile parity][head]
    __shared__ __align__(16) int32_t vis_lo[kNV], vis_hi[kNV], vis_shi[kNV];  // per virtual head
    __shared__ float sinv[kNV];  // merge: 1 / l* per virtual head
    __shared__ int s_is_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hk = blockIdx.x, split = blockIdx.y;
    const int col0 = hk * kD;  // the KV head's first column in the caches
    int t0, t1;
    split_tiles(g, split, t0, t1);
    const int ntile = t1 - t0;
    const int nk = ntile * kC;  // items of each ring

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNK; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kempty[i], kKReleases);
            mbar_init(&split_done[i], 4);
        }
        for (int i = 0; i < kNVR; ++i) {
            mbar_init(&vfull[i], 1);
            mbar_init(&vempty[i], 1);
        }
        for (int b = 0; b < 2; ++b) {  // per softmax group (its tiles use buffer b)
            mbar_init(&s_full[b], 1);
            mbar_init(&s_free[b], 4);
            mbar_init(&p_full[b], 4);
            mbar_init(&p_free[b], 1);
            mbar_init(&o_full[b], 1);
            mbar_init(&o_free[b], 4);
            mbar_init(&vt_free[b], 1);  // P.V of the tiles with parity b is done with V^T
        }
        mbar_init(&q_full, 8);  // the softmax warps, once the query tiles are in place
        mbar_init(&vt_full, 4);
        fence_barrier_init();
    }
    if (threadIdx.x < kNV) {
        // Visible keys of virtual head v (query row v / G): the window's
        // range [lo, hi] and the sinks up to vis_shi (int32: S < 2^31).
        const AttnDesc& a = g.a;
        const int v = threadIdx.x;
        int64_t lo = a.S, hi = -1, shi = -1;
        if (v < g.nv) {
            const int64_t pos = a.pos_offset + v / a.G;
            hi = a.causal ? pos : (a.window > 0 ? pos + a.window : a.S - 1);
            lo = a.window > 0 ? (a.causal ? pos - a.window + 1 : pos - a.window) : 0;
            shi = a.causal ? pos : a.S - 1;
            if (hi > a.S - 1) hi = a.S - 1;
            if (shi > a.S - 1) shi = a.S - 1;
            if (lo < 0) lo = 0;
            if (lo > a.S) lo = a.S;
            if (hi < -1) hi = -1;
            if (shi < -1) shi = -1;
        }
        vis_lo[v] = (int32_t)lo;
        vis_hi[v] = (int32_t)hi;
        vis_shi[v] = (int32_t)shi;
    }
    if (warp == 1) tmem_alloc(&tmem_base_s, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp == 0 || warp == 2) {
        // ---- producers: warp 0 the score ring, warp 2 the value ring; first
        // the step's new K (warp 0) or V (warp 2) rows this CTA reads ----
        if (g.cw.hi > g.cw.lo)
            write_new_rows(g, split, t0, t1, hk, lane, warp == 0 ? g.cw.kc : g.cw.vc,
                           warp == 0 ? g.cw.k_new : g.cw.v_new, warp == 0 && g.rope.half > 0);
        if (lane == 0) {
            const bool scores = warp == 0;
            const CUtensorMap* map = scores ? &tm_k : &tm_v;
            const int ns = scores ? kNK : kNVR;
            const uint32_t slot_bytes = scores ? kKSlot : kBlockBytes;
            unsigned char* ring = scores ? kring : vring;
            uint64_t* fullb = scores ? kfull : vfull;
            uint64_t* emptyb = scores ? kempty : vempty;
            prefetch_tensormap(map);
            int it = 0;
            for (; it < nk; ++it) {
                const int s = it % ns;
                const int tl = it / kC, c = it % kC;
                if (it >= ns && !mbar_wait(&emptyb[s], (uint32_t)((it / ns - 1) & 1))) {
                    raise_device_error(&g_decode_tc_device_error, kErrDtEmpty);
                    break;
                }
                int64_t r0, rend;
                tile_rows(g, t0 + tl, r0, rend);
                mbar_arrive_expect_tx(&fullb[s], kBlockBytes);
                tma_load_2d(ring + (size_t)s * slot_bytes, map, col0 + 32 * c, (int)r0, &fullb[s]);
            }
            // No copy may be in flight when the CTA exits.
            for (int j = it - ns < 0 ? 0 : it - ns; j < it; ++j)
                if (!mbar_wait(&fullb[j % ns], (uint32_t)((j / ns) & 1)))
                    raise_device_error(&g_decode_tc_device_error, kErrDtDrain);
        }
    } else if (warp == 1) {
        // ---- score MMAs: S^T = K_hi.Q_hi + K_hi.Q_lo + K_lo.Q_hi into buffer tl & 1 ----
        if (lane == 0 && nk > 0) {
            constexpr uint32_t idesc = idesc_tf32(kKT, kNV);
            bool ok = mbar_wait(&q_full, 0);
            if (!ok) raise_device_error(&g_decode_tc_device_error, kErrDtFull);
            uint32_t sd_phase = 0;  // one parity bit per slot
            for (int it = 0; ok && it < nk; ++it) {
                const int s = it % kNK;
                const int tl = it / kC, c = it % kC;
                const int b = tl & 1;
                if (c == 0 && tl >= 2 && !mbar_wait(&s_free[b], (uint32_t)(((tl - 2) >> 1) & 1))) {
                    raise_device_error(&g_decode_tc_device_error, kErrDtFree);
                    break;
                }
                if (!mbar_wait(&split_done[s], (sd_phase >> s) & 1u)) {
                    raise_device_error(&g_decode_tc_device_error, kErrDtSplit);
                    break;
                }
                sd_phase ^= 1u << s;
                tc_fence_after();
                unsigned char* slot = kring + (size_t)s * kKSlot;
                const uint64_t khi = smem_desc_sw128(slot);
                const uint32_t klo = tmem + kColKlo + 32 * s;  // K_lo of the slot: TMEM operand A
                const uint64_t qhi = smem_desc_sw128(qsm + c * kQChunk);
                const uint64_t qlo = smem_desc_sw128(qsm + (kC + c) * kQChunk);
                const uint32_t d = tmem + kColS + b * kNV;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    mma_tf32_ss(d, khi + 2 * k, qhi + 2 * k, idesc, (c > 0 || k > 0) ? 1u : 0u);
                    mma_tf32_ss_acc(d, khi + 2 * k, qlo + 2 * k, idesc);
                    mma_tf32_ts_acc(d, klo + 8 * k, qhi + 2 * k, idesc);
                }
                mma_commit(&kempty[s]);
                if (c == kC - 1) mma_commit(&s_full[b]);
            }
        }
    } else if (warp == 3) {
        // ---- P.V MMAs: O^T[dims, heads] = V^T_hi.P^T_hi + V^T_hi.P^T_lo + V^T_lo.P^T_hi ----
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_tf32(kD, kNV);
            for (int tl = 0; tl < ntile; ++tl) {
                const int b = tl & 1;
                if (!mbar_wait(&p_full[b], (uint32_t)((tl >> 1) & 1)) || !mbar_wait(&vt_full, (uint32_t)(tl & 1))) {
                    raise_device_error(&g_decode_tc_device_error, kErrDtPV);
                    break;
                }
                if (tl >= 2 && !mbar_wait(&o_free[b], (uint32_t)(((tl - 2) >> 1) & 1))) {
                    raise_device_error(&g_decode_tc_device_error, kErrDtPV);
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + kColO + b * kNV;
#pragma unroll
                for (int j = 0; j < kKT / 8; ++j) {  // 8 rows of the tile per MMA
                    const uint32_t vhi = tmem + kColVhi + 8 * j, vlo = tmem + kColVlo + 8 * j;
                    unsigned char* ptb = pt + b * kPTBytes;
                    const uint64_t phi = smem_desc_sw128(ptb + (j >> 2) * kQChunk) + 2 * (j & 3);
                    const uint64_t plo = smem_desc_sw128(ptb + (kKT / 32 + (j >> 2)) * kQChunk) + 2 * (j & 3);
                    mma_tf32_ts(d, vhi, phi, idesc, j > 0 ? 1u : 0u);
                    mma_tf32_ts_acc(d, vhi, plo, idesc);
                    mma_tf32_ts_acc(d, vlo, phi, idesc);
                }
                mma_commit(&p_free[b]);
                mma_commit(&vt_free[b]);
                mma_commit(&o_full[b]);
            }
        }
    } else if (warp <= 7) {
        // ---- splitters: K block -> K_hi in place, K_lo into the slot's TMEM
        // block.  Warp 4 + q takes rows 32 q .. 32 q + 31 of the block (TMEM
        // lanes 32 q ..), a thread one row: chunk c (dims 4 c .. 4 c + 3) of
        // row r sits at byte r * 128 + (c ^ (r % 8)) * 16 (128-byte swizzle).
        const int r = 32 * (warp & 3) + lane;
        const uint32_t rlanes = (uint32_t)(32 * (warp & 3)) << 16;
        uint32_t f_phase = 0;
        for (int it = 0; it < nk; ++it) {
            const int s = it % kNK;
            const bool got = __all_sync(FULL, mbar_wait(&kfull[s], (f_phase >> s) & 1u));
            f_phase ^= 1u << s;
            if (!got) {
                raise_device_error(&g_decode_tc_device_error, kErrDtFull);
                break;
            }
            float4* row = reinterpret_cast<float4*>(kring + (size_t)s * kKSlot + r * 128);
            float lo[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int pc = c ^ (r & 7);
                const float4 x = row[pc];
                const float4 h = make_float4(tf32_trunc(x.x), tf32_trunc(x.y), tf32_trunc(x.z), tf32_trunc(x.w));
                row[pc] = h;
                lo[4 * c + 0] = x.x - h.x;
                lo[4 * c + 1] = x.y - h.y;
                lo[4 * c + 2] = x.z - h.z;
                lo[4 * c + 3] = x.w - h.w;
            }
            tmem_st32(tmem + rlanes + kColKlo + 32 * s, lo);
            tmem_wait_st();
            tc_fence_before();
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // generic writes -> MMA
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&split_done[s]);
                mbar_arrive(&kempty[s]);  // the MMAs hold the slot until their own commits
            }
        }
    } else {
        // ---- softmax groups: warps 8 .. 11 take the even tiles, 12 .. 15 the
        // odd ones; thread = a row of the tile, all 16 heads ----
        const int grp = (warp - 8) >> 2;
        const int quarter = warp & 3;           // TMEM lanes 32 quarter .. + 31
        const int key_l = 32 * quarter + lane;  // this thread's row of a tile
        const uint32_t lanes = (uint32_t)(32 * quarter) << 16;
        // The query tiles: q of virtual head v (row v / G, head hk G + v % G)
        // scaled by scale log2 e, split into Q_hi (tf32, rounded to nearest)
        // and Q_lo = q - Q_hi, in the K-major blocks the score MMA reads
        // (block = dim / 32, head v's row of a block is 128 bytes, 128-byte
        // swizzle); zero rows past T G.  Under a rotary embedding q is
        // turned first (row t at position posOffset + t, as op "rope" turns
        // it), with the T x rotary_dim/2 (cos, sin) pairs worked out once into
        // group 0's P^T buffer, idle until the first score tile (which needs
        // every softmax warp's query tiles).
        {
            const int u = threadIdx.x - 8 * 32;  // 0 .. 255
            constexpr int kPer = kNV * kD / 256;
            const int half = g.rope.half;
            float qv[kPer], qp[kPer];  // every load in flight before the first shared store
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int idx = u + 256 * k, v = idx / kD, dd = idx % kD;
                const float* qrow = g.a.q + ((int64_t)(v / g.a.G) * g.a.H + hk * g.a.G + v % g.a.G) * kD;
                qv[k] = v < g.nv ? __ldg(qrow + dd) : 0.f;
                qp[k] = 0.f;
                if (half > 0 && v < g.nv && dd < 2 * half) {
                    int j, partner;
                    bool first;
                    rope_pair_of(g.rope, dd, j, partner, first);
                    qp[k] = __ldg(qrow + partner);
                }
            }
            if (half > 0) {
                float2* cs = reinterpret_cast<float2*>(pt);  // [t][j]; T half <= 16 x 128 pairs = kPTBytes
                const int rows_t = g.nv / g.a.G;
                for (int i = u; i < rows_t * half; i += 256)
                    cs[i] = rope_cos_sin(g.rope, g.a.pos_offset + i / half, i % half);
                softmax_sync_and(true);
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int idx = u + 256 * k, v = idx / kD, dd = idx % kD;
                    if (v < g.nv && dd < 2 * half) {
                        int j, partner;
                        bool first;
                        rope_pair_of(g.rope, dd, j, partner, first);
                        qv[k] = rope_channel(qv[k], qp[k], first, cs[(v / g.a.G) * half + j]);
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int idx = u + 256 * k, v = idx / kD, dd = idx % kD;
                const float xq = qv[k] * g.a.qk_mul;
                const float qh = tf32_rna(xq);
                const int e = dd & 31;
                const uint32_t off = v * 128 + (((e >> 2) ^ (v & 7)) << 4) + (e & 3) * 4;
                *reinterpret_cast<float*>(qsm + (dd >> 5) * kQChunk + off) = qh;
                *reinterpret_cast<float*>(qsm + (kC + (dd >> 5)) * kQChunk + off) = xq - qh;
            }
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // generic writes -> MMA
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_full);
        }
        float o[kNV];  // O^T of dim 32 quarter + lane, every head
        float m_ref[kNV];
#pragma unroll
        for (int h = 0; h < kNV; ++h) {
            o[h] = 0.f;
            m_ref[h] = -INFINITY;
        }
        float l_run = 0.f;  // head `lane` (lane < 16) of the group's first warp
        bool ok = true;
        // V^T of tile vl, once the previous tile's P.V MMAs are done with
        // V^T.  Row kk, dim lane of a V block sits at byte kk * 128 +
        // ((lane / 4) ^ (kk % 8)) * 16 + (lane % 4) * 4 (128-byte swizzle).
        // Slot (t % 2) * 4 + q holds block q of tile t, and the groups take
        // turns (the group of tile t moves tile t + 1).  An mbarrier wait only
        // checks a phase's parity, so each wait below is for a phase at most
        // one ahead of one this group has already seen complete: the P.V of
        // tile vl - 1 is waited on the barrier of that tile's parity, which
        // only this group (the group of tile vl - 1) waits on, one tile after
        // the other; and that wait comes first because it also means block q
        // of tile vl - 2 has been taken out of the slot (the P.V of tile
        // vl - 1 started only after tile vl - 1's V was moved, which came
        // after tile vl - 2's).
        auto move_v = [&](int vl) -> bool {
            const int vi = vl * kC + quarter, vs = vi % kNVR;  // the ring item and its slot
            const bool vok = (vl == 0 || __all_sync(FULL, mbar_wait(&vt_free[(vl - 1) & 1], (uint32_t)(((vl - 1) >> 1) & 1)))) &&
                             __all_sync(FULL, mbar_wait(&vfull[vs], (uint32_t)((vi / kNVR) & 1)));
            if (!vok) {
                raise_device_error(&g_decode_tc_device_error, kErrDtV);
                return false;
            }
            tc_fence_after();
            const unsigned char* vblk = vring + (size_t)vs * kBlockBytes;
            const int lane_off = (lane & 3) * 4, lane_chunk = lane >> 2;
#pragma unroll 1
            for (int ch = 0; ch < kKT / 16; ++ch) {
                float vh[16], vlo[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const int kk = 16 * ch + r;
                    const float xv =
                        *reinterpret_cast<const float*>(vblk + kk * 128 + ((lane_chunk ^ (kk & 7)) << 4) + lane_off);
                    vh[r] = tf32_trunc(xv);
                    vlo[r] = xv - vh[r];
                }
                tmem_st16(tmem + lanes + kColVhi + 16 * ch, vh);
                tmem_st16(tmem + lanes + kColVlo + 16 * ch, vlo);
            }
            tmem_wait_st();
            tc_fence_before();
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // read before TMA refills the slot
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&vempty[vs]);
                mbar_arrive(&vt_full);
            }
            return true;
        };
        // o = o * alpha + O for the group's tile number fj (its P.V done).
        auto fold = [&](int fj) -> bool {
            if (!__all_sync(FULL, mbar_wait(&o_full[grp], (uint32_t)(fj & 1)))) {
                raise_device_error(&g_decode_tc_device_error, kErrDtPV);
                return false;
            }
            tc_fence_after();
            float acc[kNV];
            tmem_ld16(tmem + lanes + kColO + grp * kNV, acc);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[grp]);
            const float4* al = reinterpret_cast<const float4*>(alpha_s[grp][fj & 1]);
#pragma unroll
            for (int h4 = 0; h4 < kNV / 4; ++h4) {
                const float4 a4 = al[h4];
                o[4 * h4 + 0] = fmaf(o[4 * h4 + 0], a4.x, acc[4 * h4 + 0]);
                o[4 * h4 + 1] = fmaf(o[4 * h4 + 1], a4.y, acc[4 * h4 + 1]);
                o[4 * h4 + 2] = fmaf(o[4 * h4 + 2], a4.z, acc[4 * h4 + 2]);
                o[4 * h4 + 3] = fmaf(o[4 * h4 + 3], a4.w, acc[4 * h4 + 3]);
            }
            return true;
        };
        // Reduce-scatter of 16 values over the warp's 32 rows: lane ends with
        // the reduction for head lane / 2 (five shuffle steps, 16 shuffles).
        auto reduce16 = [&](const float (&v)[kNV], bool is_max) -> float {
            auto op = [&](float a, float b) { return is_max ? fmaxf(a, b) : a + b; };
            float a8[8], a4[4], a2[2];
            const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                a8[i] = op(b4 ? v[i + 8] : v[i], __shfl_xor_sync(FULL, b4 ? v[i] : v[i + 8], 16));
#pragma unroll
            for (int i = 0; i < 4; ++i)
                a4[i] = op(b3 ? a8[i + 4] : a8[i], __shfl_xor_sync(FULL, b3 ? a8[i] : a8[i + 4], 8));
#pragma unroll
            for (int i = 0; i < 2; ++i)
                a2[i] = op(b2 ? a4[i + 2] : a4[i], __shfl_xor_sync(FULL, b2 ? a4[i] : a4[i + 2], 4));
            float r = op(b1 ? a2[1] : a2[0], __shfl_xor_sync(FULL, b1 ? a2[0] : a2[1], 2));
            return op(r, __shfl_xor_sync(FULL, r, 1));
        };
        auto group_sync = [&](bool v) -> bool {  // named barrier 1 or 2 of the group
            return grp == 0 ? group_sync_and<1>(v) : group_sync_and<2>(v);
        };
        int j = 0;  // the group's tile count
        // Group 1 moves the first tile's V while group 0 takes its scores.
        if (grp == 1 && ntile > 0 && !move_v(0)) ok = false;
        for (int tl = grp; tl < ntile; tl += 2, ++j) {
            // A wait that gives up marks the warp; every warp of the group still
            // reaches the barriers below, which AND the marks, so the group
            // leaves together (no warp waits alone).
            float x[kNV];
#pragma unroll
            for (int h = 0; h < kNV; ++h) x[h] = -INFINITY;
            if (ok && !__all_sync(FULL, mbar_wait(&s_full[grp], (uint32_t)(j & 1)))) {
                raise_device_error(&g_decode_tc_device_error, kErrDtS);
                ok = false;
            }
            if (ok) {
                tc_fence_after();
                tmem_ld16(tmem + lanes + kColS + grp * kNV, x);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[grp]);  // the next score MMAs may overwrite buffer grp
            }
            int64_t r0, rend;
            tile_rows(g, t0 + tl, r0, rend);
            const int key = (int)(r0 + key_l);
            const int kend = (int)rend;
#pragma unroll
            for (int h4 = 0; h4 < kNV / 4; ++h4) {
                const int4 lo4 = reinterpret_cast<const int4*>(vis_lo)[h4];
                const int4 hi4 = reinterpret_cast<const int4*>(vis_hi)[h4];
                const int4 sh4 = reinterpret_cast<const int4*>(vis_shi)[h4];
                const int lo[4] = {lo4.x, lo4.y, lo4.z, lo4.w}, hi[4] = {hi4.x, hi4.y, hi4.z, hi4.w},
                          sh[4] = {sh4.x, sh4.y, sh4.z, sh4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const bool vis = key < kend && ((key >= lo[u] && key <= hi[u]) ||
                                                    (key < g.sink_lim && key <= sh[u]));
                    if (!vis) x[4 * h4 + u] = -INFINITY;
                }
            }
            // Tile max per head: the warp's 32 rows, then the group's 4 warps.
            const float wmax = reduce16(x, true);
            if (!(lane & 1)) red_max[grp][quarter][lane >> 1] = wmax;
            ok = group_sync(ok);
            if (!ok) break;
            float alpha[kNV];
#pragma unroll
            for (int h4 = 0; h4 < kNV / 4; ++h4) {
                float4 m4 = reinterpret_cast<const float4*>(red_max[grp][0])[h4];
#pragma unroll
                for (int q2 = 1; q2 < 4; ++q2) {
                    const float4 n4 = reinterpret_cast<const float4*>(red_max[grp][q2])[h4];
                    m4 = make_float4(fmaxf(m4.x, n4.x), fmaxf(m4.y, n4.y), fmaxf(m4.z, n4.z), fmaxf(m4.w, n4.w));
                }
                const float mt[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int h = 4 * h4 + u;
                    alpha[h] = 1.f;
                    if (mt[u] > m_ref[h] + kRescaleLog2) {  // lazy: keep the reference unless beaten by > 2^8
                        alpha[h] = fast_exp2(m_ref[h] - mt[u]);  // 0 while nothing was visible
                        m_ref[h] = mt[u];
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < kNV; ++h) x[h] = fast_exp2(x[h] - (m_ref[h] == -INFINITY ? 0.f : m_ref[h]));
            // P^T[head][row] into the group's K-major blocks (block = row / 32,
            // head h's row of a block is 128 bytes, 128-byte swizzle), hi and lo.
            if (j > 0 && !__all_sync(FULL, mbar_wait(&p_free[grp], (uint32_t)((j - 1) & 1)))) {
                raise_device_error(&g_decode_tc_device_error, kErrDtPV);
                ok = false;
            }
            if (ok) {
                unsigned char* blk_hi = pt + grp * kPTBytes + quarter * kQChunk;
                unsigned char* blk_lo = blk_hi + (kKT / 32) * kQChunk;
#pragma unroll
                for (int h = 0; h < kNV; ++h) {
                    const uint32_t off = h * 128 + (((lane >> 2) ^ (h & 7)) << 4) + (lane & 3) * 4;
                    const float ph = tf32_rna(x[h]);
                    *reinterpret_cast<float*>(blk_hi + off) = ph;
                    *reinterpret_cast<float*>(blk_lo + off) = x[h] - ph;
                }
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // generic writes -> MMA
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[grp]);
            }
            const float wsum = reduce16(x, false);
            if (!(lane & 1)) red_sum[grp][quarter][lane >> 1] = wsum;
            if (quarter == 0 && lane == 0) {
                float4* as = reinterpret_cast<float4*>(alpha_s[grp][j & 1]);
#pragma unroll
                for (int h4 = 0; h4 < kNV / 4; ++h4)
                    as[h4] = make_float4(alpha[4 * h4], alpha[4 * h4 + 1], alpha[4 * h4 + 2], alpha[4 * h4 + 3]);
            }
            ok = group_sync(ok);
            if (!ok) break;
            if (quarter == 0 && lane < kNV)
                l_run = fmaf(l_run, alpha_s[grp][j & 1][lane],
                             red_sum[grp][0][lane] + red_sum[grp][1][lane] + red_sum[grp][2][lane] +
                                 red_sum[grp][3][lane]);
            // A failed wait leaves the warp's mark for the next barrier.
            if (ok && j > 0 && !fold(j - 1)) ok = false;
            // The next tile's V: its P.V follows this tile's, which is issued
            // by now (this group's P^T and the other group's V^T are in).
            if (ok && tl + 1 < ntile && !move_v(tl + 1)) ok = false;
        }
        if (ok && j > 0 && !fold(j - 1)) ok = false;
        // The two groups' partial sums into one: group 1 leaves (m, l, o) in
        // the idle value ring, group 0 rescales both to the larger reference
        // and writes the CTA's partial.  (Every V block has been moved and
        // every P.V product is done once the groups have folded their last
        // tiles.)
        float* xm = reinterpret_cast<float*>(vring);  // [16] m, [16] l, then [16][128] o
        if (grp == 1) {
            if (quarter == 0 && lane < kNV) {
                float mm = m_ref[0];
#pragma unroll
                for (int h = 1; h < kNV; ++h)
                    if (lane == h) mm = m_ref[h];
                xm[lane] = j > 0 ? mm : -INFINITY;
                xm[kNV + lane] = j > 0 ? l_run : 0.f;
            }
#pragma unroll
            for (int h = 0; h < kNV; ++h) xm[2 * kNV + h * kD + 32 * quarter + lane] = o[h];
        }
        ok = softmax_sync_and(ok);
        if (grp == 0 && ok) {
            const int64_t rows = (int64_t)hk * kNV;
#pragma unroll
            for (int h = 0; h < kNV; ++h) {
                const float m0 = j > 0 ? m_ref[h] : -INFINITY, m1 = xm[h];
                const float mx = fmaxf(m0, m1);
                const float a0 = mx == -INFINITY ? 0.f : fast_exp2(m0 - mx);  // 0 for a group that saw nothing
                const float a1 = mx == -INFINITY ? 0.f : fast_exp2(m1 - mx);
                g.part_o[((rows + h) * g.splits + split) * kD + 32 * quarter + lane] =
                    o[h] * a0 + xm[2 * kNV + h * kD + 32 * quarter + lane] * a1;
                if (quarter == 0 && lane == h) {
                    g.part_m[(rows + h) * g.splits + split] = mx;
                    g.part_l[(rows + h) * g.splits + split] = l_run * a0 + xm[kNV + h] * a1;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }

    // ---- the last CTA of this KV head merges the splits' partials ----
    // (Indices are taken afresh here so that nothing stays live across the
    // roles above.)  The barrier above orders every thread's partial stores
    // before thread 0's ticket, an acquire-release atomic at gpu scope: it
    // publishes this CTA's partials and, for the last CTA, acquires the
    // others'.
    merge_splits(g, smem_raw, sinv, &s_is_last);
}


PFN_cuTensorMapEncodeTiled_v12000 dt_encoder() {
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

// Row-major [rows, cols] f32, boxes of 32 columns x box_rows rows, 128-byte swizzle.
bool encode_blocks(CUtensorMap* map, const float* p, int64_t rows, int64_t cols, int box_rows) {
    return cached_tensor_map(map, p, rows, cols, 32, box_rows, 3, [&](CUtensorMap* m) {
        auto fn = dt_encoder();
        if (!fn) return false;
        const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)cols * sizeof(float)};
        const cuuint32_t box[2] = {32u, (cuuint32_t)box_rows};
        const cuuint32_t estr[2] = {1, 1};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(p), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    });
}

size_t up256(size_t b) { return (b + 255) / 256 * 256; }

cudaError_t launch_d(const AttnDesc& a, const DecodeTcPlan& tp, void* workspace, cudaStream_t stream,
                     const DecodeCacheWrite* cw, const RopeDev* rope) {
    unsigned char* ws = static_cast<unsigned char*>(workspace) + kWorkspaceHeader;
    const size_t rows = (size_t)a.Hk * kNV * tp.splits;
    float* part_m = reinterpret_cast<float*>(ws);
    float* part_l = part_m + up256(rows * 4) / 4;
    float* part_o = part_l + up256(rows * 4) / 4;

    CUtensorMap tm_k, tm_v;
    if (!encode_blocks(&tm_k, a.k, a.S, (int64_t)a.Hk * kD, kKT) ||
        !encode_blocks(&tm_v, a.v, a.S, (int64_t)a.Hk * kD, kKT))
        return cudaErrorInvalidValue;
    DtArgs g;
    std::memset(&g, 0, sizeof(g));
    g.a = a;
    g.part_m = part_m;
    g.part_l = part_l;
    g.part_o = part_o;
    g.counters = static_cast<unsigned int*>(workspace);  // the workspace header
    g.nv = (int32_t)(a.T * a.G);
    g.sink_lim = a.window > 0 ? (int32_t)(a.sinks < a.S ? a.sinks : a.S) : 0;
    if (cw && cw->hi > cw->lo) g.cw = *cw;
    g.splits = tp.splits;
    g.sink_splits = tp.sink_splits;
    g.n_sink_tiles = tp.n_sink_tiles;
    g.n_tiles = tp.n_tiles;
    g.lo = tp.lo;
    g.sink_end = tp.sink_end;
    g.hi = tp.hi;
    if (rope) g.rope = *rope;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(decode_tc_kernel), (int)kSmem);
    if (e != cudaSuccess) return e;
    decode_tc_kernel<<<dim3(a.Hk, tp.splits), kThreads, kSmem, stream>>>(tm_k, tm_v, g);
    return cudaGetLastError();
}

}  // namespace

bool decode_tc_supported(const AttnDesc& a) {
    return a.T >= 1 && a.T * a.G <= kNV && a.D == kD && a.Dv == kD && !a.softcap_on &&
           !a.alibi_on && a.bias_kind == 0 && a.S < ((int64_t)1 << 31) &&
           a.Hk <= kMaxDecodeKvHeads;  // one arrival counter per KV head in the workspace header
}

void decode_tc_plan(const AttnDesc& a, int forced_splits, int num_sms, DecodeTcPlan* tp) {
    DecodePlan base;
    decode_plan(a, 0, 1, &base);  // the visible range and the sink range
    tp->lo = base.s_lo;
    tp->hi = base.s_end;
    tp->sink_end = base.sink_end;
    tp->n_sink_tiles = (int)((base.sink_end + kKT - 1) / kKT);
    tp->n_tiles = (int)((base.s_end - base.s_lo + kKT - 1) / kKT);
    const int total = tp->n_sink_tiles + tp->n_tiles;
    int splits = forced_splits > 0 ? forced_splits : num_sms / (a.Hk > 0 ? a.Hk : 1);
    if (splits < 1) splits = 1;
    if (splits > kDecodeTcMaxSplits) splits = kDecodeTcMaxSplits;
    if (splits > total) splits = total > 0 ? total : 1;
    // Each range takes whole splits, in proportion to its tiles.
    int ss = 0;
    if (tp->n_sink_tiles > 0) {
        ss = (int)((int64_t)splits * tp->n_sink_tiles / total);
        if (ss < 1) ss = 1;
        if (splits - ss < 1 && tp->n_tiles > 0) splits = ss + 1;
    }
    if (tp->n_tiles == 0) splits = ss;
    if (splits < 1) splits = 1;
    tp->sink_splits = ss;
    tp->splits = splits;
    const size_t rows = (size_t)a.Hk * kNV * splits;
    tp->workspace_bytes = kWorkspaceHeader + 2 * up256(rows * 4) + up256(rows * (size_t)a.D * 4);
}

cudaError_t launch_decode_tc(const AttnDesc& a, const DecodeTcPlan& tp, void* workspace, cudaStream_t stream,
                             const DecodeCacheWrite* cw, const RopeDev* rope) {
    return launch_d(a, tp, workspace, stream, cw, rope);
}

unsigned int decode_tc_take_device_error() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_decode_tc_device_error, sizeof(v)) != cudaSuccess) return 0;
    if (v) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_decode_tc_device_error, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace vtmu
