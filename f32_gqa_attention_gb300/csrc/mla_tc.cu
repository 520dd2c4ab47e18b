// mla_tc.cu -- the split-KV attention of absorbed latent attention
// (mla_attention of the IR schema page) with its score contraction on the
// tcgen05 tensor cores in 3xTF32, and P.c on the CUDA cores.
//
// Selected by kernel = 2 of vtmu_mla_params; the default is the CUDA-core
// kernel of mla.cu, which is faster on the decode shapes measured (16 heads
// over 32768 rows: 42 us against 61 us for this kernel alone).  A timeline
// of this kernel (global-timer stamps per role) shows why: with one or two
// tiles per CTA the score ring is bound by HBM latency (the first block
// lands ~4 us after the CTA starts; 18 blocks take ~12 us), and P.c, 1M
// FMAs per tile, runs at a fraction of the FMA rate because each
// 16-FMA step loads its operands through shared memory and the value ring
// (4 slots of 16 KB) cannot prefetch while every slot is in use.  P.c
// cannot move to the tensor cores without the values' key dimension
// contiguous (the cache stores rows), i.e. a transpose of every block.
//
// Every head's absorbed query q_abs[v] (576 values: the latent part, then
// the rotary part, scaled by scale * log2 e) meets the same 576-wide cache
// rows.  The roles of the MMA are swapped with respect to a prefill: a tile
// of 128 cache rows is the M side and the CTA's 16 virtual heads (query row
// x head) the N side, so one M = 128, N = 16 MMA scores 2048 (key, head)
// pairs, and the scores land in TMEM with one key per lane:
//     S^T[key, v] = sum_d K[key, d] q_abs[v, d]
// issued as K_hi.Q_hi + K_hi.Q_lo + K_lo.Q_hi (3xTF32; Q_hi / Q_lo come
// split from the absorb kernel, K is split here).  Two threads issue: one
// K_hi.Q_hi into its own accumulator, the other the two small products into
// a second one (one thread issues an MMA only every ~50 cycles, and the large
// product then takes one MMA per k-step).
//
// Work per CTA: one group of 16 virtual heads, a run of 128-row tiles of the
// cache (prefetched into L2 when the CTA starts).  Two rings: the score
// ring carries 18 items per tile (a [128 rows x 32 dims] block of the cache
// by TMA with the 128-byte swizzle, plus the heads' Q_hi / Q_lo of those 32
// dims); the value ring 16 items (the first 512 columns of the same rows
// again, from L2, for P.c), so the next tile's scores stream while this
// tile's values are used.  Warps:
//   0, 2    lane 0 streams the score ring (0) and the value ring (2) by TMA;
//   1, 3    lane 0 issues the MMAs (warp 1 owns TMEM);
//   4 .. 7  split each score block in place into K_hi (low 13 mantissa bits
//           cleared) and K_lo = K - K_hi;
//   8 .. 15 read S^T from TMEM (warps w and w + 4 share a lane quarter, each
//           half of the heads), mask, online softmax in base 2 with a lazy
//           reference max, write P[key][v] to shared memory; then P.c:
//           warps 8 + j and 12 + j share value items j, j + 4, j + 8,
//           j + 12 (32 latent dims each), one taking rows 0..63 of the tile,
//           the other rows 64..127; lane = (4 heads) x (4 dims), 16 FMAs per
//           row; the two halves are added once, at the end.
// Every role that waits on a ring releases every item of it (score ring:
// four splitter warps and the two issuers' commits; value ring: the eight
// softmax warps), after observing its arrival or using it: the TMA refills a
// slot only when every role has seen its previous item, so no role is ever
// two phases behind a slot (an mbarrier wait only checks a phase's parity).
// S is double-buffered in TMEM and P in shared memory.  The CTA writes (m, l,
// o) per virtual head, merged and projected through v_b by the kernels of
// mla.cu.  Every wait is bounded; a wait that gives up sets a bit of
// g_mla_tc_device_error.
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_common.cuh"
#include "kernels.h"
#include "launch_cache.h"
#include "tcgen05_ops.cuh"
#include "tma_sync.cuh"

namespace vtmu {

__device__ unsigned int g_mla_tc_device_error;

namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kR = kMlaKvRank, kP = kMlaRope, kW = kR + kP;
constexpr int kNV = 16;                 // virtual heads per CTA (MMA N)
constexpr int kKT = 128;                // cache rows per tile (MMA M)
constexpr int kQC = kW / 32;            // score items per tile (18)
constexpr int kVC = kR / 32;            // value items per tile (16)
constexpr int kNQ = 4;                  // score ring slots
constexpr int kNVR = 4;                 // value ring slots
// Score slot layout (bytes): cache block (hi after the split) | K_lo | Q_hi | Q_lo.
constexpr uint32_t kKBytes = kKT * 32 * 4;            // 16 KB
constexpr uint32_t kQBytes = kNV * 32 * 4;            // 2 KB
constexpr uint32_t kOffLo = kKBytes, kOffQhi = 2 * kKBytes, kOffQlo = 2 * kKBytes + kQBytes;
constexpr uint32_t kSlotBytes = 2 * kKBytes + 2 * kQBytes;  // 36 KB
constexpr uint32_t kPBytes = kKT * kNV * 4;            // 8 KB per P buffer
constexpr int kThreads = 16 * 32;
constexpr size_t kSmem = 1024 + (size_t)kNQ * kSlotBytes + (size_t)kNVR * kKBytes + 2 * kPBytes;
constexpr float kRescaleLog2 = 8.f;
constexpr uint32_t kTmemCols = 64;  // 2 buffers x 2 accumulators x 16 columns
constexpr uint32_t kQReleases = 4 + 2;  // splitter warps, issuers
constexpr uint32_t kVReleases = 8;      // softmax warps

static_assert(kSlotBytes % 1024 == 0 && kOffQhi % 1024 == 0 && kOffQlo % 1024 == 0, "1024-byte aligned tiles");
static_assert(kSmem <= 232448, "shared memory budget");

enum : unsigned int {
    kErrTcMlaFull = 1u << 20,   // a consumer gave up on an arriving ring item
    kErrTcMlaEmpty = 1u << 21,  // the producer gave up on a free slot
    kErrTcMlaSplit = 1u << 22,  // an issuer gave up on a split item
    kErrTcMlaS = 1u << 23,      // a softmax warp gave up on a score tile
    kErrTcMlaFree = 1u << 24,   // an issuer gave up on a free score buffer
    kErrTcMlaDrain = 1u << 25,  // the producer gave up draining its copies
};

struct TcArgs {
    AttnDesc a;        // S, T, H, causal, pos_offset, window, sinks (visibility)
    float* part_m;     // [V][splits]
    float* part_l;
    float* part_o;     // [V][splits][kR]
    int32_t V;         // virtual heads T * H
    int32_t splits;
    int32_t sink_splits;
    int32_t n_sink_tiles, n_tiles;  // tiles of the sink range and of the main range
    int64_t lo;        // first row of the main range (sink range starts at 0)
    int64_t sink_end, hi;
};

// Tiles [t0, t1) of this split in the concatenated (sink, main) tile list.
__device__ __forceinline__ void split_tiles(const TcArgs& g, int split, int& t0, int& t1) {
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
__device__ __forceinline__ void tile_rows(const TcArgs& g, int t, int64_t& r0, int64_t& rend) {
    if (t < g.n_sink_tiles) {
        r0 = (int64_t)t * kKT;
        rend = g.sink_end;
    } else {
        r0 = g.lo + (int64_t)(t - g.n_sink_tiles) * kKT;
        rend = g.hi;
    }
}

// Barrier over the eight softmax warps (named barrier 1, 256 threads);
// returns the AND of `v` over them.
__device__ __forceinline__ bool softmax_sync_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, 1, 256, q;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_latent_tc_kernel(const __grid_constant__ CUtensorMap tm_state, const __grid_constant__ CUtensorMap tm_qhi,
                         const __grid_constant__ CUtensorMap tm_qlo, const TcArgs g) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~uintptr_t(1023));
    unsigned char* qring = base;                                        // kNQ score slots
    unsigned char* vring = base + kNQ * kSlotBytes;                     // kNVR value slots
    float* pbuf = reinterpret_cast<float*>(vring + kNVR * kKBytes);    // [2][kKT][kNV]
    __shared__ __align__(8) uint64_t qfull[kNQ], qempty[kNQ], split_done[kNQ], vfull[kNVR], vempty[kNVR],
        s_full[2], s_free[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ float red_max[8][8], red_sum[8][8];   // per softmax warp, its 8 heads
    __shared__ __align__(16) float alpha_s[2][kNV];  // per tile: the rescale factor of each head

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = blockIdx.x, split = blockIdx.y;
    int t0, t1;
    split_tiles(g, split, t0, t1);
    const int ntile = t1 - t0;
    const int nq = ntile * kQC, nv = ntile * kVC;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNQ; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], kQReleases);
            mbar_init(&split_done[i], 4);
        }
        for (int i = 0; i < kNVR; ++i) {
            mbar_init(&vfull[i], 1);
            mbar_init(&vempty[i], kVReleases);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 2);
            mbar_init(&s_free[b], 8);
        }
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base_s, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    auto acc_col = [&](int b, int prod) -> uint32_t { return (uint32_t)((b * 2 + prod) * kNV); };

    if (warp == 0 || warp == 2) {
        // ---- producers: warp 0 the score ring, warp 2 the value ring ----
        if (lane == 0) {
            const bool scores = warp == 0;
            const int n = scores ? nq : nv, per_tile = scores ? kQC : kVC, ns = scores ? kNQ : kNVR;
            uint64_t* fullb = scores ? qfull : vfull;
            uint64_t* emptyb = scores ? qempty : vempty;
            prefetch_tensormap(&tm_state);
            if (scores) {
                prefetch_tensormap(&tm_qhi);
                prefetch_tensormap(&tm_qlo);
                // The split's rows, into L2 ahead of the ring (one HBM read;
                // the value ring reads them again from L2).
                for (int tl = 0; tl < ntile; ++tl) {
                    int64_t r0, rend;
                    tile_rows(g, t0 + tl, r0, rend);
#pragma unroll 1
                    for (int c = 0; c < kQC; ++c) tma_prefetch_2d(&tm_state, 32 * c, (int)r0);
                }
            }
            int it = 0;
            for (; it < n; ++it) {
                const int s = it % ns;
                if (it >= ns && !mbar_wait(&emptyb[s], (uint32_t)((it / ns - 1) & 1))) {
                    raise_device_error(&g_mla_tc_device_error, kErrTcMlaEmpty);
                    break;
                }
                const int tile = t0 + it / per_tile, c = it % per_tile;
                int64_t r0, rend;
                tile_rows(g, tile, r0, rend);
                if (scores) {
                    unsigned char* slot = qring + (size_t)s * kSlotBytes;
                    mbar_arrive_expect_tx(&fullb[s], kKBytes + 2 * kQBytes);
                    tma_load_2d(slot, &tm_state, 32 * c, (int)r0, &fullb[s]);
                    tma_load_2d(slot + kOffQhi, &tm_qhi, 32 * c, group * kNV, &fullb[s]);
                    tma_load_2d(slot + kOffQlo, &tm_qlo, 32 * c, group * kNV, &fullb[s]);
                } else {
                    unsigned char* slot = vring + (size_t)s * kKBytes;
                    mbar_arrive_expect_tx(&fullb[s], kKBytes);
                    tma_load_2d(slot, &tm_state, 32 * c, (int)r0, &fullb[s]);
                }
            }
            // No copy may be in flight when the CTA exits.
            for (int j = it - ns < 0 ? 0 : it - ns; j < it; ++j)
                if (!mbar_wait(&fullb[j % ns], (uint32_t)((j / ns) & 1)))
                    raise_device_error(&g_mla_tc_device_error, kErrTcMlaDrain);
        }
    } else if (warp == 1 || warp == 3) {
        // ---- issuers: warp 1 K_hi.Q_hi, warp 3 K_hi.Q_lo + K_lo.Q_hi ----
        if (lane == 0) {
            const int prod = warp == 1 ? 0 : 1;
            constexpr uint32_t idesc = idesc_tf32(kKT, kNV);
            uint32_t sd_phase = 0;  // one parity bit per slot
            for (int it = 0; it < nq; ++it) {
                const int s = it % kNQ;
                const int tl = it / kQC, c = it % kQC;
                const int b = tl & 1;
                if (c == 0 && tl >= 2 && !mbar_wait(&s_free[b], (uint32_t)(((tl - 2) >> 1) & 1))) {
                    raise_device_error(&g_mla_tc_device_error, kErrTcMlaFree);
                    break;
                }
                if (!mbar_wait(&split_done[s], (sd_phase >> s) & 1u)) {
                    raise_device_error(&g_mla_tc_device_error, kErrTcMlaSplit);
                    break;
                }
                sd_phase ^= 1u << s;
                tc_fence_after();
                unsigned char* slot = qring + (size_t)s * kSlotBytes;
                const uint64_t khi = smem_desc_sw128(slot), klo = smem_desc_sw128(slot + kOffLo);
                const uint64_t qhi = smem_desc_sw128(slot + kOffQhi), qlo = smem_desc_sw128(slot + kOffQlo);
                const uint32_t d = tmem + acc_col(b, prod);
                if (prod == 0) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) mma_tf32_ss(d, khi + 2 * k, qhi + 2 * k, idesc, (c > 0 || k > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        mma_tf32_ss(d, khi + 2 * k, qlo + 2 * k, idesc, (c > 0 || k > 0) ? 1u : 0u);
                        mma_tf32_ss_acc(d, klo + 2 * k, qhi + 2 * k, idesc);
                    }
                }
                mma_commit(&qempty[s]);
                if (c == kQC - 1) mma_commit(&s_full[b]);
            }
        }
    } else if (warp <= 7) {
        // ---- splitters: cache block -> K_hi in place, K_lo beside it ----
        const int st = threadIdx.x - 4 * 32;  // 0 .. 127
        uint32_t f_phase = 0;
        for (int it = 0; it < nq; ++it) {
            const int s = it % kNQ;
            const bool got = __all_sync(FULL, mbar_wait(&qfull[s], (f_phase >> s) & 1u));
            f_phase ^= 1u << s;
            if (!got) {
                raise_device_error(&g_mla_tc_device_error, kErrTcMlaFull);
                break;
            }
            float4* hi = reinterpret_cast<float4*>(qring + (size_t)s * kSlotBytes);
            float4* lo = reinterpret_cast<float4*>(qring + (size_t)s * kSlotBytes + kOffLo);
#pragma unroll
            for (int i = 0; i < (int)(kKBytes / 16) / 128; ++i) {
                const int j = st + 128 * i;
                const float4 x = hi[j];
                const float4 h = make_float4(tf32_trunc(x.x), tf32_trunc(x.y), tf32_trunc(x.z), tf32_trunc(x.w));
                hi[j] = h;
                lo[j] = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
            }
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // generic writes -> MMA
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&split_done[s]);
                mbar_arrive(&qempty[s]);  // the MMAs hold the slot until their own commits
            }
        }
    } else {
        // ---- softmax and P.c ----
        const int sw = warp - 8;                // 0 .. 7
        const int quarter = warp & 3;           // TMEM lanes 32 quarter .. + 31
        const int half = sw >> 2;               // heads 8 half .. + 7 of the softmax step
        const int key_l = 32 * quarter + lane;  // this thread's row of a tile
        // P.c: warps sw and sw + 4 share value items sw % 4 + 4 i (i = 0 .. 3),
        // each taking half of the tile's rows (kh); lane = (4 heads hg) x (4
        // dims dg) of an item.
        const int dg = lane & 7, hg = lane >> 3;
        const int iq = sw & 3, kh = sw >> 2;
        float o[4][4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int h = 0; h < 4; ++h) o[i][h][0] = o[i][h][1] = o[i][h][2] = o[i][h][3] = 0.f;
        // Softmax state of this thread's 8 heads (the same in every thread of the half).
        float m_ref[8], l_sum[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            m_ref[i] = -INFINITY;
            l_sum[i] = 0.f;
        }
        const int v_first = group * kNV + 8 * half;  // the half's first virtual head
        uint32_t vf_phase = 0;
        bool ok = true;
        for (int tl = 0; tl < ntile; ++tl) {
            const int b = tl & 1;
            // A wait that gives up marks the warp; every softmax warp still
            // reaches the barrier below, which ANDs the marks, so they all
            // leave together (none waits alone).
            if (ok && !__all_sync(FULL, mbar_wait(&s_full[b], (uint32_t)((tl >> 1) & 1)))) {
                raise_device_error(&g_mla_tc_device_error, kErrTcMlaS);
                ok = false;
            }
            float x[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = -INFINITY;
            if (ok) {
                tc_fence_after();
                float a0[8], a1[8];
                const uint32_t row = tmem + ((uint32_t)(32 * quarter) << 16) + 8 * half;
                tmem_ld8(row + acc_col(b, 0), a0);
                tmem_ld8(row + acc_col(b, 1), a1);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] = a0[i] + a1[i];
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free[b]);  // the next score MMAs may overwrite buffer b
            }
            int64_t r0, rend;
            tile_rows(g, t0 + tl, r0, rend);
            const int64_t key = r0 + key_l;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int v = v_first + i;
                const int64_t pos = g.a.pos_offset + (v < g.V ? v / g.a.H : 0);
                if (!(v < g.V && key < rend && key_visible<true>(g.a, pos, key))) x[i] = -INFINITY;
            }
            // Tile max per head over the 128 rows: the warp's 32, then the four
            // warps of this half through shared memory.
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float m = x[i];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, off));
                mx[i] = m;
            }
            if (lane == 0)
#pragma unroll
                for (int i = 0; i < 8; ++i) red_max[sw][i] = mx[i];
            ok = softmax_sync_and(ok);
            if (!ok) break;
            float alpha[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float m = red_max[4 * half][i];
#pragma unroll
                for (int q2 = 1; q2 < 4; ++q2) m = fmaxf(m, red_max[4 * half + q2][i]);
                alpha[i] = 1.f;
                if (m > m_ref[i] + kRescaleLog2) {  // lazy: keep the reference unless beaten by > 2^8
                    alpha[i] = fast_exp2(m_ref[i] - m);  // 0 while nothing was visible
                    m_ref[i] = m;
                }
            }
            float* pb = pbuf + (size_t)b * kKT * kNV;
            float p[8], ps[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) p[i] = fast_exp2(x[i] - (m_ref[i] == -INFINITY ? 0.f : m_ref[i]));
            *reinterpret_cast<float4*>(pb + key_l * kNV + 8 * half) = make_float4(p[0], p[1], p[2], p[3]);
            *reinterpret_cast<float4*>(pb + key_l * kNV + 8 * half + 4) = make_float4(p[4], p[5], p[6], p[7]);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float sacc = p[i];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) sacc += __shfl_xor_sync(FULL, sacc, off);
                ps[i] = sacc;
            }
            if (lane == 0)
#pragma unroll
                for (int i = 0; i < 8; ++i) red_sum[sw][i] = ps[i];
            if (quarter == 0 && lane == 0)
#pragma unroll
                for (int i = 0; i < 8; ++i) alpha_s[b][8 * half + i] = alpha[i];
            softmax_sync_and(true);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                l_sum[i] = fmaf(l_sum[i], alpha[i],
                                red_sum[4 * half][i] + red_sum[4 * half + 1][i] + red_sum[4 * half + 2][i] +
                                    red_sum[4 * half + 3][i]);
            // P.c: rescale this lane's heads, then its two value items.
            {
                const float4 a4 = *reinterpret_cast<const float4*>(&alpha_s[b][4 * hg]);
                const float al[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int h = 0; h < 4; ++h)
#pragma unroll
                        for (int d = 0; d < 4; ++d) o[i][h][d] *= al[h];
            }
            // This warp's half of the rows of one value item (32 latent dims)
            // into `acc`.
            auto pv_item = [&](const unsigned char* vblk, float (&acc)[4][4]) {
#pragma unroll 4
                for (int k2 = 0; k2 < kKT / 2; ++k2) {
                    const int kk = kh * (kKT / 2) + k2;
                    const float4 p4 = *reinterpret_cast<const float4*>(pb + kk * kNV + 4 * hg);
                    const float4 v4 = *reinterpret_cast<const float4*>(vblk + kk * 128 + ((dg ^ (kk & 7)) << 4));
                    const float pp[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        acc[h][0] = fmaf(pp[h], v4.x, acc[h][0]);
                        acc[h][1] = fmaf(pp[h], v4.y, acc[h][1]);
                        acc[h][2] = fmaf(pp[h], v4.z, acc[h][2]);
                        acc[h][3] = fmaf(pp[h], v4.w, acc[h][3]);
                    }
                }
            };
            // Every softmax warp observes and releases every value item; the
            // two warps that own it use it first.
            for (int c = 0; c < kVC; ++c) {
                const int it = tl * kVC + c, s = it % kNVR;
                const bool got = __all_sync(FULL, mbar_wait(&vfull[s], (vf_phase >> s) & 1u));
                vf_phase ^= 1u << s;
                if (!got) {
                    raise_device_error(&g_mla_tc_device_error, kErrTcMlaFull);
                    ok = false;  // the next tile's barrier takes every warp out
                    break;
                }
                if ((c & 3) == iq) {
                    const unsigned char* vblk = vring + (size_t)s * kKBytes;  // [128 rows][32 dims], 128-B swizzle
                    switch (c >> 2) {
                        case 0: pv_item(vblk, o[0]); break;
                        case 1: pv_item(vblk, o[1]); break;
                        case 2: pv_item(vblk, o[2]); break;
                        default: pv_item(vblk, o[3]); break;
                    }
                    // Read (generic proxy) before TMA refills the slot.
                    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&vempty[s]);
            }
        }
        // The two row halves of each item: the second half's warps leave
        // their sums in the (now idle) value ring, the first half's add them.
        // All eight warps reach the barrier (a failed wait only skips work).
        float* xo = reinterpret_cast<float*>(vring);  // [4 warps][4 items][16][32 lanes]
        ok = softmax_sync_and(ok);                    // every warp is done with the ring
        if (kh == 1 && ok) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int h = 0; h < 4; ++h)
#pragma unroll
                    for (int d = 0; d < 4; ++d) xo[((iq * 4 + i) * 16 + h * 4 + d) * 32 + lane] = o[i][h][d];
        }
        ok = softmax_sync_and(ok);
        // Partials of this split: m, l per head (threads of quarter 0), o per
        // (head, dim).
        if (ok) {
            if (quarter == 0 && lane < 8) {
                const int v = group * kNV + 8 * half + lane;
                if (v < g.V) {
                    const int64_t idx = (int64_t)v * g.splits + split;
                    float mm = m_ref[0], ll = l_sum[0];
#pragma unroll
                    for (int i = 1; i < 8; ++i)
                        if (lane == i) {
                            mm = m_ref[i];
                            ll = l_sum[i];
                        }
                    g.part_m[idx] = ntile > 0 ? mm : -INFINITY;
                    g.part_l[idx] = ntile > 0 ? ll : 0.f;
                }
            }
            if (kh == 0) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = iq + 4 * i;
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        float r[4];
#pragma unroll
                        for (int d = 0; d < 4; ++d) r[d] = o[i][h][d] + xo[((iq * 4 + i) * 16 + h * 4 + d) * 32 + lane];
                        const int v = group * kNV + 4 * hg + h;
                        if (v < g.V) {
                            float* po = g.part_o + ((int64_t)v * g.splits + split) * kR + 32 * c + 4 * dg;
                            *reinterpret_cast<float4*>(po) = make_float4(r[0], r[1], r[2], r[3]);
                        }
                    }
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
}

PFN_cuTensorMapEncodeTiled_v12000 tc_encoder() {
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

// Row-major [rows, kW] f32, boxes of 32 columns x box_rows rows, 128-byte swizzle.
bool encode_sw128_rows(CUtensorMap* map, const float* p, int64_t rows, int box_rows) {
    return cached_tensor_map(map, p, rows, kW, 32, box_rows, 3, [&](CUtensorMap* m) {
        auto fn = tc_encoder();
        if (!fn) return false;
        const cuuint64_t dims[2] = {(cuuint64_t)kW, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)kW * sizeof(float)};
        const cuuint32_t box[2] = {32u, (cuuint32_t)box_rows};
        const cuuint32_t estr[2] = {1, 1};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(p), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    });
}

}  // namespace

void mla_tc_plan(const MlaDesc& m, const MlaPlan& base, int num_sms, MlaTcPlan* tp) {
    const int64_t V = m.T * m.H;
    tp->groups = (int)((V + kNV - 1) / kNV);
    tp->n_sink_tiles = (int)((base.sink_end + kKT - 1) / kKT);
    tp->n_tiles = (int)((base.hi - base.lo + kKT - 1) / kKT);
    const int total = tp->n_sink_tiles + tp->n_tiles;
    int splits = num_sms / (tp->groups > 0 ? tp->groups : 1);
    if (splits < 1) splits = 1;
    if (splits > kMlaTcMaxSplits) splits = kMlaTcMaxSplits;
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
}

size_t mla_tc_smem() { return kSmem; }

cudaError_t launch_mla_latent_tc(const MlaDesc& m, const MlaPlan& base, const MlaTcPlan& tp, const float* qhi,
                                 const float* qlo, float* part_m, float* part_l, float* part_o,
                                 cudaStream_t stream) {
    CUtensorMap tm_state, tm_qhi, tm_qlo;
    const int64_t V = m.T * m.H;
    if (!encode_sw128_rows(&tm_state, m.state, m.S, kKT) || !encode_sw128_rows(&tm_qhi, qhi, V, kNV) ||
        !encode_sw128_rows(&tm_qlo, qlo, V, kNV))
        return cudaErrorInvalidValue;
    TcArgs g;
    std::memset(&g, 0, sizeof(g));
    g.a.S = m.S;
    g.a.T = m.T;
    g.a.H = m.H;
    g.a.causal = m.causal;
    g.a.pos_offset = m.pos_offset;
    g.a.window = m.window;
    g.a.sinks = m.window > 0 ? m.sinks : 0;
    g.part_m = part_m;
    g.part_l = part_l;
    g.part_o = part_o;
    g.V = (int32_t)V;
    g.splits = tp.splits;
    g.sink_splits = tp.sink_splits;
    g.n_sink_tiles = tp.n_sink_tiles;
    g.n_tiles = tp.n_tiles;
    g.lo = base.lo;
    g.sink_end = base.sink_end;
    g.hi = base.hi;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(mla_latent_tc_kernel), (int)kSmem);
    if (e != cudaSuccess) return e;
    mla_latent_tc_kernel<<<dim3(tp.groups, tp.splits), kThreads, kSmem, stream>>>(tm_state, tm_qhi, tm_qlo, g);
    return cudaGetLastError();
}

unsigned int mla_tc_take_device_error() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_mla_tc_device_error, sizeof(v)) != cudaSuccess) return 0;
    if (v) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_mla_tc_device_error, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace vtmu
