// prefill_tc.cu -- attention prefill on the tcgen05 tensor cores in 3xTF32.
//
// Op "attention" (vtmu.mpakt.dev/api/ops), f32 in and out.  Both
// contractions run on kind::tf32 UMMAs with error compensation: every f32
// operand x is split into hi = x rounded to the nearest tf32 value and
// lo = x - hi, itself rounded to tf32 (|x - hi - lo| <= 2^-22 |x|), and
// each product A.B is issued as A_hi.B_hi + A_hi.B_lo + A_lo.B_hi into f32
// accumulators.  The dropped A_lo.B_lo term is below 2^-22 relative.
// Single-pass TF32 is never used.
//
// Work split:
//  * a pre-pass (split_k_kernel, split_vt_kernel) writes K_hi / K_lo in K's
//    own layout and V^T_hi / V^T_lo transposed to [kvHeads*vHeadDim, S],
//    so every tile the MMAs read is K-major;
//  * one CTA owns 128 query rows of one head (the MMA M); per key tile of
//    BN = 64 keys, visited from the diagonal down:
//      S_j  = Q K_j^T          (TMEM accumulator, M=128)
//      P_j  = softmax part     (4 warps; thread = query row = TMEM lane;
//                               8 at headDim 256, two per lane quarter)
//      O   += P_j V_j          (TMEM accumulator, M=128 x N=vHeadDim share)
//  * operands: Q_hi and P_hi / P_lo in TMEM (A operand of the TS-form MMA),
//    Q_lo in shared memory (A operand of the SS-form MMA of the third
//    product), K and V^T hi/lo in shared memory (B operand); every shared
//    tile is K-major with the 128-byte swizzle.  The Q tile itself arrives
//    by TMA and is split in place;
//  * the two products with Q_hi come from ONE MMA: each K sub-tile holds
//    the 64 K_hi rows followed by the 64 K_lo rows, i.e. a 128-row B operand,
//    so Q_hi.[K_hi; K_lo]^T lands as [S_hihi | S_hilo] in 128 TMEM columns at
//    the full N = 128 tensor rate; the third product Q_lo.K_hi (N = 64)
//    accumulates into the second half, with the other small product, and
//    the softmax adds the two halves;
//  * TMEM columns: Q_hi | O | S | P.  At headDim <= 128 S and P are separate
//    128-column buffers: the score MMAs of tile j+1 start as soon as the
//    softmax has read S_j and run while it works on tile j; P_j (hi | lo)
//    waits only for P.V_{j-1}.  At headDim 192 P_hi takes the last 64 TMEM
//    columns and P_lo goes to shared memory (the third P.V product is then
//    SS-form), with the same overlap.  At headDim 256 P is written over S
//    and the steps alternate (vHeadDim is split over grid.z there: two CTAs,
//    each half of P.V);
//  * warp 0 lane 0 streams every K and V^T tile by TMA through one ring of
//    32 KB items (16 KB at headDim 192), in the order the MMAs consume them;
//    warp 1 owns TMEM and one of its threads issues the score MMAs, one
//    thread of warp 6 the P.V MMAs (at headDim 192 and 256 warp 1 issues
//    both, consuming the ring in order); warps 2-5 (2-9 at headDim 256)
//    split Q, run the tile-specialised epilogue and online softmax (base 2,
//    O rescaled only when a row max grows by more than 2^8), write P hi/lo
//    into TMEM and finally normalise and store O;
//  * attention sinks are a template flag: with them, the key tiles holding
//    keys before `sinks` follow the window's tiles (or join them).
//
// Every wait is bounded (tma_sync.cuh); a wait that gives up sets a bit of
// g_tc_device_error and the kernel unwinds.
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_common.cuh"
#include "softcap.cuh"
#include "kernels.h"
#include "launch_cache.h"
#include "tcgen05_ops.cuh"
#include "tma_sync.cuh"

namespace vtmu {

__device__ unsigned int g_tc_device_error;

namespace {

constexpr int kBM = 128;      // query rows per CTA = MMA M = TMEM lanes
constexpr int kBN = 64;       // keys per tile = score MMA N
constexpr float kRescaleLog2 = 8.f;  // rescale O when a row max grows by more
constexpr size_t kSmemLimit = 227 * 1024;
#ifndef VTMU_TC_BSTAGE_MAX_D
#define VTMU_TC_BSTAGE_MAX_D 192  // widest headDim that stages bias blocks in shared memory
#endif
#ifndef VTMU_TC_MAX_SLOTS
#define VTMU_TC_MAX_SLOTS 6  // shared-memory ring slots (32 KB each) at most
#endif

enum TcError : unsigned int {
    kErrTcFull = 1u << 8,
    kErrTcEmpty = 1u << 9,
    kErrTcDrain = 1u << 10,
    kErrTcQ = 1u << 11,
    kErrTcS = 1u << 12,
    kErrTcP = 1u << 13,
    kErrTcPv = 1u << 14,
};

template <int D, int DV>
struct TcCfg {
    static constexpr int DVC = DV <= 128 ? DV : DV / 2;       // V columns per CTA (grid.z = DV / DVC)
    static constexpr int KB = D / 32;                          // 32-dim K sub-tiles per key tile
    // Where S and P live.  PMODE 2 (headDim <= 128): 128-column S and P
    // buffers in TMEM, score and P.V MMAs from two threads.  PMODE 1 (headDim
    // 192): S and a 64-column P_hi in TMEM, P_lo in shared memory, one issuing
    // thread.  With either, the next score MMAs may start as soon as the
    // softmax has read S.  PMODE 0 (headDim 256): one 128-column buffer, P
    // written over S, the steps alternate from one thread.  S is stacked:
    // [S_hihi | S_hilo] in 128 columns.
    static constexpr int PMODE = D + DVC + 4 * kBN <= 512 ? 2 : (D + DVC + 3 * kBN <= 512 ? 1 : 0);
    static constexpr bool TWO_ISSUERS = PMODE == 2;
    // Softmax warps.  Four (one per TMEM lane quarter, 64 keys each), or with
    // PMODE 0, where the softmax is not overlapped with the score MMAs, eight:
    // two per lane quarter, 32 keys each, exchanging row maxima per tile.
    // Warp 0 is the TMA thread, warp 1 issues MMAs, warps 2 .. 1 + SMW run the
    // softmax; with 224 threads warp 6 issues the P.V MMAs (PMODE 2).
    static constexpr int SMW = PMODE == 0 ? 8 : 4;
    static constexpr int NCOL = kBN * 4 / SMW;  // keys per softmax thread and tile
    static constexpr int THREADS = PMODE == 0 ? 32 * (2 + SMW) : 224;
    static constexpr bool SPLIT = PMODE != 0;  // S and P apart
    // With P over S the softmax warps fold O into registers every tile: each
    // tile's P.V starts a fresh TMEM accumulator and is added to the running
    // total in f32 round-to-nearest.  The tensor pipe's accumulation rounds
    // toward zero, so a total built in TMEM over thousands of keys shrinks by
    // ~1e-5 relative; per tile the shrink stays ~1e-7 and does not add up.
    static constexpr bool FOLD = PMODE == 0;
    static constexpr int SCOLS = 2 * kBN;
    static constexpr int QLO_FLOATS = kBM * D;                 // Q_lo: KB x [128 x 32]
    static constexpr int PLO_FLOATS = PMODE == 1 ? kBM * kBN : 0;  // P_lo: 2 x [128 x 32]
    // Ring slots of 32 KB (16 KB with PMODE 1, where P_lo takes shared
    // memory).  A K item holds KPI 32-dim sub-tiles, each K_hi (64 rows) then
    // K_lo (64 rows); a V item holds V^T_hi then V^T_lo of VCH 32-key chunks,
    // or, when a chunk's hi + lo exceed a slot (VHALF), one of the two.
    static constexpr int KSUB_FLOATS = 2 * kBN * 32;
    static constexpr int KPI = PMODE == 1 ? 1 : 2;
    static constexpr int SLOT_FLOATS = KPI * KSUB_FLOATS;
    static constexpr int KITEMS = (KB + KPI - 1) / KPI;
    static constexpr int VCHUNK_FLOATS = 2 * DVC * 32;
    static constexpr bool VHALF = VCHUNK_FLOATS > SLOT_FLOATS;
    static constexpr int VCH = VHALF ? 1 : (2 * VCHUNK_FLOATS <= SLOT_FLOATS ? 2 : 1);
    static constexpr int VITEMS = VHALF ? 2 * (kBN / 32) : (kBN / 32) / VCH;
    static constexpr uint32_t SLOT_BYTES = SLOT_FLOATS * sizeof(float);
    // Bias blocks staged by TMA: per softmax warp 32 rows x 64 keys as two
    // 128-byte-swizzled [32 x 32] boxes (headDim <= 192; wider heads leave no
    // room next to Q_lo and three ring slots, and read the bias from global).
    static constexpr bool BSTAGE = D <= VTMU_TC_BSTAGE_MAX_D;
    static constexpr int BWARP_FLOATS = 32 * kBN;
    static constexpr int BIAS_FLOATS = BSTAGE ? 4 * BWARP_FLOATS : 0;
    static constexpr size_t FIXED = (size_t)(QLO_FLOATS + BIAS_FLOATS + PLO_FLOATS) * sizeof(float) + 1024;
    static constexpr int NS_FIT = (int)((kSmemLimit - FIXED) / SLOT_BYTES);
    static constexpr int NS = NS_FIT > VTMU_TC_MAX_SLOTS ? VTMU_TC_MAX_SLOTS : NS_FIT;  // ring slots
    static constexpr int QLO_OFF = 0, BIAS_OFF = QLO_FLOATS, PLO_OFF = QLO_FLOATS + BIAS_FLOATS,
                         RING_OFF = QLO_FLOATS + BIAS_FLOATS + PLO_FLOATS;
    static constexpr size_t SMEM = FIXED + (size_t)NS * SLOT_BYTES;
    // TMEM columns
    static constexpr uint32_t Q_HI = 0, O = D, S = D + DVC, P = SPLIT ? S + SCOLS : S,
                              COLS = PMODE == 2 ? P + 2 * kBN : (PMODE == 1 ? P + kBN : S + SCOLS);
    static_assert(D % 32 == 0 && DVC % 32 == 0 && D <= 256 && DVC <= 128 && DV % DVC == 0, "tcgen05 prefill shape");
    static_assert((VHALF ? VCHUNK_FLOATS / 2 : VCH * VCHUNK_FLOATS) <= SLOT_FLOATS && (DVC * 32 * 4) % 1024 == 0,
                  "V^T chunk layout");
    static_assert(PLO_OFF + PLO_FLOATS == RING_OFF, "shared-memory layout");
    static_assert(COLS <= 512, "TMEM budget");
    static_assert(NS >= 3 && SMEM <= kSmemLimit, "shared memory budget");
    // With two issuing threads each skips the other's ring items, and an
    // mbarrier wait only checks the parity of a slot's phase: a wait for item
    // i is sound only if the slot's previous item, i - NS, has landed.  Each
    // issuer's own earlier items cover that when the score and P.V items of
    // one tile fit in the ring together.
    static_assert(!TWO_ISSUERS || KITEMS + VITEMS <= NS, "two-issuer ring: a tile's items must fit in the ring");
    // Paired softmax warps rely on P over S (the landing of S_j implies P.V_{j-1}
    // is done) and read the bias from global memory.
    static_assert(SMW == 4 || (!SPLIT && !BSTAGE && DVC % 64 == 0 && KB % 2 == 0), "paired softmax warps");
};

// Barrier over the two softmax warps of one TMEM lane quarter (named barrier
// `id`, 64 threads); returns the AND of `v` over them.
__device__ __forceinline__ bool pair_sync_and(uint32_t id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.and.pred p, %2, 64, q;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id)
        : "memory");
    return r != 0;
}

// Pairwise (tree) max: short dependency chains.
template <int N>
__device__ __forceinline__ float tree_max(const float (&v)[N]) {
    float m[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) m[i] = fmaxf(v[i], v[i + N / 2]);
#pragma unroll
    for (int w = N / 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
    return m[0];
}

// Pairwise (tree) sum on packed pairs: pair k holds elements (2k, 2k+1) and
// (2k + N/2, 2k+1 + N/2) first, then halves until one pair is left.
template <int N>
__device__ __forceinline__ float tree_sum(const float (&v)[N]) {
    uint64_t m[N / 4];
#pragma unroll
    for (int k = 0; k < N / 4; ++k)
        m[k] = f2_add(f2_pack(v[2 * k], v[2 * k + 1]), f2_pack(v[2 * k + N / 2], v[2 * k + 1 + N / 2]));
#pragma unroll
    for (int w = N / 8; w >= 1; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k) m[k] = f2_add(m[k], m[k + w]);
    float a, b;
    f2_unpack(m[0], a, b);
    return a + b;
}

// Element (row r, k) of a [rows x 32] f32 tile stored K-major with the
// 128-byte swizzle: rows of 128 B, 16-byte chunk c of row r at chunk c ^ (r % 8).
__device__ __forceinline__ int sw128_offset(int r, int chunk) { return r * 32 + ((chunk ^ (r & 7)) << 2); }

// The fused score epilogue over one key tile of one query row, in base 2:
// scale (or softcap), ALiBi, bias, then the mask -- slots outside
// [lo_i, hi_i] become -inf.  `full` tiles skip the mask.  Features are
// template flags so that each combination compiles to straight-line code.
// BIAS: 0 none; 1 `bias` is this row's bias at the tile's first key (global);
// 2 `bias` is the warp's staged block, row = lane, read as swizzled float4s.
template <int BIAS>
__device__ __forceinline__ float bias_slot(const float* bias, int i, float (&b4)[4]) {
    if constexpr (BIAS == 1) return __ldg(bias + i);
    if ((i & 3) == 0) {
        const float4 t = *reinterpret_cast<const float4*>(bias + (i >> 5) * 1024 +
                                                          sw128_offset(threadIdx.x & 31, (i & 31) >> 2));
        b4[0] = t.x; b4[1] = t.y; b4[2] = t.z; b4[3] = t.w;
    }
    return b4[i & 3];
}

template <bool SOFTCAP, bool ALIBI, int BIAS, int N>
__device__ __forceinline__ void tile_epilogue(const AttnDesc& a, float (&x)[N], float slope, int rel0,
                                              const float* bias, int lo_i, int hi_i, bool full) {
    float b4[4] = {0.f, 0.f, 0.f, 0.f};
    if (SOFTCAP) softcap_tile<N>(x, a.qk_mul, a.cap_log2);
    // ALiBi distance of slot i as (float)rel0 + i: the same value as
    // (float)(rel0 + i) while distances stay below 2^24, without an int ->
    // float conversion per slot.
    const float frel0 = (float)rel0;
    if (full) {
        const uint64_t qk2 = f2_pack(a.qk_mul, a.qk_mul), sl2 = f2_pack(slope, slope),
                       fr2 = f2_pack(frel0, frel0), l2e = f2_pack(kLog2e, kLog2e);
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            uint64_t v = f2_pack(x[i], x[i + 1]);
            if (!SOFTCAP) v = f2_mul(v, qk2);
            if (ALIBI) v = f2_fma(sl2, f2_add(fr2, f2_pack((float)i, (float)(i + 1))), v);
            if (BIAS) {
                const float b0 = bias_slot<BIAS>(bias, i, b4);
                v = f2_fma(f2_pack(b0, bias_slot<BIAS>(bias, i + 1, b4)), l2e, v);
            }
            f2_unpack(v, x[i], x[i + 1]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const bool vis = i >= lo_i && i <= hi_i;
            float v = SOFTCAP ? x[i] : x[i] * a.qk_mul;
            if (ALIBI) v = fmaf(slope, frel0 + (float)i, v);
            if (BIAS == 1) v = fmaf(vis ? __ldg(bias + i) : 0.f, kLog2e, v);
            if (BIAS == 2) v = fmaf(bias_slot<BIAS>(bias, i, b4), kLog2e, v);
            x[i] = vis ? v : -INFINITY;
        }
    }
}

template <int N>
__device__ __forceinline__ void run_epilogue(int feat, const AttnDesc& a, float (&x)[N], float slope, int rel0,
                                             const float* bias, int lo_i, int hi_i, bool full) {
    switch (feat) {
        case 0: tile_epilogue<false, false, 0>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 1: tile_epilogue<true, false, 0>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 2: tile_epilogue<false, true, 0>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 3: tile_epilogue<true, true, 0>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 4: tile_epilogue<false, false, 1>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 5: tile_epilogue<true, false, 1>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 6: tile_epilogue<false, true, 1>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        default: tile_epilogue<true, true, 1>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
    }
}

// The same with the bias read from the warp's staged block.
template <int N>
__device__ __forceinline__ void run_epilogue_staged(int feat, const AttnDesc& a, float (&x)[N], float slope,
                                                    int rel0, const float* block, int lo_i, int hi_i, bool full) {
    switch (feat & 3) {
        case 0: tile_epilogue<false, false, 2>(a, x, slope, rel0, block, lo_i, hi_i, full); break;
        case 1: tile_epilogue<true, false, 2>(a, x, slope, rel0, block, lo_i, hi_i, full); break;
        case 2: tile_epilogue<false, true, 2>(a, x, slope, rel0, block, lo_i, hi_i, full); break;
        default: tile_epilogue<true, true, 2>(a, x, slope, rel0, block, lo_i, hi_i, full); break;
    }
}

// SINKS: attention sinks are on (a separate instantiation, so that the
// common path carries none of their bookkeeping).
template <int D, int DV, bool SINKS>
__global__ void __launch_bounds__(TcCfg<D, DV>::THREADS, 1)
    prefill_tc_kernel(const AttnDesc a, const AlibiTable alibi, const int bias_staged, const int hgroup,
                      const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_bias,
                      const __grid_constant__ CUtensorMap tm_khi,
                      const __grid_constant__ CUtensorMap tm_klo, const __grid_constant__ CUtensorMap tm_vhi,
                      const __grid_constant__ CUtensorMap tm_vlo) {
    using C = TcCfg<D, DV>;
    constexpr int NS = C::NS, KB = C::KB, DVC = C::DVC;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    float* smem = reinterpret_cast<float*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    float* qlo = smem + C::QLO_OFF;
    float* ring = smem + C::RING_OFF;
    __shared__ __align__(8) uint64_t r_full[NS], r_empty[NS], s_full, s_free, p_full, pv_done, q_full,
        q_ready, b_full[4];
    __shared__ uint32_t tmem_base_s;
    // Paired softmax warps: a partial value per key half and row (at headDim
    // 256 static shared memory has room for one such array, 1 KB).
    __shared__ float pair_x[C::SMW == 8 ? 2 * kBM : 1];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_qt = (int)((a.T + kBM - 1) / kBM);
    // CTAs start in linear block order (V half innermost).  When the query
    // tiles' work differs (causal or windowed), the heads come in groups of
    // `hgroup` whose K/V hi/lo fit in L2 together; within a group the query
    // tile is outermost, latest (heaviest) first, so the longest CTAs start
    // first and short ones fill the tail, and the CTAs running together share
    // the group's K/V in L2.  When every tile sees the same keys, heads are
    // outermost so that the CTAs running together share one head's K/V.
    const int nz = (int)gridDim.z;
    const int64_t lin = blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
    const int zz = (int)(lin % nz);
    const bool uniform = !a.causal && a.window <= 0;
    int h, qt;
    if (uniform) {
        h = (int)(lin / ((int64_t)nz * n_qt));
        qt = n_qt - 1 - (int)((lin / nz) % n_qt);
    } else {
        const int64_t r = lin / nz, per_group = (int64_t)n_qt * hgroup;
        const int64_t grp = r / per_group, rem = r % per_group;
        h = (int)(grp * hgroup + rem % hgroup);
        qt = n_qt - 1 - (int)(rem / hgroup);
    }
    const int kh = h / a.G;
    const int dv0 = zz * DVC;  // this CTA's V columns [dv0, dv0 + DVC)
    const int64_t t0 = (int64_t)qt * kBM;
    const int64_t t_last = (t0 + kBM < a.T ? t0 + kBM : a.T) - 1;

    // Key tiles any row of this query tile can see.
    const int64_t p_first = a.pos_offset + t0, p_last = a.pos_offset + t_last;
    int64_t s_lo = 0, s_hi = a.S - 1;
    if (a.causal) {
        if (p_last < s_hi) s_hi = p_last;
        if (a.window > 0) s_lo = p_first - a.window + 1;
    } else if (a.window > 0) {
        s_lo = p_first - a.window;
        if (p_last + a.window < s_hi) s_hi = p_last + a.window;
    }
    if (s_lo < 0) s_lo = 0;
    int64_t jt_begin = s_lo / kBN;
    int64_t jt_end = (s_hi >= s_lo) ? s_hi / kBN + 1 : jt_begin;
    // Attention sinks: keys s < sink_end stay visible (within the causal
    // limit).  Their tiles come after the window's, or join them into one
    // range when the two touch.
    const int64_t sinks = SINKS ? a.sinks : 0;
    const int64_t sink_cap = a.causal ? s_hi + 1 : a.S;
    const int64_t sink_end = sinks < sink_cap ? sinks : sink_cap;
    const int64_t n_st = sink_end > 0 ? (sink_end + kBN - 1) / kBN : 0;
    int n_sink = 0;
    if (n_st > 0 && n_st >= jt_begin) {
        if (n_st > jt_end) jt_end = n_st;
        jt_begin = 0;
    } else {
        n_sink = (int)n_st;
    }
    const int n_win = (int)(jt_end - jt_begin);
    const int n_tiles = n_win + n_sink;
    // Window tiles run from the last (nearest the diagonal) down: with ALiBi
    // the largest scores come first and the running max rarely moves, so O is
    // seldom rescaled.  The producer, the MMA threads and the softmax share it.
    auto tile_key0 = [&](int j) -> int64_t {
        if constexpr (SINKS) return (j < n_win ? jt_begin + (n_win - 1 - j) : (int64_t)(j - n_win)) * kBN;
        return (jt_begin + (n_win - 1 - j)) * kBN;
    };

    if (threadIdx.x == 0) {
        // One barrier per buffer: no wait ever targets a phase two behind.
        for (int b = 0; b < NS; ++b) {
            mbar_init(&r_full[b], 1);
            mbar_init(&r_empty[b], 1);
        }
        // Each completes once per key tile: tile j waits on phase j & 1.
        mbar_init(&s_full, 1);
        mbar_init(&s_free, 4);
        mbar_init(&p_full, C::SMW);
        mbar_init(&pv_done, 1);
        mbar_init(&q_full, 1);
        mbar_init(&q_ready, C::SMW);
        for (int b = 0; b < 4; ++b) mbar_init(&b_full[b], 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base_s, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    // The TMA thread and the MMA threads walk the same sequence of ring
    // items: the score step of tile j takes KITEMS items (K_hi + K_lo of two
    // 32-dim sub-tiles each), the P.V step VITEMS (V^T_hi and V^T_lo of VCH
    // 32-key chunks each).  With two S buffers the steps run S_0, then
    // S_{j+1}, PV_j for every j; with one, S_j, PV_j.
    if (warp == 0) {
        // ------------------------------ TMA producer -----------------------------
        if (lane == 0) {
            // The Q tile lands in the Q_lo area (128-byte swizzled, rows past T
            // read as zero); the softmax warps split it in place.
            mbar_arrive_expect_tx(&q_full, (uint32_t)(kBM * D * sizeof(float)));
            for (int kb = 0; kb < KB; ++kb) tma_load_2d(qlo + kb * kBM * 32, &tm_q, h * D + kb * 32, (int)t0, &q_full);
        }
        if (lane == 0 && n_tiles > 0) {
            prefetch_tensormap(&tm_khi);
            prefetch_tensormap(&tm_klo);
            prefetch_tensormap(&tm_vhi);
            prefetch_tensormap(&tm_vlo);
            int it = 0;
            auto acquire = [&](uint32_t bytes) -> float* {
                const int slot = it % NS;
                if (it >= NS && !mbar_wait(&r_empty[slot], ((it / NS) - 1) & 1)) {
                    raise_device_error(&g_tc_device_error, kErrTcEmpty);
                    return nullptr;
                }
                mbar_arrive_expect_tx(&r_full[slot], bytes);
                return ring + slot * C::SLOT_FLOATS;
            };
            auto load_s = [&](int j) -> bool {
                const int n0 = (int)tile_key0(j);
                for (int ki = 0; ki < C::KITEMS; ++ki) {
                    const int nsub = KB - C::KPI * ki < C::KPI ? KB - C::KPI * ki : C::KPI;
                    float* dst = acquire((uint32_t)nsub * C::KSUB_FLOATS * sizeof(float));
                    if (!dst) return false;
                    for (int u = 0; u < nsub; ++u) {
                        const int x = kh * D + (C::KPI * ki + u) * 32;
                        float* sub = dst + u * C::KSUB_FLOATS;
                        tma_load_2d(sub, &tm_khi, x, n0, &r_full[it % NS]);
                        tma_load_2d(sub + kBN * 32, &tm_klo, x, n0, &r_full[it % NS]);
                    }
                    ++it;
                }
                return true;
            };
            auto load_pv = [&](int j) -> bool {
                const int n0 = (int)tile_key0(j);
                for (int vi = 0; vi < C::VITEMS; ++vi) {
                    if constexpr (C::VHALF) {
                        // item 2c: V^T_hi of chunk c; item 2c + 1: V^T_lo.
                        float* dst = acquire(DVC * 32 * sizeof(float));
                        if (!dst) return false;
                        tma_load_2d(dst, (vi & 1) ? &tm_vlo : &tm_vhi, n0 + (vi >> 1) * 32, kh * DV + dv0,
                                    &r_full[it % NS]);
                    } else {
                        float* dst = acquire(C::VCH * C::VCHUNK_FLOATS * sizeof(float));
                        if (!dst) return false;
                        for (int u = 0; u < C::VCH; ++u) {
                            const int key = n0 + (vi * C::VCH + u) * 32;
                            float* chunk = dst + u * C::VCHUNK_FLOATS;
                            tma_load_2d(chunk, &tm_vhi, key, kh * DV + dv0, &r_full[it % NS]);
                            tma_load_2d(chunk + DVC * 32, &tm_vlo, key, kh * DV + dv0, &r_full[it % NS]);
                        }
                    }
                    ++it;
                }
                return true;
            };
            bool ok = true;
            if constexpr (C::SPLIT) {
                ok = load_s(0);
                for (int j = 0; ok && j < n_tiles; ++j) ok = (j + 1 >= n_tiles || load_s(j + 1)) && load_pv(j);
            } else {
                for (int j = 0; ok && j < n_tiles; ++j) ok = load_s(j) && load_pv(j);
            }
            // Drain: every copy issued has landed before the CTA exits.
            bool drained = true;
            for (int c = it > NS ? it - NS : 0; c < it; ++c) drained &= mbar_wait(&r_full[c % NS], (c / NS) & 1);
            if (!drained) raise_device_error(&g_tc_device_error, kErrTcDrain);
        }
    } else if (warp == 1 || (C::SMW == 4 && warp == 6)) {
        // ---------- MMA issuers: warp 1 the scores, warp 6 P.V (PMODE 2); warp 1 both (PMODE 1) ----------
        // One kind::tf32 MMA issues at most every ~53 cycles from one thread, so
        // with PMODE 2 the score and P.V streams come from two threads (two
        // warps) and meet in the tensor pipe.  Both index the ring sequence of
        // the TMA thread: item numbers follow from the step order S_0, then
        // S_{j+1}, PV_j for every j.  With PMODE 1 one thread issues both in
        // that order and consumes the ring in order.
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t id_s2 = idesc_tf32(kBM, 2 * kBN), id_s = idesc_tf32(kBM, kBN),
                               id_o = idesc_tf32(kBM, DVC);
            constexpr int KI = C::KITEMS, VI = C::VITEMS;
            auto s_first = [&](int j) -> int {
                return C::SPLIT ? (j == 0 ? 0 : KI + (j - 1) * (KI + VI)) : j * (KI + VI);
            };
            auto pv_first = [&](int j) -> int {
                return C::SPLIT ? KI + j * (KI + VI) + (j + 1 < n_tiles ? KI : 0) : j * (KI + VI) + KI;
            };
            auto take = [&](int item) -> bool {
                if (!mbar_wait(&r_full[item % NS], (uint32_t)(item / NS) & 1u)) {
                    raise_device_error(&g_tc_device_error, kErrTcFull);
                    return false;
                }
                tc_fence_after();
                return true;
            };
            // Descriptors are base + byte offset / 16, computed once.
            const uint64_t ring_d = smem_desc_sw128(ring), qlo_d = smem_desc_sw128(qlo);
            const uint64_t plo_d = smem_desc_sw128(smem + C::PLO_OFF);
            constexpr uint64_t SLOT_D = C::SLOT_FLOATS * 4 / 16, KSUB_D = C::KSUB_FLOATS * 4 / 16,
                               QSUB_D = kBM * 32 * 4 / 16,
                               VCH_D = C::VCHUNK_FLOATS * 4 / 16, VLO_D = DVC * 32 * 4 / 16, KSTEP_D = 32 / 16,
                               PLO_CHUNK_D = kBM * 32 * 4 / 16;
            // S: [Q_hi K_hi^T | Q_hi K_lo^T + Q_lo K_hi^T]: the two small
            // correction products share the second half, so the large first
            // half takes one product per k-step (the tensor pipe truncates each
            // accumulation, with an error relative to the accumulator).
            auto issue_s = [&](int j) -> bool {
                const uint32_t d = tmem + C::S;
                const int it0 = s_first(j);
#pragma unroll
                for (int ki = 0; ki < KI; ++ki) {
                    const int item = it0 + ki;
                    if (!take(item)) return false;
                    const uint64_t b_slot = ring_d + (uint64_t)(item % NS) * SLOT_D;
#pragma unroll
                    for (int u = 0; u < C::KPI; ++u) {
                        const int kb = C::KPI * ki + u;
                        if (kb < KB) {
                            const uint64_t b_k = b_slot + u * KSUB_D;  // [K_hi; K_lo]
                            const uint64_t a_lo = qlo_d + kb * QSUB_D;
                            const uint32_t a_hi = tmem + C::Q_HI + kb * 32;
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint64_t bk = b_k + k * KSTEP_D;
                                if (kb == 0 && k == 0)
                                    mma_tf32_ts(d, a_hi, bk, id_s2, 0u);
                                else
                                    mma_tf32_ts_acc(d, a_hi + k * 8, bk, id_s2);
                                mma_tf32_ss_acc(d + kBN, a_lo + k * KSTEP_D, bk, id_s);
                            }
                        }
                    }
                    mma_commit(&r_empty[item % NS]);
                }
                mma_commit(&s_full);
                return true;
            };
            // O += P_hi V_hi + P_hi V_lo + P_lo V_hi for one 32-key chunk c of
            // tile j; P_lo from TMEM (PMODE 2) or shared memory (PMODE 1).
            auto pv_chunk = [&](int j, int c, uint64_t v_hi, uint64_t v_lo) {
                const uint32_t o = tmem + C::O;
                const uint32_t p_hi = tmem + C::P, p_lo = p_hi + kBN;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t col = c * 32 + k * 8;
                    if (c == 0 && k == 0)
                        mma_tf32_ts(o, p_hi + col, v_hi + k * KSTEP_D, id_o, (C::FOLD || j == 0) ? 0u : 1u);
                    else
                        mma_tf32_ts_acc(o, p_hi + col, v_hi + k * KSTEP_D, id_o);
                    mma_tf32_ts_acc(o, p_hi + col, v_lo + k * KSTEP_D, id_o);
                    if constexpr (C::PMODE == 1)
                        mma_tf32_ss_acc(o, plo_d + c * PLO_CHUNK_D + k * KSTEP_D, v_hi + k * KSTEP_D, id_o);
                    else
                        mma_tf32_ts_acc(o, p_lo + col, v_hi + k * KSTEP_D, id_o);
                }
            };
            auto issue_pv = [&](int j) -> bool {
                if (!mbar_wait(&p_full, (uint32_t)j & 1u)) {
                    raise_device_error(&g_tc_device_error, kErrTcP);
                    return false;
                }
                const int it0 = pv_first(j);
                if constexpr (C::VHALF) {
#pragma unroll
                    for (int c = 0; c < kBN / 32; ++c) {
                        const int ih = it0 + 2 * c, il = ih + 1;  // V^T_hi item, V^T_lo item
                        if (!take(ih) || !take(il)) return false;
                        pv_chunk(j, c, ring_d + (uint64_t)(ih % NS) * SLOT_D, ring_d + (uint64_t)(il % NS) * SLOT_D);
                        mma_commit(&r_empty[ih % NS]);
                        mma_commit(&r_empty[il % NS]);
                    }
                } else {
#pragma unroll
                    for (int vi = 0; vi < VI; ++vi) {
                        const int item = it0 + vi;
                        if (!take(item)) return false;
                        const uint64_t v_slot = ring_d + (uint64_t)(item % NS) * SLOT_D;
#pragma unroll
                        for (int u = 0; u < C::VCH; ++u) {
                            const uint64_t v_hi = v_slot + u * VCH_D;
                            pv_chunk(j, vi * C::VCH + u, v_hi, v_hi + VLO_D);
                        }
                        mma_commit(&r_empty[item % NS]);
                    }
                }
                mma_commit(&pv_done);
                return true;
            };
            // S_j overwrites S_{j-1} once the softmax has read it.
            auto wait_s_free = [&](int j) -> bool {
                if (j >= 1) {
                    if (!mbar_wait(&s_free, (uint32_t)(j - 1) & 1u)) {
                        raise_device_error(&g_tc_device_error, kErrTcS);
                        return false;
                    }
                    tc_fence_after();
                }
                return true;
            };
            if (warp == 1) {
                bool ok = mbar_wait(&q_ready, 0);
                if (!ok) raise_device_error(&g_tc_device_error, kErrTcQ);
                tc_fence_after();
                if constexpr (C::TWO_ISSUERS) {
                    for (int j = 0; ok && j < n_tiles; ++j) ok = wait_s_free(j) && issue_s(j);
                } else if constexpr (C::SPLIT) {
                    ok = ok && issue_s(0);
                    for (int j = 0; ok && j < n_tiles; ++j)
                        ok = (j + 1 >= n_tiles || (wait_s_free(j + 1) && issue_s(j + 1))) && issue_pv(j);
                } else {
                    // P over S: in issue order P.V_j reads P_j before S_{j+1} lands.
                    for (int j = 0; ok && j < n_tiles; ++j) ok = issue_s(j) && issue_pv(j);
                }
            } else if (C::TWO_ISSUERS) {
                bool ok = true;
                for (int j = 0; ok && j < n_tiles; ++j) ok = issue_pv(j);
            }
        }
    } else {
        // --------------------- softmax warps: thread = query row ---------------------
        constexpr bool PAIR = C::SMW == 8;
        constexpr int NCOL = C::NCOL;
        const uint32_t lrow = 32u * (uint32_t)(warp & 3);  // TMEM lane quarter of this warp
        const int r = (int)lrow + lane;
        // Paired warps: half 0 (warps 2-5) takes keys [0, 32) of each tile, the
        // first half of the Q sub-tiles and of O; half 1 (warps 6-9) the rest.
        const int half = PAIR ? (warp - 2) >> 2 : 0;
        const int c0 = half * NCOL;                      // this warp's first key of a tile
        const int oc0 = half * (DVC / (PAIR ? 2 : 1));   // and its first O column
        constexpr int OCOLS = DVC / (PAIR ? 2 : 1);
        const uint32_t pair_id = 1u + (uint32_t)(warp & 3);
        const int64_t t = t0 + r;
        const bool row_ok = t < a.T;
        const uint32_t trow = tmem + (lrow << 16);
        const float slope = a.alibi_on ? alibi.slope_log2[h] : 0.f;
        // Q row (staged by TMA) -> hi (TMEM) / lo (in place, shared memory).
        {
            if (!__all_sync(FULL, mbar_wait(&q_full, 0))) raise_device_error(&g_tc_device_error, kErrTcQ);
#pragma unroll 1
            for (int kb = half * (KB / (PAIR ? 2 : 1)); kb < (half + 1) * (KB / (PAIR ? 2 : 1)); ++kb) {
                float* sub = qlo + kb * kBM * 32;
                float hi[32], lo[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float4 v4 = *reinterpret_cast<const float4*>(sub + sw128_offset(r, c));
                    const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        hi[4 * c + e] = tf32_trunc(vv[e]);
                        lo[4 * c + e] = vv[e] - hi[4 * c + e];
                    }
                }
                tmem_st32(trow + C::Q_HI + kb * 32, hi);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<float4*>(sub + sw128_offset(r, c)) =
                        make_float4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
            }
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // Q_lo -> MMA (async proxy)
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_ready);
        }
        // Keys this row can see: one contiguous range [lo_t, hi_t] (empty for
        // padding rows past T).
        const int64_t p = a.pos_offset + t;
        int64_t lo_t = 0, hi_t = a.S - 1;
        if (a.causal) {
            if (p < hi_t) hi_t = p;
            if (a.window > 0) lo_t = p - a.window + 1;
        } else if (a.window > 0) {
            lo_t = p - a.window;
            if (p + a.window < hi_t) hi_t = p + a.window;
        }
        if (!row_ok) {
            lo_t = 1;
            hi_t = 0;
        }
        // Attention sinks: keys below sink_t are visible too (0 when none;
        // key indices fit 31 bits, as the TMA coordinates do).
        const bool has_sinks = SINKS && a.sinks > 0;  // the same for every thread
        int sink_t = 0;
        if (has_sinks && row_ok) {
            const int64_t cap = a.causal ? hi_t + 1 : a.S;
            sink_t = (int)(a.sinks < cap ? a.sinks : cap);
        }
        const float* brow = a.bias_kind == 0 ? nullptr
                            : a.bias_kind == 1 ? a.bias + t * a.S
                                               : a.bias + ((int64_t)h * a.T + t) * a.S;
        // Staged bias: lane 0 of each softmax warp loads the warp's 32 rows x 64
        // keys of tile j + 1 as soon as the epilogue of tile j has read tile j's.
        const bool bstage = C::BSTAGE && bias_staged && a.bias_kind != 0;
        const int wq = warp & 3;
        float* bbuf = smem + C::BIAS_OFF + wq * C::BWARP_FLOATS;
        const int brow0 = (int)((a.bias_kind == 2 ? (int64_t)h * a.T : 0) + t0) + 32 * wq;
        int b_issued = 0;  // bias blocks requested (tiles 0 .. b_issued - 1)
        auto issue_bias = [&](int j) {
            if (lane == 0) {
                const int n0 = (int)tile_key0(j);
                mbar_arrive_expect_tx(&b_full[wq], (uint32_t)(C::BWARP_FLOATS * sizeof(float)));
                tma_load_2d(bbuf, &tm_bias, n0, brow0, &b_full[wq]);
                tma_load_2d(bbuf + 32 * 32, &tm_bias, n0 + 32, brow0, &b_full[wq]);
            }
            ++b_issued;
        };
        if (bstage && n_tiles > 0) issue_bias(0);
        const int feat = (a.softcap_on ? 1 : 0) | (a.alibi_on ? 2 : 0) | (a.bias_kind ? 4 : 0);
        float m_ref = -INFINITY, l = 0.f;
        // FOLD: this thread's O columns, summed over the tiles folded so far
        // (in units of the current reference max).
        float otot[C::FOLD ? OCOLS : 1];
#pragma unroll
        for (int i = 0; i < (C::FOLD ? OCOLS : 1); ++i) otot[i] = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            bool got = __all_sync(FULL, mbar_wait(&s_full, j & 1));
            if (!got) raise_device_error(&g_tc_device_error, kErrTcS);
            if constexpr (PAIR) {
                // P over S: S_j has landed, so P.V_{j-1} is done and this wait
                // returns at once.  Both warps of the pair leave the loop
                // together, at the barrier below.
                if (got && j >= 1) {
                    got = __all_sync(FULL, mbar_wait(&pv_done, (j - 1) & 1));
                    if (!got) raise_device_error(&g_tc_device_error, kErrTcPv);
                }
            } else if (!got) {
                ok = false;
                break;
            }
            if (bstage && !__all_sync(FULL, mbar_wait(&b_full[wq], j & 1))) {
                raise_device_error(&g_tc_device_error, kErrTcFull);
                ok = false;
                break;
            }
            tc_fence_after();
            float x[NCOL];
#pragma unroll
            for (int h2 = 0; h2 < NCOL; h2 += 32) {  // S = first half + second half
                float y[32];
                tmem_ld32(trow + C::S + c0 + h2, x + h2);
                tmem_ld32(trow + C::S + kBN + c0 + h2, y);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 2)
                    f2_unpack(f2_add(f2_pack(x[h2 + i], x[h2 + i + 1]), f2_pack(y[i], y[i + 1])), x[h2 + i],
                              x[h2 + i + 1]);
            }
            if constexpr (C::SPLIT) {
                // The scores are in registers: the next score MMAs may overwrite S.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_free);
            }
            const int64_t n0 = tile_key0(j) + c0;
            // Visible slots of this warp's keys, clamped to [-1, NCOL].
            const int64_t lo64 = lo_t - n0, hi64 = hi_t - n0;
            int lo_i = (int)(lo64 < -1 ? -1 : (lo64 > NCOL ? NCOL : lo64));
            int hi_i = (int)(hi64 < -1 ? -1 : (hi64 > NCOL ? NCOL : hi64));
            // Attention sinks in this tile (rare): slots below sk_i are visible
            // too.  The epilogue then covers [0, max(hi_i, sk_i - 1)] and the
            // gap [sk_i, lo_i) between the sinks and the window is masked after
            // it (its keys lie inside the key range, so the bias reads stay in
            // bounds).
            int gap_lo = NCOL, gap_hi = NCOL;
            if (has_sinks) {
                const int sk_r = sink_t - (int)n0;
                const int sk_i = sk_r < 0 ? 0 : (sk_r > NCOL ? NCOL : sk_r);
                if (sk_i > 0) {
                    if (sk_i < lo_i) {
                        gap_lo = sk_i;
                        gap_hi = lo_i < NCOL ? lo_i : NCOL;
                    }
                    lo_i = 0;
                    if (hi_i < sk_i - 1) hi_i = sk_i - 1;
                }
            }
            const bool full = lo_i <= 0 && hi_i >= NCOL - 1 && gap_lo >= gap_hi;
            // Plain scaled scores (no softcap, ALiBi or bias) with a positive
            // scale: the mask alone here, and the scale goes into the exp2's FFMA.
            const bool fold = feat == 0 && a.qk_mul > 0.f;
            if (!fold) {
                if (!bstage) {
                    run_epilogue<NCOL>(feat, a, x, slope, (int)(n0 - p), brow ? brow + n0 : nullptr, lo_i, hi_i,
                                       full);
                } else {
                    run_epilogue_staged<NCOL>(feat, a, x, slope, (int)(n0 - p), bbuf, lo_i, hi_i, full);
                }
                if (bstage && j + 1 < n_tiles) {
                    // The block has been read (generic proxy) before TMA refills it.
                    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
                    __syncwarp();
                    issue_bias(j + 1);
                }
            } else if (!full) {
#pragma unroll
                for (int i = 0; i < NCOL; ++i) x[i] = (i >= lo_i && i <= hi_i) ? x[i] : -INFINITY;
            }
            if (has_sinks && gap_lo < gap_hi) {  // sinks and window apart in this tile: hide the keys between
#pragma unroll
                for (int i = 0; i < NCOL; ++i)
                    if (i >= gap_lo && i < gap_hi) x[i] = -INFINITY;
            }
            const float cx = fold ? a.qk_mul : 1.f;
            float mt = tree_max<NCOL>(x) * cx;
            if constexpr (PAIR) {
                // The partner reads this slot after the barrier and before its
                // p_full arrival (its P depends on the value), and tile j + 1's
                // write waits for S_{j+1}, which waits for that arrival: one
                // array serves every tile.
                pair_x[half * kBM + r] = mt;
                if (!pair_sync_and(pair_id, got)) {
                    ok = false;
                    break;
                }
                mt = fmaxf(mt, pair_x[(half ^ 1) * kBM + r]);
            }
            // Lazy rescale: keep the reference max unless this tile beats it by > 2^8.
            float alpha = 1.f;
            if (mt > m_ref + kRescaleLog2) {
                alpha = fast_exp2(m_ref - mt);  // 0 on the first visible tile
                m_ref = mt;
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
#pragma unroll
            for (int i = 0; i < NCOL; i += 2) {
                float e0, e1;
                f2_unpack(f2_fma(f2_pack(x[i], x[i + 1]), f2_pack(cx, cx), f2_pack(-m_use, -m_use)), e0, e1);
                x[i] = fast_exp2(e0);
                x[i + 1] = fast_exp2(e1);
            }
            l = fmaf(l, alpha, tree_sum<NCOL>(x));
            float plo[NCOL];
            const uint64_t m1 = f2_pack(-1.f, -1.f);
#pragma unroll
            for (int i = 0; i < NCOL; i += 2) {  // P_hi replaces P in registers; P_lo = P - P_hi (exact)
                const float h0 = tf32_trunc(x[i]), h1 = tf32_trunc(x[i + 1]);
                f2_unpack(f2_fma(f2_pack(h0, h1), m1, f2_pack(x[i], x[i + 1])), plo[i], plo[i + 1]);
                x[i] = h0;
                x[i + 1] = h1;
            }
            // P_{j-1} has been read and O holds P.V_{j-1} (with P over S the
            // landing of S_j already implies it, and the wait costs nothing).
            if (!PAIR && j >= 1 && !__all_sync(FULL, mbar_wait(&pv_done, (j - 1) & 1))) {
                raise_device_error(&g_tc_device_error, kErrTcPv);
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < NCOL; c += 32) tmem_st32(trow + C::P + c0 + c, x + c);
            if constexpr (C::PMODE == 1) {
                // P_lo row r -> shared memory, K-major 128-byte-swizzled [128 x 32]
                // chunks (the A operand of the SS-form product).
                float* pl = smem + C::PLO_OFF;
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<float4*>(pl + c * kBM * 32 + sw128_offset(r, q)) =
                            make_float4(plo[32 * c + 4 * q], plo[32 * c + 4 * q + 1], plo[32 * c + 4 * q + 2],
                                        plo[32 * c + 4 * q + 3]);
                asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");  // P_lo -> MMA (async proxy)
            } else {
#pragma unroll
                for (int c = 0; c < NCOL; c += 32) tmem_st32(trow + C::P + kBN + c0 + c, plo + c);
            }
            if constexpr (C::FOLD) {
                // O holds P.V_{j-1} alone (S_j has landed, so it is done, and
                // P.V_j overwrites it only after this warp's p_full arrival):
                // add it to the total, then bring the total to this tile's max.
                if (j >= 1) {
#pragma unroll
                    for (int c = 0; c < OCOLS; c += 32) {
                        float o[32];
                        tmem_ld32(trow + C::O + oc0 + c, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) otot[c + i] = (otot[c + i] + o[i]) * alpha;
                    }
                }
            }
            if (!C::FOLD && j > 0 && __any_sync(FULL, alpha != 1.f)) {
#pragma unroll 1
                for (int c = oc0; c < oc0 + OCOLS; c += 32) {
                    float o[32];
                    tmem_ld32(trow + C::O + c, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tmem_st32(trow + C::O + c, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full);
        }
        // No bias block may still be in flight when the CTA exits (a loop
        // that stopped early can leave one).
        if (bstage && b_issued > 0 && !__all_sync(FULL, mbar_wait(&b_full[wq], (b_issued - 1) & 1)))
            raise_device_error(&g_tc_device_error, kErrTcDrain);
        // Epilogue: O / l -> out.
        if (ok && n_tiles > 0) {
            const int last = n_tiles - 1;
            if (!__all_sync(FULL, mbar_wait(&pv_done, last & 1))) {
                raise_device_error(&g_tc_device_error, kErrTcPv);
                ok = false;
            }
        }
        if constexpr (PAIR) {
            // Row sum over both key halves (each warp of the pair reaches this
            // barrier once: both left the loop together).
            ok = pair_sync_and(pair_id, ok);  // both have read the last maxima
            pair_x[half * kBM + r] = l;
            pair_sync_and(pair_id, true);
            l += pair_x[(half ^ 1) * kBM + r];
        }
        tc_fence_after();
        const float inv = (ok && l > 0.f) ? 1.f / l : 0.f;
        float* orow = a.out + t * (int64_t)a.H * DV + (int64_t)h * DV + dv0;
        // Row r's output: O / l (with FOLD: the folded total plus the last
        // tile's P.V, in an unrolled loop so that the total stays in registers).
        auto store_row = [&](int c, float (&o)[32]) {
            if (row_ok) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4*>(orow + c + i) =
                        make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
            }
        };
        auto load_o = [&](int c, float (&o)[32]) {
            if (n_tiles > 0) {
                tmem_ld32(trow + C::O + c, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = 0.f;
            }
        };
        if constexpr (C::FOLD) {
#pragma unroll
            for (int cc = 0; cc < OCOLS; cc += 32) {
                float o[32];
                load_o(oc0 + cc, o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] += otot[cc + i];
                store_row(oc0 + cc, o);
            }
        } else {
#pragma unroll 1
            for (int c = oc0; c < oc0 + OCOLS; c += 32) {
                float o[32];
                load_o(c, o);
                store_row(c, o);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---- pre-pass: tf32 hi/lo split of K, and of V transposed -------------------------
// Elementwise and HBM-bound: 16-byte accesses when K is 16-byte aligned
// (the workspace halves always are), so that each thread keeps 16 bytes in
// flight per load instead of 4.
__global__ void split_k_kernel(const float* __restrict__ k, float* __restrict__ khi, float* __restrict__ klo,
                               int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if ((reinterpret_cast<uintptr_t>(k) & 15u) == 0 && (n & 3) == 0) {
        const float4* k4 = reinterpret_cast<const float4*>(k);
        float4* hi4 = reinterpret_cast<float4*>(khi);
        float4* lo4 = reinterpret_cast<float4*>(klo);
        for (int64_t i = i0; i < n / 4; i += stride) {
            const float4 x = __ldg(k4 + i);
            const float4 h = make_float4(tf32_rna(x.x), tf32_rna(x.y), tf32_rna(x.z), tf32_rna(x.w));
            hi4[i] = h;
            lo4[i] = make_float4(tf32_rna(x.x - h.x), tf32_rna(x.y - h.y), tf32_rna(x.z - h.z), tf32_rna(x.w - h.w));
        }
        return;
    }
    for (int64_t i = i0; i < n; i += stride) {
        const float x = __ldg(k + i);
        const float hi = tf32_rna(x);
        khi[i] = hi;
        klo[i] = tf32_rna(x - hi);
    }
}

// v [S, cols] -> vt_hi / vt_lo [cols, s_pad]; columns s >= S are zero.
// Blocks of 32 x 8 threads; the four loads (and stores) of a thread are
// independent, so they are all in flight at once.
constexpr int kSplitVtRows = 8;
__global__ void split_vt_kernel(const float* __restrict__ v, float* __restrict__ vthi, float* __restrict__ vtlo,
                                int64_t S, int64_t s_pad, int cols) {
    __shared__ float tile[32][33];
    const int64_t s0 = (int64_t)blockIdx.x * 32;
    const int c0 = blockIdx.y * 32;
#pragma unroll
    for (int rr = 0; rr < 32 / kSplitVtRows; ++rr) {
        const int r = threadIdx.y + rr * kSplitVtRows;
        const int64_t s = s0 + r;
        const int c = c0 + threadIdx.x;
        tile[r][threadIdx.x] = (s < S && c < cols) ? __ldg(v + s * cols + c) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < 32 / kSplitVtRows; ++rr) {
        const int r = threadIdx.y + rr * kSplitVtRows;
        const int c = c0 + r;
        const int64_t s = s0 + threadIdx.x;
        if (c < cols && s < s_pad) {
            const float x = tile[threadIdx.x][r];
            const float hi = tf32_rna(x);
            vthi[(int64_t)c * s_pad + s] = hi;
            vtlo[(int64_t)c * s_pad + s] = tf32_rna(x - hi);
        }
    }
}

// ---- host side ----------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// [rows, cols] f32 row-major, 128-byte swizzled boxes of 32 columns x box_rows.
bool encode_sw128(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, int box_rows) {
    return cached_tensor_map(map, base, rows, cols, 32, box_rows, 128, [&](CUtensorMap* m) {
        auto fn = encoder();
        if (!fn) return false;
        const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)cols * sizeof(float)};
        const cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
        const cuuint32_t estr[2] = {1, 1};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    });
}

size_t up256(size_t b) { return (b + 255) / 256 * 256; }

struct TcLayout {
    int64_t s_pad;
    size_t k_bytes, vt_bytes, total;
};

TcLayout tc_layout(const AttnDesc& a) {
    TcLayout L;
    L.s_pad = (a.S + 3) / 4 * 4;
    L.k_bytes = up256((size_t)a.S * a.Hk * a.D * sizeof(float));
    L.vt_bytes = up256((size_t)a.Hk * a.Dv * L.s_pad * sizeof(float));
    L.total = kWorkspaceHeader + 2 * L.k_bytes + 2 * L.vt_bytes;
    return L;
}

template <int D, int DV, bool SINKS>
cudaError_t launch_cfg(const AttnDesc& a, const AlibiTable& alibi, float* khi, float* klo, float* vthi,
                       float* vtlo, int64_t s_pad, cudaStream_t stream) {
    using C = TcCfg<D, DV>;
    CUtensorMap m_q, m_bias, m_khi, m_klo, m_vhi, m_vlo;
    // The bias goes through TMA when a row of it starts on a 16-byte boundary.
    std::memset(&m_bias, 0, sizeof(m_bias));
    int bias_staged = 0;
    if (C::BSTAGE && a.bias_kind != 0 && (reinterpret_cast<uintptr_t>(a.bias) & 15u) == 0 && a.S % 4 == 0) {
        const int64_t rows = a.bias_kind == 2 ? (int64_t)a.H * a.T : a.T;
        if (!encode_sw128(&m_bias, a.bias, rows, a.S, 32)) return cudaErrorInvalidValue;
        bias_staged = 1;
    }
    if (!encode_sw128(&m_q, a.q, a.T, (int64_t)a.H * D, kBM) ||
        !encode_sw128(&m_khi, khi, a.S, (int64_t)a.Hk * D, kBN) ||
        !encode_sw128(&m_klo, klo, a.S, (int64_t)a.Hk * D, kBN) ||
        !encode_sw128(&m_vhi, vthi, (int64_t)a.Hk * DV, s_pad, C::DVC) ||
        !encode_sw128(&m_vlo, vtlo, (int64_t)a.Hk * DV, s_pad, C::DVC))
        return cudaErrorInvalidValue;
    auto kern = prefill_tc_kernel<D, DV, SINKS>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), (int)C::SMEM);
    if (e != cudaSuccess) return e;
    // Query heads per launch-order group: whole KV groups (a divisor of
    // kvHeads) whose K and V^T hi/lo over the keys of a few concurrent query
    // tiles stay under ~40 MB of the 126 MB L2 (80 MB let the headDim-256
    // windowed prefill read its K/V from DRAM ~1.8 times; 20 MB slowed the
    // ALiBi prefill by splitting its heads too finely).
    const int64_t keys = a.window > 0 ? (a.window + 5 * kBM < a.S ? a.window + 5 * kBM : a.S) : a.S;
    const double per_kv = (double)keys * (D + DV) * 2 * sizeof(float);
    int gk = a.Hk;
    while (gk > 1 && (a.Hk % gk != 0 || per_kv * gk > 40e6)) --gk;
    const int hgroup = gk * a.G;
    dim3 grid((unsigned)((a.T + kBM - 1) / kBM), (unsigned)a.H, (unsigned)(DV / C::DVC));
    kern<<<grid, C::THREADS, C::SMEM, stream>>>(a, alibi, bias_staged, hgroup, m_q, m_bias, m_khi, m_klo, m_vhi,
                                                m_vlo);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const AttnDesc& a) {
    const bool dims = ((a.D == 32 || a.D == 64 || a.D == 96 || a.D == 128 || a.D == 256) && a.Dv == a.D) ||
                      (a.D == 192 && a.Dv == 128);
    const bool out_aligned = (reinterpret_cast<uintptr_t>(a.out) & 15u) == 0;
    const bool q_aligned = (reinterpret_cast<uintptr_t>(a.q) & 15u) == 0;
    return dims && a.T >= 1 && a.S >= 1 && a.S < ((int64_t)1 << 31) && a.pos_offset + a.T < ((int64_t)1 << 31) &&
           (a.T + kBM - 1) / kBM < (1 << 30) &&
           (a.out == nullptr || out_aligned) && (a.q == nullptr || q_aligned);
}

size_t prefill_tc_workspace(const AttnDesc& a) { return tc_layout(a).total; }

cudaError_t launch_prefill_tc(const AttnDesc& a, const AlibiTable& alibi, void* workspace, cudaStream_t stream) {
    const TcLayout L = tc_layout(a);
    char* w = static_cast<char*>(workspace) + kWorkspaceHeader;  // the header is the decode kernel's
    float* khi = reinterpret_cast<float*>(w);
    float* klo = reinterpret_cast<float*>(w + L.k_bytes);
    float* vthi = reinterpret_cast<float*>(w + 2 * L.k_bytes);
    float* vtlo = reinterpret_cast<float*>(w + 2 * L.k_bytes + L.vt_bytes);
    const int64_t nk = a.S * a.Hk * a.D;
    int64_t blocks = (nk + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    split_k_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a.k, khi, klo, nk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int cols = a.Hk * a.Dv;
    dim3 g2((unsigned)((L.s_pad + 31) / 32), (unsigned)((cols + 31) / 32));
    split_vt_kernel<<<g2, dim3(32, kSplitVtRows), 0, stream>>>(a.v, vthi, vtlo, a.S, L.s_pad, cols);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
#define VTMU_TC(D_, DV_)                                                                                     \
    if (a.D == D_ && a.Dv == DV_)                                                                            \
        return a.sinks > 0 ? launch_cfg<D_, DV_, true>(a, alibi, khi, klo, vthi, vtlo, L.s_pad, stream)      \
                           : launch_cfg<D_, DV_, false>(a, alibi, khi, klo, vthi, vtlo, L.s_pad, stream);
    VTMU_TC(32, 32) VTMU_TC(64, 64) VTMU_TC(96, 96) VTMU_TC(128, 128) VTMU_TC(192, 128) VTMU_TC(256, 256)
#undef VTMU_TC
    return cudaErrorInvalidValue;
}

unsigned int tc_take_device_error() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_device_error, sizeof(v)) != cudaSuccess) return 0;
    if (v) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_tc_device_error, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace vtmu
