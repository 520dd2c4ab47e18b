// prefill_tc.cu -- attention prefill on the tcgen05 tensor cores in 3xTF32.
//
// Op "attention" (vtmu.mpakt.dev/api/ops), f32 in and out.  Both
// contractions run on kind::tf32 UMMAs with error compensation: every f32
// operand x is split into hi = x with the low 13 mantissa bits cleared
// (exactly a tf32 value) and lo = x - hi (exact in f32), and each product
// A.B is issued as A_hi.B_hi + A_hi.B_lo + A_lo.B_hi into one f32
// accumulator.  The dropped A_lo.B_lo term and the tf32 rounding of lo are
// both of order 2^-21 relative, so the result matches an f32 FMA kernel.
// Single-pass TF32 is never used.
//
// Work split:
//  * a pre-pass (split_k_kernel, split_vt_kernel) writes K_hi / K_lo in K's
//    own layout and V^T_hi / V^T_lo transposed to [kvHeads*vHeadDim, S],
//    so every tile the MMAs read is K-major;
//  * one CTA owns 128 query rows of one head (the MMA M); per key tile of
//    BN = 64 keys:
//      S_j  = Q K_j^T          (TMEM accumulator, M=128 x N=64)
//      P_j  = softmax part     (4 warps; thread = query row = TMEM lane)
//      O   += P_j V_j          (TMEM accumulator, M=128 x N=vHeadDim)
//    A kind::tf32 MMA takes at least ~46 cycles to issue whatever its N, so
//    the score MMAs use N = 64 (70 % of the tensor rate; N = 32 reaches 35 %);
//  * warp 0 issues TMA loads: a 2-deep ring of K hi/lo tiles and one V^T
//    hi/lo tile (V_j is needed only after the softmax of tile j, so one
//    buffer, refilled as soon as P.V_j completes, keeps it ahead);
//    warp 1 owns TMEM and one of its threads issues every MMA; warps 2-5
//    load Q (split into TMEM), run the fused epilogue and online softmax
//    (base 2, rescaling O only when a row max grows by more than 2^8),
//    write P hi/lo into TMEM and finally normalise and store O;
//  * Q hi/lo and P hi/lo live in TMEM (the MMA's A operand), K and V^T in
//    shared memory (B operand, 128-byte swizzled).  TMEM columns:
//    Q_hi | Q_lo | O | S (= P_hi) | P_lo = 2D + Dv + 2*64 <= 512.
//    P_hi of tile j overwrites S_j once the scores are in registers; the
//    MMAs of one thread execute in issue order, so S_{j+1} (issued after
//    P.V_j) overwrites it only after P.V_j has read it.
//
// Every wait is bounded (tma_sync.cuh); a wait that gives up sets a bit of
// g_tc_device_error and the kernel unwinds.
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn_common.cuh"
#include "kernels.h"
#include "tcgen05_ops.cuh"
#include "tma_sync.cuh"

namespace vtmu {

__device__ unsigned int g_tc_device_error;

namespace {

constexpr int kBM = 128;      // query rows per CTA = MMA M = TMEM lanes
constexpr int kBN = 64;       // keys per tile = score MMA N
constexpr int kThreads = 192; // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr float kRescaleLog2 = 8.f;  // rescale O when a row max grows by more

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
    static constexpr int KB = D / 32;                    // 32-float K sub-tiles
    static constexpr int K_FLOATS = kBN * D;             // one K tile (hi or lo): KB x [64 x 32]
    static constexpr int V_FLOATS = DV * kBN;            // one V^T tile (hi or lo): 2 x [DV x 32]
    static constexpr int KSTAGE_FLOATS = 2 * K_FLOATS;   // K hi + lo
    static constexpr uint32_t KSTAGE_BYTES = KSTAGE_FLOATS * sizeof(float);
    static constexpr uint32_t V_BYTES = 2 * V_FLOATS * sizeof(float);
    static constexpr int V_OFF = 2 * KSTAGE_FLOATS;      // after the two K stages
    static constexpr size_t SMEM = (size_t)(2 * KSTAGE_FLOATS + 2 * V_FLOATS) * sizeof(float) + 1024;
    // TMEM columns
    static constexpr uint32_t Q_HI = 0, Q_LO = D, O = 2 * D, S = 2 * D + DV, P_LO = S + kBN, COLS = P_LO + kBN;
    static_assert(D % 32 == 0 && DV % 32 == 0 && D <= 128 && DV <= 128, "tcgen05 prefill shape");
    static_assert(COLS <= 512, "TMEM budget");
    static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// Pairwise (tree) max and sum: short dependency chains.
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

template <int N>
__device__ __forceinline__ float tree_sum(const float (&v)[N]) {
    float m[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) m[i] = v[i] + v[i + N / 2];
#pragma unroll
    for (int w = N / 4; w >= 1; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] = m[i] + m[i + w];
    return m[0];
}

// The fused score epilogue over one key tile of one query row, in base 2:
// scale (or softcap), ALiBi, bias, then the mask -- slots outside
// [lo_i, hi_i] become -inf.  `full` tiles skip the mask.  Features are
// template flags so that each combination compiles to straight-line code.
template <bool SOFTCAP, bool ALIBI, bool BIAS, int N>
__device__ __forceinline__ void tile_epilogue(const AttnDesc& a, float (&x)[N], float slope, int rel0,
                                              const float* bias, int lo_i, int hi_i, bool full) {
    if (full) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            float v = SOFTCAP ? a.cap_log2 * tanhf(x[i] * a.qk_mul) : x[i] * a.qk_mul;
            if (ALIBI) v = fmaf(slope, (float)(rel0 + i), v);
            if (BIAS) v = fmaf(__ldg(bias + i), kLog2e, v);
            x[i] = v;
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const bool vis = i >= lo_i && i <= hi_i;
            float v = SOFTCAP ? a.cap_log2 * tanhf(x[i] * a.qk_mul) : x[i] * a.qk_mul;
            if (ALIBI) v = fmaf(slope, (float)(rel0 + i), v);
            if (BIAS) v = fmaf(vis ? __ldg(bias + i) : 0.f, kLog2e, v);
            x[i] = vis ? v : -INFINITY;
        }
    }
}

template <int N>
__device__ __forceinline__ void run_epilogue(int feat, const AttnDesc& a, float (&x)[N], float slope, int rel0,
                                             const float* bias, int lo_i, int hi_i, bool full) {
    switch (feat) {
        case 0: tile_epilogue<false, false, false>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 1: tile_epilogue<true, false, false>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 2: tile_epilogue<false, true, false>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 3: tile_epilogue<true, true, false>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 4: tile_epilogue<false, false, true>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 5: tile_epilogue<true, false, true>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        case 6: tile_epilogue<false, true, true>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
        default: tile_epilogue<true, true, true>(a, x, slope, rel0, bias, lo_i, hi_i, full); break;
    }
}

template <int D, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const AttnDesc a, const AlibiTable alibi, const __grid_constant__ CUtensorMap tm_khi,
                      const __grid_constant__ CUtensorMap tm_klo, const __grid_constant__ CUtensorMap tm_vhi,
                      const __grid_constant__ CUtensorMap tm_vlo) {
    using C = TcCfg<D, DV>;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    float* smem = reinterpret_cast<float*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    __shared__ __align__(8) uint64_t k_full[2], k_empty[2], v_full, v_empty, s_full, p_full, pv_done, q_ready;
    __shared__ uint32_t tmem_base_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_qt = (int)((a.T + kBM - 1) / kBM);
    const int qt = n_qt - 1 - (int)blockIdx.x;  // heaviest (latest) query tiles first
    const int h = blockIdx.y, kh = h / a.G;
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
    const int64_t jt_begin = s_lo / kBN;
    const int n_tiles = (s_hi >= s_lo) ? (int)(s_hi / kBN + 1 - jt_begin) : 0;

    if (threadIdx.x == 0) {
        // Every barrier below completes once per tile (k_* once per two
        // tiles), and no wait ever targets a phase two behind the current.
        for (int b = 0; b < 2; ++b) {
            mbar_init(&k_full[b], 1);
            mbar_init(&k_empty[b], 1);
        }
        mbar_init(&v_full, 1);
        mbar_init(&v_empty, 1);
        mbar_init(&s_full, 1);
        mbar_init(&p_full, 4);
        mbar_init(&pv_done, 1);
        mbar_init(&q_ready, 4);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base_s, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0 && n_tiles > 0) {
            prefetch_tensormap(&tm_khi);
            prefetch_tensormap(&tm_klo);
            prefetch_tensormap(&tm_vhi);
            prefetch_tensormap(&tm_vlo);
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int n0 = (int)((jt_begin + j) * kBN);
                const int b = j & 1;
                if (j >= 2 && !mbar_wait(&k_empty[b], ((j >> 1) - 1) & 1)) {
                    raise_device_error(&g_tc_device_error, kErrTcEmpty);
                    break;
                }
                float* ks = smem + b * C::KSTAGE_FLOATS;
                mbar_arrive_expect_tx(&k_full[b], C::KSTAGE_BYTES);
#pragma unroll
                for (int kb = 0; kb < C::KB; ++kb) {
                    tma_load_2d(ks + kb * kBN * 32, &tm_khi, kh * D + kb * 32, n0, &k_full[b]);
                    tma_load_2d(ks + C::K_FLOATS + kb * kBN * 32, &tm_klo, kh * D + kb * 32, n0, &k_full[b]);
                }
                ++k_issued;
                if (j >= 1 && !mbar_wait(&v_empty, (j - 1) & 1)) {
                    raise_device_error(&g_tc_device_error, kErrTcEmpty);
                    break;
                }
                float* vs = smem + C::V_OFF;
                mbar_arrive_expect_tx(&v_full, C::V_BYTES);
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c) {
                    tma_load_2d(vs + c * DV * 32, &tm_vhi, n0 + c * 32, kh * DV, &v_full);
                    tma_load_2d(vs + C::V_FLOATS + c * DV * 32, &tm_vlo, n0 + c * 32, kh * DV, &v_full);
                }
                ++v_issued;
            }
            // Drain: every copy issued has landed before the CTA moves on.
            bool drained = true;
            for (int j = k_issued > 2 ? k_issued - 2 : 0; j < k_issued; ++j)
                drained &= mbar_wait(&k_full[j & 1], (j >> 1) & 1);
            if (v_issued > 0) drained &= mbar_wait(&v_full, (v_issued - 1) & 1);
            if (!drained) raise_device_error(&g_tc_device_error, kErrTcDrain);
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer --------------------------------
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t id_s = idesc_tf32(kBM, kBN), id_o = idesc_tf32(kBM, DV);
            bool ok = mbar_wait(&q_ready, 0);
            if (!ok) raise_device_error(&g_tc_device_error, kErrTcQ);
            tc_fence_after();
            for (int j = 0; ok && j < n_tiles; ++j) {
                // S_j = Q_hi K_hi + Q_hi K_lo + Q_lo K_hi.  Issued after P.V_{j-1},
                // which read P_hi_{j-1} from the same columns.
                const int b = j & 1;
                if (!mbar_wait(&k_full[b], (j >> 1) & 1)) {
                    raise_device_error(&g_tc_device_error, kErrTcFull);
                    break;
                }
                tc_fence_after();
                const float* ks = smem + b * C::KSTAGE_FLOATS;
                uint32_t acc = 0;
#pragma unroll
                for (int pass = 0; pass < 3; ++pass) {
                    const uint32_t a_col = pass == 2 ? C::Q_LO : C::Q_HI;
                    const float* kt = ks + (pass == 1 ? C::K_FLOATS : 0);
#pragma unroll
                    for (int kb = 0; kb < C::KB; ++kb) {
                        const uint64_t bd = smem_desc_sw128(kt + kb * kBN * 32);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            mma_tf32_ts(tmem + C::S, tmem + a_col + kb * 32 + k * 8, bd + (uint64_t)((k * 32) >> 4),
                                        id_s, acc);
                            acc = 1;
                        }
                    }
                }
                mma_commit(&s_full);
                mma_commit(&k_empty[b]);
                // O += P_hi V_hi + P_hi V_lo + P_lo V_hi.
                if (!mbar_wait(&p_full, j & 1)) {
                    raise_device_error(&g_tc_device_error, kErrTcP);
                    break;
                }
                if (!mbar_wait(&v_full, j & 1)) {
                    raise_device_error(&g_tc_device_error, kErrTcFull);
                    break;
                }
                tc_fence_after();
                const float* vs = smem + C::V_OFF;
#pragma unroll
                for (int pass = 0; pass < 3; ++pass) {
                    const uint32_t a_col = pass == 2 ? C::P_LO : C::S;
                    const float* vt = vs + (pass == 1 ? C::V_FLOATS : 0);
#pragma unroll
                    for (int c = 0; c < kBN / 32; ++c) {
                        const uint64_t bd = smem_desc_sw128(vt + c * DV * 32);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_tf32_ts(tmem + C::O, tmem + a_col + c * 32 + k * 8, bd + (uint64_t)((k * 32) >> 4),
                                        id_o, (j > 0 || pass > 0 || c > 0 || k > 0) ? 1u : 0u);
                    }
                }
                mma_commit(&pv_done);
                mma_commit(&v_empty);
            }
        }
    } else {
        // --------------------- softmax warps: thread = query row ---------------------
        const uint32_t lrow = 32u * (uint32_t)(warp & 3);  // TMEM lane quarter of this warp
        const int r = (int)lrow + lane;
        const int64_t t = t0 + r;
        const bool row_ok = t < a.T;
        const uint32_t trow = tmem + (lrow << 16);
        const float slope = a.alibi_on ? alibi.slope_log2[h] : 0.f;
        // Q row -> hi / lo -> TMEM.
        {
            const float* qrow = a.q + t * (int64_t)a.H * D + (int64_t)h * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                float hi[32], lo[32];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    float4 v4 = row_ok ? __ldg(reinterpret_cast<const float4*>(qrow + c0 + i)) : make_float4(0, 0, 0, 0);
                    const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        hi[i + e] = tf32_hi(vv[e]);
                        lo[i + e] = vv[e] - hi[i + e];
                    }
                }
                tmem_st32(trow + C::Q_HI + c0, hi);
                tmem_st32(trow + C::Q_LO + c0, lo);
            }
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
        const float* brow = a.bias_kind == 0 ? nullptr
                            : a.bias_kind == 1 ? a.bias + t * a.S
                                               : a.bias + ((int64_t)h * a.T + t) * a.S;
        const int feat = (a.softcap_on ? 1 : 0) | (a.alibi_on ? 2 : 0) | (a.bias_kind ? 4 : 0);
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            if (!__all_sync(FULL, mbar_wait(&s_full, j & 1))) {
                raise_device_error(&g_tc_device_error, kErrTcS);
                ok = false;
                break;
            }
            tc_fence_after();
            float x[kBN];
            tmem_ld32(trow + C::S, x);
            tmem_ld32(trow + C::S + 32, x + 32);
            tmem_wait_ld();
            const int64_t n0 = (jt_begin + j) * kBN;
            // Visible slots of this tile, clamped to [-1, kBN].
            const int64_t lo64 = lo_t - n0, hi64 = hi_t - n0;
            const int lo_i = (int)(lo64 < -1 ? -1 : (lo64 > kBN ? kBN : lo64));
            const int hi_i = (int)(hi64 < -1 ? -1 : (hi64 > kBN ? kBN : hi64));
            const bool full = lo_i <= 0 && hi_i >= kBN - 1;
            run_epilogue<kBN>(feat, a, x, slope, (int)(n0 - p), brow ? brow + n0 : nullptr, lo_i, hi_i, full);
            const float mt = tree_max<kBN>(x);
            // Lazy rescale: keep the reference max unless this tile beats it by > 2^8.
            float alpha = 1.f;
            if (mt > m_ref + kRescaleLog2) {
                alpha = fast_exp2(m_ref - mt);  // 0 on the first visible tile
                m_ref = mt;
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
            float plo[kBN];
#pragma unroll
            for (int i = 0; i < kBN; ++i) {
                const float pi = fast_exp2(x[i] - m_use);
                x[i] = tf32_hi(pi);  // P_hi replaces the score in registers
                plo[i] = pi - x[i];
            }
            l = fmaf(l, alpha, tree_sum<kBN>(x) + tree_sum<kBN>(plo));
            // P.V_{j-1} has completed: it ran before S_j in issue order.  The
            // wait costs nothing and makes the O rescale below safe.
            if (j > 0 && !__all_sync(FULL, mbar_wait(&pv_done, (j - 1) & 1))) {
                raise_device_error(&g_tc_device_error, kErrTcPv);
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_st32(trow + C::S, x);
            tmem_st32(trow + C::S + 32, x + 32);
            tmem_st32(trow + C::P_LO, plo);
            tmem_st32(trow + C::P_LO + 32, plo + 32);
            if (j > 0 && __any_sync(FULL, alpha != 1.f)) {
#pragma unroll 1
                for (int c0 = 0; c0 < DV; c0 += 32) {
                    float o[32];
                    tmem_ld32(trow + C::O + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tmem_st32(trow + C::O + c0, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full);
        }
        // Epilogue: O / l -> out.
        if (ok && n_tiles > 0 && !__all_sync(FULL, mbar_wait(&pv_done, (n_tiles - 1) & 1))) {
            raise_device_error(&g_tc_device_error, kErrTcPv);
            ok = false;
        }
        tc_fence_after();
        const float inv = (ok && l > 0.f) ? 1.f / l : 0.f;
        float* orow = a.out + t * (int64_t)a.H * DV + (int64_t)h * DV;
#pragma unroll 1
        for (int c0 = 0; c0 < DV; c0 += 32) {
            float o[32];
            if (n_tiles > 0) {
                tmem_ld32(trow + C::O + c0, o);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = 0.f;
            }
            if (row_ok) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4*>(orow + c0 + i) =
                        make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
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
__global__ void split_k_kernel(const float* __restrict__ k, float* __restrict__ khi, float* __restrict__ klo,
                               int64_t n) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float x = __ldg(k + i);
        const float hi = tf32_hi(x);
        khi[i] = hi;
        klo[i] = x - hi;
    }
}

// v [S, cols] -> vt_hi / vt_lo [cols, s_pad]; columns s >= S are zero.
__global__ void split_vt_kernel(const float* __restrict__ v, float* __restrict__ vthi, float* __restrict__ vtlo,
                                int64_t S, int64_t s_pad, int cols) {
    __shared__ float tile[32][33];
    const int64_t s0 = (int64_t)blockIdx.x * 32;
    const int c0 = blockIdx.y * 32;
    for (int r = threadIdx.y; r < 32; r += blockDim.y) {
        const int64_t s = s0 + r;
        const int c = c0 + threadIdx.x;
        tile[r][threadIdx.x] = (s < S && c < cols) ? __ldg(v + s * cols + c) : 0.f;
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += blockDim.y) {
        const int c = c0 + r;
        const int64_t s = s0 + threadIdx.x;
        if (c < cols && s < s_pad) {
            const float x = tile[threadIdx.x][r];
            const float hi = tf32_hi(x);
            vthi[(int64_t)c * s_pad + s] = hi;
            vtlo[(int64_t)c * s_pad + s] = x - hi;
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
    auto fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * sizeof(float)};
    const cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

template <int D, int DV>
cudaError_t launch_cfg(const AttnDesc& a, const AlibiTable& alibi, float* khi, float* klo, float* vthi,
                       float* vtlo, int64_t s_pad, cudaStream_t stream) {
    using C = TcCfg<D, DV>;
    CUtensorMap m_khi, m_klo, m_vhi, m_vlo;
    if (!encode_sw128(&m_khi, khi, a.S, (int64_t)a.Hk * D, kBN) ||
        !encode_sw128(&m_klo, klo, a.S, (int64_t)a.Hk * D, kBN) ||
        !encode_sw128(&m_vhi, vthi, (int64_t)a.Hk * DV, s_pad, DV) ||
        !encode_sw128(&m_vlo, vtlo, (int64_t)a.Hk * DV, s_pad, DV))
        return cudaErrorInvalidValue;
    auto kern = prefill_tc_kernel<D, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.T + kBM - 1) / kBM), (unsigned)a.H);
    kern<<<grid, kThreads, C::SMEM, stream>>>(a, alibi, m_khi, m_klo, m_vhi, m_vlo);
    return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const AttnDesc& a) {
    const bool dims = (a.D == 32 || a.D == 64 || a.D == 96 || a.D == 128) && a.Dv == a.D;
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
    split_vt_kernel<<<g2, dim3(32, 8), 0, stream>>>(a.v, vthi, vtlo, a.S, L.s_pad, cols);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
#define VTMU_TC(D_) \
    if (a.D == D_) return launch_cfg<D_, D_>(a, alibi, khi, klo, vthi, vtlo, L.s_pad, stream);
    VTMU_TC(32) VTMU_TC(64) VTMU_TC(96) VTMU_TC(128)
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
