// prefill_ffma.cu -- tiled online-softmax attention on FP32 FMA (any T).
//
// Op "attention" (vtmu.mpakt.dev/api/ops).  One CTA owns BM query rows of one
// head and walks the key tiles that the causal/window masks leave visible
// for those rows (tiles wholly outside are never loaded).  Per key tile of
// BN = 64 keys:
//
//   S = Q K^T           register-tiled: thread (ty, tx) holds rows
//                       ty + TY*i (i < 8) x keys tx + TX*j (j < BN/TX)
//   fused epilogue      scale, softcap, ALiBi, bias, mask -- in registers
//   online softmax      running max / sum per row in base 2, rows reduced
//                       across the TX lanes that share them
//   O += P V            P goes through shared memory; thread holds the same
//                       8 rows x dims {tx*4 + TX*4*c + 0..3}
//
// The score tile never reaches global memory.  Q stays in shared memory for
// the CTA's life; K and V tiles are staged with cp.async so that the load of
// V_j overlaps S_j and the load of K_{j+1} overlaps P V_j.  Shared rows are
// padded by 4 floats so the float4 reads of 8 consecutive lanes fall in
// distinct banks.
#include "attn_common.cuh"
#include "kernels.h"
#include "launch_cache.h"

namespace vtmu {
namespace {

template <int BM_, int TX_, int DMAX_, int DVMAX_>
struct PfCfg {
    static constexpr int BM = BM_, TX = TX_, DMAX = DMAX_, DVMAX = DVMAX_;
    static constexpr int BN = 64;
    static constexpr int RPT = 8;              // rows per thread
    static constexpr int TY = BM / RPT;
    static constexpr int THREADS = TY * TX;
    static constexpr int KPT = BN / TX;        // keys per thread
    static constexpr int NDC = DVMAX / (TX * 4);  // float4 value groups per thread
    static constexpr int QLD = DMAX + 4, KLD = DMAX + 4, VLD = DVMAX + 4, PLD = BN + 4;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + BM * QLD;
    static constexpr int V_OFF = K_OFF + BN * KLD;
    static constexpr int P_OFF = V_OFF + BN * VLD;
    static constexpr int FLOATS = P_OFF + BM * PLD;
    static constexpr size_t SMEM = (size_t)FLOATS * sizeof(float);
    static_assert(BM % RPT == 0 && BN % TX == 0 && DVMAX % (TX * 4) == 0, "bad prefill tile");
    static_assert(SMEM <= 227 * 1024, "prefill tile exceeds shared memory");
};

// Copy rows [r0, r0+nrows) x cols [0, ncols_pad) of a row-major global matrix
// (row stride ld, starting column col0) to shared memory (row stride sld).
// Rows >= rmax are zero-filled; columns >= ncols are zero-filled.
template <bool VEC16, int THREADS>
__device__ __forceinline__ void stage_rows(float* sdst, int sld, const float* g, int64_t ld,
                                           int64_t col0, int64_t r0, int nrows, int64_t rmax,
                                           int ncols, int ncols_pad) {
    if constexpr (VEC16) {
        const int cpr = ncols_pad / 4;
        for (int c = threadIdx.x; c < nrows * cpr; c += THREADS) {
            const int row = c / cpr, col = (c % cpr) * 4;
            const int64_t r = r0 + row;
            const bool ok = r < rmax;
            const float* src = g + (ok ? r : 0) * ld + col0 + col;
            cp_async16(sdst + row * sld + col, src, ok ? 16 : 0);
        }
    } else {
        for (int c = threadIdx.x; c < nrows * ncols_pad; c += THREADS) {
            const int row = c / ncols_pad, col = c % ncols_pad;
            const int64_t r = r0 + row;
            const bool ok = r < rmax && col < ncols;
            const float* src = g + (ok ? r * ld + col0 + col : 0);
            cp_async4(sdst + row * sld + col, src, ok ? 4 : 0);
        }
    }
}

// SINKS: attention sinks are on (a separate instantiation keeps their tile
// bookkeeping and mask test out of the common path).
template <class C, bool VEC16, bool SINKS>
__global__ void __launch_bounds__(C::THREADS, 1)
    prefill_ffma_kernel(const AttnDesc a, const AlibiTable alibi) {
    constexpr int BM = C::BM, BN = C::BN, TX = C::TX, TY = C::TY, RPT = C::RPT;
    constexpr int KPT = C::KPT, NDC = C::NDC;
    extern __shared__ __align__(16) float smem[];
    float* sQ = smem + C::Q_OFF;
    float* sK = smem + C::K_OFF;
    float* sV = smem + C::V_OFF;
    float* sP = smem + C::P_OFF;

    const int n_qt = (int)((a.T + BM - 1) / BM);
    // Linear block order: when the query tiles' work differs (causal or
    // windowed), query tile outermost, latest (heaviest) first, so the longest
    // CTAs of every head start first; otherwise heads outermost, so the CTAs
    // running together share one head's K/V in L2.
    const int64_t lin = blockIdx.x + (int64_t)gridDim.x * blockIdx.y;
    const bool uniform = !a.causal && a.window <= 0;
    const int h = (int)(uniform ? lin / n_qt : lin % a.H);
    const int qt = n_qt - 1 - (int)(uniform ? lin % n_qt : lin / a.H);
    const int kh = h / a.G;
    const int tx = threadIdx.x % TX;
    const int ty = threadIdx.x / TX;
    const int64_t t0 = (int64_t)qt * BM;
    const int64_t t_last = (t0 + BM < a.T ? t0 + BM : a.T) - 1;
    const int Dp = (a.D + 3) & ~3;
    const int Dvp = (a.Dv + 3) & ~3;

    // Keys any row of this tile can see.
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
    int64_t jt_begin = s_lo / BN;
    int64_t jt_end = (s_hi >= s_lo) ? s_hi / BN + 1 : jt_begin;
    // Attention sinks: keys s < sink_end stay visible (within the causal
    // limit).  Their tiles come first, or join the window's into one range
    // when the two touch.
    const int64_t sink_cap = a.causal ? s_hi + 1 : a.S;
    const int64_t sinks = SINKS ? a.sinks : 0;
    const int64_t sink_end = sinks < sink_cap ? sinks : sink_cap;
    const int64_t n_st = sink_end > 0 ? (sink_end + BN - 1) / BN : 0;
    int64_t n_sink = 0;
    if (n_st > 0 && n_st >= jt_begin) {
        if (n_st > jt_end) jt_end = n_st;
        jt_begin = 0;
    } else {
        n_sink = n_st;
    }
    const int64_t n_tiles = n_sink + (jt_end - jt_begin);
    auto tile_of = [&](int64_t it) -> int64_t { return it < n_sink ? it : jt_begin + (it - n_sink); };

    const int64_t ldq = (int64_t)a.H * a.D, ldk = (int64_t)a.Hk * a.D, ldv = (int64_t)a.Hk * a.Dv;
    const float slope = a.alibi_on ? alibi.slope_log2[h] : 0.f;

    // Prologue: Q and K_0 in one group, V_0 in the next.
    stage_rows<VEC16, C::THREADS>(sQ, C::QLD, a.q, ldq, (int64_t)h * a.D, t0, BM, a.T, a.D, Dp);
    if (n_tiles > 0)
        stage_rows<VEC16, C::THREADS>(sK, C::KLD, a.k, ldk, (int64_t)kh * a.D, tile_of(0) * BN, BN,
                                      a.S, a.D, Dp);
    cp_async_commit();
    if (n_tiles > 0)
        stage_rows<VEC16, C::THREADS>(sV, C::VLD, a.v, ldv, (int64_t)kh * a.Dv, tile_of(0) * BN, BN,
                                      a.S, a.Dv, Dvp);
    cp_async_commit();

    float m_run[RPT], l_run[RPT];
    float o[RPT][NDC][4];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.f;
#pragma unroll
        for (int c = 0; c < NDC; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[i][c][e] = 0.f;
    }

    for (int64_t it = 0; it < n_tiles; ++it) {
        const int64_t n0 = tile_of(it) * BN;
        const int64_t n_next = it + 1 < n_tiles ? tile_of(it + 1) * BN : 0;
        cp_async_wait<1>();
        __syncthreads();  // K_jt (and Q) landed

        // ---- S = Q K^T ------------------------------------------------------
        float sacc[RPT][KPT];
#pragma unroll
        for (int i = 0; i < RPT; ++i)
#pragma unroll
            for (int j = 0; j < KPT; ++j) sacc[i][j] = 0.f;
#pragma unroll 2
        for (int d = 0; d < Dp; d += 4) {
            float4 qf[RPT], kf[KPT];
#pragma unroll
            for (int i = 0; i < RPT; ++i)
                qf[i] = *reinterpret_cast<const float4*>(sQ + (ty + TY * i) * C::QLD + d);
#pragma unroll
            for (int j = 0; j < KPT; ++j)
                kf[j] = *reinterpret_cast<const float4*>(sK + (tx + TX * j) * C::KLD + d);
#pragma unroll
            for (int i = 0; i < RPT; ++i)
#pragma unroll
                for (int j = 0; j < KPT; ++j) {
                    float acc = sacc[i][j];
                    acc = fmaf(qf[i].x, kf[j].x, acc);
                    acc = fmaf(qf[i].y, kf[j].y, acc);
                    acc = fmaf(qf[i].z, kf[j].z, acc);
                    acc = fmaf(qf[i].w, kf[j].w, acc);
                    sacc[i][j] = acc;
                }
        }

        // ---- fused epilogue + online softmax ------------------------------------
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int64_t t = t0 + ty + TY * i;
            const int64_t p = a.pos_offset + t;
            float mt = -INFINITY;
#pragma unroll
            for (int j = 0; j < KPT; ++j) {
                const int64_t s = n0 + tx + TX * j;
                float x = -INFINITY;
                if (t < a.T && key_visible<SINKS>(a, p, s)) {
                    const float bv = a.bias_kind ? bias_at(a, h, t, s) : 0.f;
                    x = score_log2(a, sacc[i][j], slope, s - p, bv);
                }
                sacc[i][j] = x;
                mt = fmaxf(mt, x);
            }
#pragma unroll
            for (int off = 1; off < TX; off <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            const float m_new = fmaxf(m_run[i], mt);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = exp2f(m_run[i] - m_use);
            float rs = 0.f;
#pragma unroll
            for (int j = 0; j < KPT; ++j) {
                const float pj = exp2f(sacc[i][j] - m_use);
                rs += pj;
                sP[(ty + TY * i) * C::PLD + tx + TX * j] = pj;
            }
            l_run[i] = fmaf(l_run[i], alpha, rs);
            m_run[i] = m_new;
#pragma unroll
            for (int c = 0; c < NDC; ++c)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[i][c][e] *= alpha;
        }
        __syncthreads();  // P written, K_jt consumed

        if (it + 1 < n_tiles)
            stage_rows<VEC16, C::THREADS>(sK, C::KLD, a.k, ldk, (int64_t)kh * a.D, n_next, BN, a.S,
                                          a.D, Dp);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();  // V_jt landed

        // ---- O += P V ---------------------------------------------------------
#pragma unroll 2
        for (int n = 0; n < BN; n += 4) {
            float4 pf[RPT];
#pragma unroll
            for (int i = 0; i < RPT; ++i)
                pf[i] = *reinterpret_cast<const float4*>(sP + (ty + TY * i) * C::PLD + n);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                for (int c = 0; c < NDC; ++c) {
                    const float4 vf =
                        *reinterpret_cast<const float4*>(sV + (n + kk) * C::VLD + tx * 4 + TX * 4 * c);
#pragma unroll
                    for (int i = 0; i < RPT; ++i) {
                        const float pv = kk == 0 ? pf[i].x : kk == 1 ? pf[i].y : kk == 2 ? pf[i].z : pf[i].w;
                        o[i][c][0] = fmaf(pv, vf.x, o[i][c][0]);
                        o[i][c][1] = fmaf(pv, vf.y, o[i][c][1]);
                        o[i][c][2] = fmaf(pv, vf.z, o[i][c][2]);
                        o[i][c][3] = fmaf(pv, vf.w, o[i][c][3]);
                    }
                }
            }
        }
        __syncthreads();  // V_jt and P consumed
        if (it + 1 < n_tiles)
            stage_rows<VEC16, C::THREADS>(sV, C::VLD, a.v, ldv, (int64_t)kh * a.Dv, n_next, BN, a.S,
                                          a.Dv, Dvp);
        cp_async_commit();
    }
    cp_async_wait<0>();

    // ---- normalise and store --------------------------------------------------
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        float l = l_run[i];
#pragma unroll
        for (int off = 1; off < TX; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        const int64_t t = t0 + ty + TY * i;
        if (t >= a.T) continue;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float* orow = a.out + t * (int64_t)a.H * a.Dv + (int64_t)h * a.Dv;
#pragma unroll
        for (int c = 0; c < NDC; ++c) {
            const int d0 = tx * 4 + TX * 4 * c;
            if constexpr (VEC16) {
                if (d0 < a.Dv) {
                    float4 r = make_float4(o[i][c][0] * inv, o[i][c][1] * inv, o[i][c][2] * inv,
                                           o[i][c][3] * inv);
                    *reinterpret_cast<float4*>(orow + d0) = r;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (d0 + e < a.Dv) orow[d0 + e] = o[i][c][e] * inv;
            }
        }
    }
}

using CfgA = PfCfg<128, 16, 128, 128>;  // headDim, vHeadDim <= 128
using CfgB = PfCfg<128, 16, 192, 128>;  // headDim <= 192, vHeadDim <= 128
using CfgC = PfCfg<64, 32, 256, 256>;   // anything up to 256

template <class C, bool VEC16, bool SINKS>
cudaError_t launch_cfg(const AttnDesc& a, const AlibiTable& alibi, cudaStream_t stream) {
    auto kern = prefill_ffma_kernel<C, VEC16, SINKS>;
    cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), (int)C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.T + C::BM - 1) / C::BM), (unsigned)a.H);
    kern<<<grid, C::THREADS, C::SMEM, stream>>>(a, alibi);
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

bool prefill_ffma_supported(const AttnDesc& a) {
    return a.D >= 1 && a.D <= 256 && a.Dv >= 1 && a.Dv <= 256 && a.T <= (int64_t)0x7fffffff * 64;
}

cudaError_t launch_prefill_ffma(const AttnDesc& a, const AlibiTable& alibi, cudaStream_t stream) {
    const bool vec16 = (a.D % 4 == 0) && (a.Dv % 4 == 0) && aligned16(a.q) && aligned16(a.k) &&
                       aligned16(a.v) && aligned16(a.out);
    const bool sinks = a.sinks > 0;
    auto pick = [&](auto cfg) -> cudaError_t {
        using C = decltype(cfg);
        if (sinks)
            return vec16 ? launch_cfg<C, true, true>(a, alibi, stream) : launch_cfg<C, false, true>(a, alibi, stream);
        return vec16 ? launch_cfg<C, true, false>(a, alibi, stream) : launch_cfg<C, false, false>(a, alibi, stream);
    };
    if (a.D <= 128 && a.Dv <= 128) return pick(CfgA{});
    if (a.D <= 192 && a.Dv <= 128) return pick(CfgB{});
    return pick(CfgC{});
}

}  // namespace vtmu
