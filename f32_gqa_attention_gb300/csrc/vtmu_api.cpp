// vtmu_api.cpp -- the C ABI (include/vtmu_attention.h): parameter checks,
// the op's defaults, ALiBi slope tables, kernel choice and launch.
//
// Defaults and parameter meanings follow op "attention" of the op catalog
// (vtmu.mpakt.dev/api/ops): kvHeads defaults to heads, vHeadDim to headDim,
// causal to true, scale to 1/sqrt(headDim); softcap and window are off when
// absent.  A request the build cannot serve is refused with the parameter or
// feature named, as the catalog refuses a graph by naming the missing feature.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda_runtime.h>

#include "kernels.h"
#include "vtmu_attention.h"

namespace {

thread_local std::string g_last_error;

vtmu_status fail(vtmu_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

vtmu_status ok() {
    g_last_error.clear();
    return VTMU_OK;
}

vtmu_status cuda_fail(cudaError_t e, const char* what) {
    return fail(VTMU_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// BLOOM slopes: c = largest power of two <= heads; the first c heads take
// powers 1..c of 2^(-8/c), the rest take the odd powers 1, 3, 5, ... of
// 2^(-4/c).
void bloom_slopes(int heads, double* out) {
    int c = 1;
    while (2 * c <= heads) c *= 2;
    const double base = std::exp2(-8.0 / c);
    double acc = 1.0;
    for (int i = 0; i < c; ++i) {
        acc *= base;
        out[i] = acc;
    }
    const double base2 = std::exp2(-4.0 / c);
    for (int j = 0; j < heads - c; ++j) out[c + j] = std::pow(base2, 2 * j + 1);
}

// MPT slopes with alibi_bias_max b: n = smallest power of two >= heads,
// s_i = 2^(-(i+1) b / n); when n != heads take s_1, s_3, ... (even
// exponents first) then s_0, s_2, ..., cut to heads.
void mpt_slopes(int heads, double bmax, double* out) {
    int n = 1;
    while (n < heads) n *= 2;
    int w = 0;
    if (n == heads) {
        for (int i = 0; i < n; ++i) out[i] = std::exp2(-(i + 1) * bmax / n);
        return;
    }
    for (int i = 1; i < n && w < heads; i += 2) out[w++] = std::exp2(-(i + 1) * bmax / n);
    for (int i = 0; i < n && w < heads; i += 2) out[w++] = std::exp2(-(i + 1) * bmax / n);
}

int device_sm_count() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cached[dev] = n;
    }
    return cached[dev];
}

// Query rows from which AUTO prefers the tensor-core prefill (one 128-row
// MMA tile is then at least half full).
constexpr int64_t kTcMinRows = 64;
// AUTO takes the decode kernel up to this many query rows: it reads K/V once
// per row group (8 virtual heads), where the prefill kernels would read them
// once per query head and fill 64- or 128-row tiles with a few rows.
constexpr int64_t kDecodeAutoRows = 8;

struct Resolved {
    vtmu::AttnDesc a;
    int kernel;  // resolved vtmu_kernel (never AUTO)
};

// Checks that need no pointer, resolves defaults.  Fills r.a except pointers.
vtmu_status resolve(const vtmu_attention_params* p, Resolved* r) {
    if (!p) return fail(VTMU_ERR_INVALID, "params is NULL");
    vtmu::AttnDesc& a = r->a;
    std::memset(&a, 0, sizeof(a));
    if (p->T < 0) return fail(VTMU_ERR_INVALID, "T must be >= 0 (got %lld)", (long long)p->T);
    if (p->S < 0) return fail(VTMU_ERR_INVALID, "S must be >= 0 (got %lld)", (long long)p->S);
    if (p->heads <= 0) return fail(VTMU_ERR_INVALID, "heads must be > 0 (got %d)", p->heads);
    const int Hk = p->kv_heads == 0 ? p->heads : p->kv_heads;
    if (Hk <= 0) return fail(VTMU_ERR_INVALID, "kvHeads must be > 0 (got %d)", p->kv_heads);
    if (p->heads % Hk != 0)
        return fail(VTMU_ERR_INVALID, "heads (%d) must be a multiple of kvHeads (%d)", p->heads, Hk);
    if (p->head_dim <= 0) return fail(VTMU_ERR_INVALID, "headDim must be > 0 (got %d)", p->head_dim);
    const int Dv = p->v_head_dim == 0 ? p->head_dim : p->v_head_dim;
    if (Dv <= 0) return fail(VTMU_ERR_INVALID, "vHeadDim must be > 0 (got %d)", p->v_head_dim);
    if (p->head_dim > 256) return fail(VTMU_ERR_UNSUPPORTED, "headDim %d > 256 is not supported", p->head_dim);
    if (Dv > 256) return fail(VTMU_ERR_UNSUPPORTED, "vHeadDim %d > 256 is not supported", Dv);
    if (p->pos_offset < 0) return fail(VTMU_ERR_RANGE, "posOffset must be >= 0 (got %lld)", (long long)p->pos_offset);
    if (p->window < 0) return fail(VTMU_ERR_INVALID, "window must be >= 0 (got %lld)", (long long)p->window);
    if (p->sinks < 0) return fail(VTMU_ERR_INVALID, "sinks must be >= 0 (got %lld)", (long long)p->sinks);
    if (!(p->softcap >= 0.f) || !std::isfinite(p->softcap))
        return fail(VTMU_ERR_INVALID, "softcap must be finite and >= 0");
    if (p->has_scale && !std::isfinite(p->scale)) return fail(VTMU_ERR_INVALID, "scale must be finite");
    if (p->bias_kind < VTMU_BIAS_NONE || p->bias_kind > VTMU_BIAS_HTS)
        return fail(VTMU_ERR_INVALID, "bias_kind %d is not a vtmu_bias_kind", p->bias_kind);
    if (p->alibi < VTMU_ALIBI_NONE || p->alibi > VTMU_ALIBI_SLOPES)
        return fail(VTMU_ERR_INVALID, "alibi %d is not a vtmu_alibi_kind", p->alibi);
    if (p->alibi == VTMU_ALIBI_SLOPES && !p->alibi_slopes)
        return fail(VTMU_ERR_INVALID, "alibiSlopes: slopes pointer is NULL");
    if (p->alibi == VTMU_ALIBI_MPT && !(p->alibi_max > 0.f && std::isfinite(p->alibi_max)))
        return fail(VTMU_ERR_INVALID, "alibiMax must be finite and > 0");
    if (p->alibi != VTMU_ALIBI_NONE && p->heads > vtmu::kMaxAlibiHeads)
        return fail(VTMU_ERR_UNSUPPORTED, "attention.alibi with heads %d > %d is not supported", p->heads,
                    vtmu::kMaxAlibiHeads);
    if (p->kernel < VTMU_KERNEL_AUTO || p->kernel > VTMU_KERNEL_DECODE_TF32X3)
        return fail(VTMU_ERR_INVALID, "kernel %d is not a vtmu_kernel", p->kernel);
    if (p->decode_splits < 0) return fail(VTMU_ERR_INVALID, "decode_splits must be >= 0");
    if (p->heads > 65535 || Hk > 65535) return fail(VTMU_ERR_UNSUPPORTED, "more than 65535 heads");

    a.T = p->T;
    a.S = p->S;
    a.H = p->heads;
    a.Hk = Hk;
    a.G = p->heads / Hk;
    a.D = p->head_dim;
    a.Dv = Dv;
    a.causal = p->causal ? 1 : 0;
    a.pos_offset = p->pos_offset;
    a.window = p->window;
    a.sinks = p->window > 0 ? p->sinks : 0;  // without a window no key is dropped
    a.bias_kind = p->bias_kind;
    const double scale = p->has_scale ? (double)p->scale : 1.0 / std::sqrt((double)p->head_dim);
    if (p->softcap > 0.f) {
        a.softcap_on = 1;
        a.qk_mul = (float)(scale / (double)p->softcap);
        a.cap_log2 = (float)((double)p->softcap * 1.4426950408889634);
    } else {
        a.softcap_on = 0;
        a.qk_mul = (float)(scale * 1.4426950408889634);
        a.cap_log2 = 0.f;
    }
    a.alibi_on = p->alibi != VTMU_ALIBI_NONE;

    int kernel = p->kernel;
    if (kernel == VTMU_KERNEL_AUTO) {
        if (a.T >= 2 && vtmu::decode_tc_supported(a))
            kernel = VTMU_KERNEL_DECODE_TF32X3;
        else if (a.T <= kDecodeAutoRows && vtmu::decode_supported(a))
            kernel = VTMU_KERNEL_DECODE;
        else if (a.T >= kTcMinRows && vtmu::prefill_tc_supported(a))
            kernel = VTMU_KERNEL_PREFILL_TF32X3;
        else
            kernel = VTMU_KERNEL_PREFILL_FFMA;
    } else if (kernel == VTMU_KERNEL_DECODE) {
        if (a.T < 1 || a.T > vtmu::kDecodeMaxRows)
            return fail(VTMU_ERR_INVALID, "kernel DECODE needs 1 <= T <= %d (got %lld)", vtmu::kDecodeMaxRows,
                        (long long)a.T);
        if (!vtmu::decode_supported(a))
            return fail(VTMU_ERR_UNSUPPORTED,
                        "kernel DECODE covers headDim == vHeadDim in {32,64,128} and group size "
                        "heads/kvHeads in {1,2,4,8} (got headDim %d, vHeadDim %d, group %d)",
                        a.D, a.Dv, a.G);
    } else if (kernel == VTMU_KERNEL_DECODE_TF32X3) {
        if (a.T < 1 || !vtmu::decode_tc_supported(a))
            return fail(VTMU_ERR_UNSUPPORTED,
                        "kernel DECODE_TF32X3 covers 1 <= T * group size <= 16, headDim == vHeadDim == 128, "
                        "no softcap, ALiBi or bias (got T %lld, group %d, headDim %d, vHeadDim %d)",
                        (long long)a.T, a.G, a.D, a.Dv);
    } else if (kernel == VTMU_KERNEL_PREFILL_TF32X3) {
        if (!vtmu::prefill_tc_supported(a))
            return fail(VTMU_ERR_UNSUPPORTED,
                        "kernel PREFILL_TF32X3 covers headDim == vHeadDim in {32,64,96,128,256} and headDim 192 "
                        "with vHeadDim 128, with S >= 1 "
                        "(got headDim %d, vHeadDim %d, S %lld)",
                        a.D, a.Dv, (long long)a.S);
    }
    r->kernel = kernel;
    return VTMU_OK;
}

void fill_alibi(const vtmu_attention_params* p, vtmu::AlibiTable* t) {
    if (p->alibi == VTMU_ALIBI_NONE) return;
    double s[vtmu::kMaxAlibiHeads];
    if (p->alibi == VTMU_ALIBI_BLOOM)
        bloom_slopes(p->heads, s);
    else if (p->alibi == VTMU_ALIBI_MPT)
        mpt_slopes(p->heads, (double)p->alibi_max, s);
    else
        for (int h = 0; h < p->heads; ++h) s[h] = (double)p->alibi_slopes[h];
    for (int h = 0; h < p->heads; ++h) t->slope_log2[h] = (float)(s[h] * 1.4426950408889634);
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

size_t decode_workspace(const vtmu::AttnDesc& a) {
    vtmu::DecodePlan plan;
    vtmu::decode_plan(a, 256, 1, &plan);  // upper bound: the most splits
    return plan.workspace_bytes;
}

size_t decode_tc_workspace(const vtmu::AttnDesc& a) {
    vtmu::DecodeTcPlan plan;
    vtmu::decode_tc_plan(a, 0, 1 << 20, &plan);  // upper bound: the most splits
    return plan.workspace_bytes;
}

size_t attention_workspace(const Resolved& r) {
    return r.kernel == VTMU_KERNEL_DECODE_TF32X3  ? decode_tc_workspace(r.a)
           : r.kernel == VTMU_KERNEL_DECODE         ? decode_workspace(r.a)
           : r.kernel == VTMU_KERNEL_PREFILL_TF32X3 ? vtmu::prefill_tc_workspace(r.a)
                                                    : 0;
}

// Checks op "rope"'s parameters and resolves them for the kernels: the
// inverse frequencies base^(-2j / rotary_dim) (or the given ones) in double,
// with a linear scaling factor divided out.
vtmu_status resolve_rope(const vtmu_rope_params* r, vtmu::RopeDev* out) {
    if (!r) return fail(VTMU_ERR_INVALID, "rope params is NULL");
    if (r->head_dim <= 0 || r->head_dim > 4096)
        return fail(VTMU_ERR_INVALID, "rope: head_dim %d outside 1..4096", r->head_dim);
    const int rd = r->rotary_dim ? r->rotary_dim : r->head_dim;
    if (rd < 0 || rd % 2 != 0 || rd > r->head_dim)
        return fail(VTMU_ERR_INVALID, "rope.rotaryDim: %d must be even and at most head_dim %d", rd, r->head_dim);
    if (rd > 2 * vtmu::kRopeMaxPairs)
        return fail(VTMU_ERR_UNSUPPORTED, "rope.rotaryDim: %d above the %d this build turns", rd,
                    2 * vtmu::kRopeMaxPairs);
    const double base = r->base == 0.f ? 10000.0 : (double)r->base;
    if (!(base > 0.0) || !std::isfinite(base)) return fail(VTMU_ERR_INVALID, "rope: base must be finite and > 0");
    double divisor = 1.0;
    if (r->scaling == VTMU_ROPE_SCALING_LINEAR) {
        divisor = r->scaling_factor;
        if (!(divisor > 0.0) || !std::isfinite(divisor))
            return fail(VTMU_ERR_INVALID, "rope.scaling: linear factor must be finite and > 0");
    } else if (r->scaling != VTMU_ROPE_SCALING_NONE) {
        return fail(VTMU_ERR_UNSUPPORTED,
                    "rope.scaling: kind %d is not served (linear, or explicit inv_freq and attention_factor)",
                    r->scaling);
    }
    const float af = r->attention_factor == 0.f ? 1.f : r->attention_factor;
    if (!std::isfinite(af)) return fail(VTMU_ERR_INVALID, "rope.scaling: attention_factor must be finite");
    std::memset(out, 0, sizeof(*out));
    out->half = rd / 2;
    out->interleaved = r->interleaved ? 1 : 0;
    out->attn = af;
    for (int j = 0; j < rd / 2; ++j) {
        double f = r->inv_freq ? (double)r->inv_freq[j] : std::pow(base, -2.0 * j / rd);
        if (!std::isfinite(f)) return fail(VTMU_ERR_INVALID, "rope.scaling: inv_freq[%d] is not finite", j);
        out->inv_freq[j] = f / divisor;
    }
    return ok();
}

// Workspace of vtmu_decode_step_host: the attention workspace, then the
// staging areas of q, k_new, v_new, bias and out (byte offsets, 256-aligned).
struct HostStaging {
    size_t q, k_new, v_new, bias, out, total;
    size_t q_b, k_new_b, v_new_b, bias_b, out_b;
};

// The device's address of a page-locked host buffer (cudaHostAlloc,
// cudaMallocHost, cudaHostRegister), or nullptr for any other pointer.
void* device_view_of_host(const void* hp) {
    if (!hp) return nullptr;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, hp) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

HostStaging host_staging(const Resolved& r, int64_t new_rows) {
    const vtmu::AttnDesc& a = r.a;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    HostStaging h;
    h.q_b = (size_t)a.T * a.H * a.D * 4;
    h.k_new_b = (size_t)new_rows * a.Hk * a.D * 4;
    h.v_new_b = (size_t)new_rows * a.Hk * a.Dv * 4;
    h.bias_b = a.bias_kind == VTMU_BIAS_TS    ? (size_t)a.T * a.S * 4
               : a.bias_kind == VTMU_BIAS_HTS ? (size_t)a.H * a.T * a.S * 4
                                              : 0;
    h.out_b = (size_t)a.T * a.H * a.Dv * 4;
    h.q = up(attention_workspace(r));
    h.k_new = h.q + up(h.q_b);
    h.v_new = h.k_new + up(h.k_new_b);
    h.bias = h.v_new + up(h.v_new_b);
    h.out = h.bias + up(h.bias_b);
    h.total = h.out + up(h.out_b);
    return h;
}

// Checks of mla_attention's parameters that need no pointer; fills the
// kernels' description (pointers excepted).
vtmu_status resolve_mla(const vtmu_mla_params* p, vtmu::MlaDesc* m) {
    if (!p) return fail(VTMU_ERR_INVALID, "mla params is NULL");
    std::memset(m, 0, sizeof(*m));
    if (p->T < 0 || p->S < 0)
        return fail(VTMU_ERR_INVALID, "mla: T and S must be >= 0 (got %lld, %lld)", (long long)p->T, (long long)p->S);
    if (p->heads <= 0) return fail(VTMU_ERR_INVALID, "mla: heads must be > 0 (got %d)", p->heads);
    if (p->kv_rank <= 0 || p->qk_rope < 0 || p->qk_nope < 0 || p->v_head_dim <= 0 || p->qk_nope + p->qk_rope <= 0)
        return fail(VTMU_ERR_INVALID, "mla: kv_rank, v_head_dim must be > 0 and qk_nope, qk_rope >= 0");
    if (p->kv_rank != vtmu::kMlaKvRank || p->qk_rope != vtmu::kMlaRope)
        return fail(VTMU_ERR_UNSUPPORTED, "mla: this build serves kv_rank %d with qk_rope %d (got %d, %d)",
                    vtmu::kMlaKvRank, vtmu::kMlaRope, p->kv_rank, p->qk_rope);
    if (p->qk_nope > 512) return fail(VTMU_ERR_UNSUPPORTED, "mla: qk_nope %d above 512", p->qk_nope);
    if (p->v_head_dim > 4096) return fail(VTMU_ERR_UNSUPPORTED, "mla: v_head_dim %d above 4096", p->v_head_dim);
    if (p->pos_offset < 0) return fail(VTMU_ERR_RANGE, "mla: posOffset must be >= 0 (got %lld)", (long long)p->pos_offset);
    if (p->window < 0 || p->sinks < 0) return fail(VTMU_ERR_INVALID, "mla: window and sinks must be >= 0");
    if (p->has_scale && !std::isfinite(p->scale)) return fail(VTMU_ERR_INVALID, "mla: scale must be finite");
    if (p->S >= ((int64_t)1 << 31)) return fail(VTMU_ERR_UNSUPPORTED, "mla: S above 2^31 - 1");
    if (p->T * (int64_t)p->heads > 65536)
        return fail(VTMU_ERR_UNSUPPORTED, "mla: T * heads %lld above 65536 (this is the decode form)",
                    (long long)(p->T * (int64_t)p->heads));
    m->T = p->T;
    m->S = p->S;
    m->H = p->heads;
    m->N = p->qk_nope;
    m->Dv = p->v_head_dim;
    m->causal = p->causal ? 1 : 0;
    m->pos_offset = p->pos_offset;
    m->window = p->window;
    m->sinks = p->window > 0 ? p->sinks : 0;  // without a window no key is dropped
    const double scale = p->has_scale ? (double)p->scale : 1.0 / std::sqrt((double)(p->qk_nope + p->qk_rope));
    m->qscale = (float)(scale * 1.4426950408889634);
    if (p->kernel < 0 || p->kernel > 2) return fail(VTMU_ERR_INVALID, "mla: kernel %d is not 0, 1 or 2", p->kernel);
    m->use_tc = p->kernel == 2 ? 1 : 0;
    return VTMU_OK;
}

size_t mla_workspace(const vtmu::MlaDesc& m) {
    // Upper bound over devices: the most splits the plan can choose.
    vtmu::MlaPlan plan;
    vtmu::mla_plan(m, 1 << 20, &plan);
    return plan.workspace_bytes;
}

}  // namespace

namespace vtmu {
// Records `message` as this thread's vtmu_last_error() and returns `status`.
vtmu_status report_error(vtmu_status status, const char* message) { return fail(status, "%s", message); }
}  // namespace vtmu

extern "C" {

void vtmu_attention_params_init(vtmu_attention_params* p) {
    if (!p) return;
    std::memset(p, 0, sizeof(*p));
    p->causal = 1;
}

vtmu_status vtmu_attention_workspace_size(const vtmu_attention_params* p, size_t* bytes) {
    if (!bytes) return fail(VTMU_ERR_INVALID, "bytes is NULL");
    Resolved r;
    vtmu_status st = resolve(p, &r);
    if (st != VTMU_OK) return st;
    *bytes = attention_workspace(r);
    return ok();
}

}  // extern "C"

namespace {

// The pointer checks of op "attention" (nulls, alignment, bias against
// bias_kind, out overlapping an input); launches nothing.
vtmu_status check_pointers(const vtmu::AttnDesc& a, const float* q, const float* k, const float* v,
                           const float* bias, const float* out, const vtmu_attention_params* p) {
    if (!q) return fail(VTMU_ERR_INVALID, "q is NULL");
    if (!out) return fail(VTMU_ERR_INVALID, "out is NULL");
    if (a.S > 0 && (!k || !v)) return fail(VTMU_ERR_INVALID, "k or v is NULL");
    if ((p->bias_kind != VTMU_BIAS_NONE) != (bias != nullptr))
        return fail(VTMU_ERR_INVALID, "attention.bias: bias pointer and bias_kind disagree");
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out) |
                          reinterpret_cast<uintptr_t>(bias);
    if (mis & 3u) return fail(VTMU_ERR_INVALID, "tensor pointers must be 4-byte aligned");
    const size_t out_b = (size_t)a.T * a.H * a.Dv * 4;
    const size_t q_b = (size_t)a.T * a.H * a.D * 4, k_b = (size_t)a.S * a.Hk * a.D * 4,
                 v_b = (size_t)a.S * a.Hk * a.Dv * 4;
    const size_t b_b = p->bias_kind == VTMU_BIAS_TS    ? (size_t)a.T * a.S * 4
                       : p->bias_kind == VTMU_BIAS_HTS ? (size_t)a.H * a.T * a.S * 4
                                                       : 0;
    if (overlaps(out, out_b, q, q_b) || overlaps(out, out_b, k, k_b) || overlaps(out, out_b, v, v_b) ||
        overlaps(out, out_b, bias, b_b))
        return fail(VTMU_ERR_INVALID, "out overlaps an input");
    return VTMU_OK;
}

}  // namespace

namespace vtmu {
// Every check that vtmu_attention makes before it launches the decode kernel
// with params `p` (p->kernel must be VTMU_KERNEL_DECODE), and the scratch
// bytes that launch needs; launches nothing and touches no device memory.
vtmu_status check_decode_call(const vtmu_attention_params* p, const float* q, const float* k, const float* v,
                              const float* bias, const float* out, size_t* scratch_bytes) {
    Resolved r;
    vtmu_status st = resolve(p, &r);
    if (st != VTMU_OK) return st;
    if (r.kernel != VTMU_KERNEL_DECODE) return fail(VTMU_ERR_INVALID, "check_decode_call: kernel is not DECODE");
    if (r.a.T == 0) return fail(VTMU_ERR_INVALID, "decode needs T >= 1");
    st = check_pointers(r.a, q, k, v, bias, out, p);
    if (st != VTMU_OK) return st;
    const uintptr_t m16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out);
    if (m16 & 15u) return fail(VTMU_ERR_UNSUPPORTED, "kernel DECODE needs 16-byte aligned q, k, v, out");
    *scratch_bytes = decode_workspace(r.a);
    return VTMU_OK;
}
}  // namespace vtmu

namespace {

// op "attention" after resolve(); with `cw`, the two cache writes of a
// decode step come first (fused into the decode launch when it runs).
vtmu_status run_attention(Resolved& r, const float* q, const float* k, const float* v, const float* bias,
                          float* out, const vtmu_attention_params* p, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream, const vtmu::DecodeCacheWrite* cw,
                          const vtmu::RopeDev* rope = nullptr) {
    vtmu::AttnDesc& a = r.a;
    cudaError_t e;
    auto write_caches = [&]() -> cudaError_t {
        if (!cw) return cudaSuccess;
        cudaError_t ce = vtmu::launch_cache_write(cw->kc, (int64_t)a.Hk * a.D, cw->k_new, cw->hi - cw->lo,
                                                  cw->lo, stream);
        if (ce != cudaSuccess) return ce;
        return vtmu::launch_cache_write(cw->vc, (int64_t)a.Hk * a.Dv, cw->v_new, cw->hi - cw->lo, cw->lo, stream);
    };
    if (a.T == 0) {
        e = write_caches();
        return e == cudaSuccess ? ok() : cuda_fail(e, "cache_write launch");
    }
    vtmu_status pst = check_pointers(a, q, k, v, bias, out, p);
    if (pst != VTMU_OK) return pst;
    a.q = q;
    a.k = k;
    a.v = v;
    a.bias = bias;
    a.out = out;

    vtmu::AlibiTable alibi;
    fill_alibi(p, &alibi);

    if (r.kernel == VTMU_KERNEL_DECODE_TF32X3) {
        const uintptr_t m16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                              reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out);
        if (m16 & 15u) {
            if (p->kernel == VTMU_KERNEL_DECODE_TF32X3)
                return fail(VTMU_ERR_UNSUPPORTED, "kernel DECODE_TF32X3 needs 16-byte aligned q, k, v, out");
            r.kernel = vtmu::decode_supported(a) && a.T <= kDecodeAutoRows ? VTMU_KERNEL_DECODE
                                                                            : VTMU_KERNEL_PREFILL_FFMA;
        }
    }
    if (r.kernel == VTMU_KERNEL_DECODE_TF32X3) {
        const size_t need = decode_tc_workspace(a);
        if (!workspace || workspace_bytes < need)
            return fail(VTMU_ERR_WORKSPACE, "tensor-core decode needs a workspace of %zu bytes (got %zu)", need,
                        workspace ? workspace_bytes : (size_t)0);
        if (reinterpret_cast<uintptr_t>(workspace) & 255u)
            return fail(VTMU_ERR_WORKSPACE, "workspace must be 256-byte aligned");
        // The new rows go in with the query split when every pointer allows
        // float4 copies, else by the cache_write kernel first.
        const vtmu::DecodeCacheWrite* fused = nullptr;
        if (cw) {
            const uintptr_t c16 = reinterpret_cast<uintptr_t>(cw->kc) | reinterpret_cast<uintptr_t>(cw->vc) |
                                  reinterpret_cast<uintptr_t>(cw->k_new) | reinterpret_cast<uintptr_t>(cw->v_new);
            if (c16 & 15u) {
                if (rope)
                    return fail(VTMU_ERR_UNSUPPORTED,
                                "decode_step_rope: the tensor-core decode turns new keys only from 16-byte aligned "
                                "caches and new rows; compose vtmu_rope and vtmu_decode_step otherwise");
                e = write_caches();
                if (e != cudaSuccess) return cuda_fail(e, "cache_write launch");
            } else {
                fused = cw;
            }
        }
        vtmu::DecodeTcPlan plan;
        vtmu::decode_tc_plan(a, p->decode_splits, device_sm_count(), &plan);
        e = vtmu::launch_decode_tc(a, plan, workspace, stream, fused, rope);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core decode launch");
        return ok();
    }
    if (r.kernel == VTMU_KERNEL_DECODE) {
        const uintptr_t m16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                              reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out);
        if (m16 & 15u) {
            if (p->kernel == VTMU_KERNEL_DECODE)
                return fail(VTMU_ERR_UNSUPPORTED, "kernel DECODE needs 16-byte aligned q, k, v, out");
            r.kernel = VTMU_KERNEL_PREFILL_FFMA;
        }
    }
    if (rope && (r.kernel != VTMU_KERNEL_DECODE || a.T != 1))
        return fail(VTMU_ERR_UNSUPPORTED,
                    "decode_step_rope: the fused step needs a shape of the tensor-core decode, or T == 1 and a "
                    "decode-kernel shape, with 16-byte aligned q, caches, out (T = %lld); compose vtmu_rope and "
                    "vtmu_decode_step otherwise",
                    (long long)a.T);
    if (r.kernel == VTMU_KERNEL_DECODE) {
        const size_t need = decode_workspace(a);
        if (!workspace || workspace_bytes < need)
            return fail(VTMU_ERR_WORKSPACE, "decode needs a zero-initialised workspace of %zu bytes (got %zu)",
                        need, workspace ? workspace_bytes : (size_t)0);
        if (reinterpret_cast<uintptr_t>(workspace) & 255u)
            return fail(VTMU_ERR_WORKSPACE, "workspace must be 256-byte aligned");
        vtmu::DecodePlan plan;
        vtmu::decode_plan(a, p->decode_splits, device_sm_count(), &plan);
        e = vtmu::launch_decode(a, alibi, plan, workspace, stream, cw, rope);
        if (e != cudaSuccess) return cuda_fail(e, "decode launch");
        return ok();
    }
    if (r.kernel == VTMU_KERNEL_PREFILL_TF32X3 && !vtmu::prefill_tc_supported(a)) {
        if (p->kernel == VTMU_KERNEL_PREFILL_TF32X3)
            return fail(VTMU_ERR_UNSUPPORTED, "kernel PREFILL_TF32X3 needs 16-byte aligned q and out");
        r.kernel = VTMU_KERNEL_PREFILL_FFMA;
    }
    if (r.kernel == VTMU_KERNEL_PREFILL_TF32X3) {
        const size_t need = vtmu::prefill_tc_workspace(a);
        if (!workspace || workspace_bytes < need)
            return fail(VTMU_ERR_WORKSPACE, "tensor-core prefill needs a workspace of %zu bytes (got %zu)", need,
                        workspace ? workspace_bytes : (size_t)0);
        if (reinterpret_cast<uintptr_t>(workspace) & 255u)
            return fail(VTMU_ERR_WORKSPACE, "workspace must be 256-byte aligned");
        e = write_caches();
        if (e != cudaSuccess) return cuda_fail(e, "cache_write launch");
        e = vtmu::launch_prefill_tc(a, alibi, workspace, stream);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core prefill launch");
        return ok();
    }
    if (!vtmu::prefill_ffma_supported(a)) return fail(VTMU_ERR_UNSUPPORTED, "shape not covered by the prefill kernel");
    e = write_caches();
    if (e != cudaSuccess) return cuda_fail(e, "cache_write launch");
    e = vtmu::launch_prefill_ffma(a, alibi, stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return ok();
}

}  // namespace

extern "C" {

vtmu_status vtmu_attention(const float* q, const float* k, const float* v, const float* bias, float* out,
                           const vtmu_attention_params* p, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
    Resolved r;
    vtmu_status st = resolve(p, &r);
    if (st != VTMU_OK) return st;
    return run_attention(r, q, k, v, bias, out, p, workspace, workspace_bytes, stream, nullptr);
}

// vtmu_decode_step, with the rotary embedding fused in when `rope` is set.
static vtmu_status decode_step_impl(float* k_cache, float* v_cache, int64_t max_rows, const float* k_new,
                                    const float* v_new, int64_t new_rows, int64_t offset, const float* q,
                                    const float* bias, float* out, const vtmu_attention_params* p,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream,
                                    const vtmu::RopeDev* rope) {
    Resolved r;
    vtmu_status st = resolve(p, &r);
    if (st != VTMU_OK) return st;
    const vtmu::AttnDesc& a = r.a;
    if (rope && a.T < 1)
        return fail(VTMU_ERR_UNSUPPORTED,
                    "decode_step_rope: no query row (T = 0); turn the new keys with vtmu_rope and write them "
                    "with vtmu_decode_step");
    if (max_rows < 0 || new_rows < 0)
        return fail(VTMU_ERR_INVALID, "decode_step: negative size (max_rows %lld, new_rows %lld)",
                    (long long)max_rows, (long long)new_rows);
    if (offset < 0 || offset > max_rows || new_rows > max_rows - offset)
        return fail(VTMU_ERR_RANGE, "decode_step: offset %lld + rows %lld exceeds maxRows %lld", (long long)offset,
                    (long long)new_rows, (long long)max_rows);
    if (a.S > max_rows)
        return fail(VTMU_ERR_INVALID, "decode_step: S %lld exceeds the cache's %lld rows", (long long)a.S,
                    (long long)max_rows);
    if (new_rows == 0) return run_attention(r, q, k_cache, v_cache, bias, out, p, workspace, workspace_bytes,
                                            stream, nullptr, rope);
    if (!k_cache || !v_cache || !k_new || !v_new)
        return fail(VTMU_ERR_INVALID, "decode_step: a cache or new-row pointer is NULL");
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
         reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 3u)
        return fail(VTMU_ERR_INVALID, "decode_step: pointers must be 4-byte aligned");
    const int64_t wk = (int64_t)a.Hk * a.D, wv = (int64_t)a.Hk * a.Dv;
    const size_t kc_b = (size_t)(max_rows * wk) * 4, vc_b = (size_t)(max_rows * wv) * 4;
    const size_t kn_b = (size_t)(new_rows * wk) * 4, vn_b = (size_t)(new_rows * wv) * 4;
    if (overlaps(k_cache, kc_b, v_cache, vc_b)) return fail(VTMU_ERR_INVALID, "decode_step: the caches overlap");
    if (overlaps(k_new, kn_b, k_cache, kc_b) || overlaps(k_new, kn_b, v_cache, vc_b) ||
        overlaps(v_new, vn_b, k_cache, kc_b) || overlaps(v_new, vn_b, v_cache, vc_b))
        return fail(VTMU_ERR_INVALID, "decode_step: new rows overlap a cache");
    if (out && (overlaps(out, (size_t)a.T * a.H * a.Dv * 4, k_cache, kc_b) ||
                overlaps(out, (size_t)a.T * a.H * a.Dv * 4, v_cache, vc_b)))
        return fail(VTMU_ERR_INVALID, "decode_step: out overlaps a cache");
    vtmu::DecodeCacheWrite cw{k_cache, v_cache, k_new, v_new, offset, offset + new_rows};
    return run_attention(r, q, k_cache, v_cache, bias, out, p, workspace, workspace_bytes, stream, &cw, rope);
}

vtmu_status vtmu_decode_step(float* k_cache, float* v_cache, int64_t max_rows, const float* k_new,
                             const float* v_new, int64_t new_rows, int64_t offset, const float* q,
                             const float* bias, float* out, const vtmu_attention_params* p, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
    return decode_step_impl(k_cache, v_cache, max_rows, k_new, v_new, new_rows, offset, q, bias, out, p, workspace,
                            workspace_bytes, stream, nullptr);
}

void vtmu_rope_params_init(vtmu_rope_params* r) {
    if (r) std::memset(r, 0, sizeof(*r));
}

vtmu_status vtmu_rope(const float* x, float* out, int64_t T, int32_t heads, int64_t offset,
                      const vtmu_rope_params* rp, cudaStream_t stream) {
    vtmu::RopeDev rd;
    vtmu_status st = resolve_rope(rp, &rd);
    if (st != VTMU_OK) return st;
    if (T < 0 || heads <= 0)
        return fail(VTMU_ERR_INVALID, "rope: T %lld and heads %d must be >= 0 and > 0", (long long)T, heads);
    if (offset < 0) return fail(VTMU_ERR_RANGE, "rope: offset %lld is negative", (long long)offset);
    if (T == 0) return ok();
    if (!x || !out) return fail(VTMU_ERR_INVALID, "rope: x or out is NULL");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 3u)
        return fail(VTMU_ERR_INVALID, "rope: pointers must be 4-byte aligned");
    const size_t nb = (size_t)T * heads * rp->head_dim * 4;
    if (x != out && overlaps(x, nb, out, nb))
        return fail(VTMU_ERR_INVALID, "rope: out overlaps x without being x");
    cudaError_t e = vtmu::launch_rope(x, out, T, heads, rp->head_dim, offset, rd, stream);
    if (e != cudaSuccess) return cuda_fail(e, "rope launch");
    return ok();
}

vtmu_status vtmu_decode_step_rope(float* k_cache, float* v_cache, int64_t max_rows, const float* k_new,
                                  const float* v_new, int64_t new_rows, int64_t offset, const float* q,
                                  const float* bias, float* out, const vtmu_attention_params* p,
                                  const vtmu_rope_params* rope, void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream) {
    vtmu::RopeDev rd;
    vtmu_status st = resolve_rope(rope, &rd);
    if (st != VTMU_OK) return st;
    if (!p) return fail(VTMU_ERR_INVALID, "params is NULL");
    if (rope->head_dim != p->head_dim)
        return fail(VTMU_ERR_INVALID, "decode_step_rope: rope head_dim %d differs from head_dim %d", rope->head_dim,
                    p->head_dim);
    return decode_step_impl(k_cache, v_cache, max_rows, k_new, v_new, new_rows, offset, q, bias, out, p, workspace,
                            workspace_bytes, stream, &rd);
}

vtmu_status vtmu_decode_step_host_workspace_size(const vtmu_attention_params* p, int64_t new_rows, size_t* bytes) {
    if (!bytes) return fail(VTMU_ERR_INVALID, "bytes is NULL");
    if (new_rows < 0) return fail(VTMU_ERR_INVALID, "decode_step_host: negative new_rows %lld", (long long)new_rows);
    Resolved r;
    vtmu_status st = resolve(p, &r);
    if (st != VTMU_OK) return st;
    *bytes = host_staging(r, new_rows).total;
    return ok();
}

vtmu_status vtmu_decode_step_host(float* k_cache, float* v_cache, int64_t max_rows, const float* k_new_host,
                                  const float* v_new_host, int64_t new_rows, int64_t offset, const float* q_host,
                                  const float* bias_host, float* out_host, const vtmu_attention_params* p,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    Resolved r;
    vtmu_status st = resolve(p, &r);
    if (st != VTMU_OK) return st;
    const vtmu::AttnDesc& a = r.a;
    if (max_rows < 0 || new_rows < 0)
        return fail(VTMU_ERR_INVALID, "decode_step_host: negative size (max_rows %lld, new_rows %lld)",
                    (long long)max_rows, (long long)new_rows);
    if (offset < 0 || offset > max_rows || new_rows > max_rows - offset)
        return fail(VTMU_ERR_RANGE, "decode_step_host: offset %lld + rows %lld exceeds maxRows %lld",
                    (long long)offset, (long long)new_rows, (long long)max_rows);
    const HostStaging h = host_staging(r, new_rows);
    if (!workspace || workspace_bytes < h.total)
        return fail(VTMU_ERR_WORKSPACE, "decode_step_host: workspace of %zu bytes, %zu needed", workspace_bytes,
                    h.total);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(VTMU_ERR_INVALID, "decode_step_host: workspace must be 256-byte aligned");
    if ((h.q_b && !q_host) || (h.out_b && !out_host) || (h.k_new_b && !k_new_host) ||
        (h.v_new_b && !v_new_host))
        return fail(VTMU_ERR_INVALID, "decode_step_host: a host buffer is NULL");
    if ((p->bias_kind != VTMU_BIAS_NONE) != (bias_host != nullptr))
        return fail(VTMU_ERR_INVALID, "attention.bias: bias pointer and bias_kind disagree");
    if (new_rows > 0 && (!k_cache || !v_cache))
        return fail(VTMU_ERR_INVALID, "decode_step_host: a cache pointer is NULL");
    if (a.S > max_rows)
        return fail(VTMU_ERR_INVALID, "decode_step_host: S %lld exceeds the cache's %lld rows", (long long)a.S,
                    (long long)max_rows);
    char* w = static_cast<char*>(workspace);
    // On a decode kernel, which reads q and the new rows with plain loads
    // and writes the output row with plain stores, page-locked buffers the
    // device can address are used in place: the kernel pulls q and the new
    // rows over the host link and pushes the output row back, with no
    // staging copies.
    // Only when all of them qualify and they and the caches are 16-byte
    // aligned (so that the decode kernel runs and none of its fallbacks) and
    // no bias is given; otherwise every buffer goes through the workspace.
    const bool decode_kernel = r.kernel == VTMU_KERNEL_DECODE || r.kernel == VTMU_KERNEL_DECODE_TF32X3;
    if (decode_kernel && !bias_host && h.q_b && h.out_b) {
        void* q_d = device_view_of_host(q_host);
        void* out_d = device_view_of_host(out_host);
        void* kn_d = h.k_new_b ? device_view_of_host(k_new_host) : nullptr;
        void* vn_d = h.v_new_b ? device_view_of_host(v_new_host) : nullptr;
        const uintptr_t m16 = reinterpret_cast<uintptr_t>(q_d) | reinterpret_cast<uintptr_t>(out_d) |
                              reinterpret_cast<uintptr_t>(kn_d) | reinterpret_cast<uintptr_t>(vn_d) |
                              reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache);
        if (q_d && out_d && (!h.k_new_b || (kn_d && vn_d)) && (m16 & 15u) == 0) {
            st = vtmu_decode_step(k_cache, v_cache, max_rows, static_cast<const float*>(kn_d),
                                  static_cast<const float*>(vn_d), new_rows, offset, static_cast<const float*>(q_d),
                                  nullptr, static_cast<float*>(out_d), p, workspace, h.q, stream);
            if (st != VTMU_OK) return st;
            const cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return cuda_fail(e, "decode_step_host: stream synchronisation");
            return ok();
        }
    }
    auto stage = [&](size_t off, const float* src, size_t n) -> cudaError_t {
        return n ? cudaMemcpyAsync(w + off, src, n, cudaMemcpyHostToDevice, stream) : cudaSuccess;
    };
    cudaError_t e = stage(h.q, q_host, h.q_b);
    if (e == cudaSuccess) e = stage(h.k_new, k_new_host, h.k_new_b);
    if (e == cudaSuccess) e = stage(h.v_new, v_new_host, h.v_new_b);
    if (e == cudaSuccess) e = stage(h.bias, bias_host, h.bias_b);
    if (e != cudaSuccess) return cuda_fail(e, "decode_step_host: host to device copy");
    auto dev = [&](size_t off, size_t n) -> float* { return n ? reinterpret_cast<float*>(w + off) : nullptr; };
    st = vtmu_decode_step(k_cache, v_cache, max_rows, dev(h.k_new, h.k_new_b), dev(h.v_new, h.v_new_b), new_rows,
                          offset, dev(h.q, h.q_b), dev(h.bias, h.bias_b), dev(h.out, h.out_b), p, workspace, h.q,
                          stream);
    if (st != VTMU_OK) return st;
    if (h.out_b) {
        e = cudaMemcpyAsync(out_host, w + h.out, h.out_b, cudaMemcpyDeviceToHost, stream);
        if (e != cudaSuccess) return cuda_fail(e, "decode_step_host: device to host copy");
    }
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode_step_host: stream synchronisation");
    return ok();
}

vtmu_status vtmu_cache_write(float* cache, int64_t max_rows, int64_t width, const float* values, int64_t rows,
                             int64_t offset, cudaStream_t stream) {
    if (max_rows < 0 || width < 0 || rows < 0)
        return fail(VTMU_ERR_INVALID, "cache_write: negative size (max_rows %lld, width %lld, rows %lld)",
                    (long long)max_rows, (long long)width, (long long)rows);
    if (offset < 0 || offset > max_rows || rows > max_rows - offset)
        return fail(VTMU_ERR_RANGE, "cache_write: offset %lld + rows %lld exceeds maxRows %lld", (long long)offset,
                    (long long)rows, (long long)max_rows);
    if (rows == 0 || width == 0) return ok();
    if (!cache || !values) return fail(VTMU_ERR_INVALID, "cache_write: cache or values is NULL");
    if ((reinterpret_cast<uintptr_t>(cache) | reinterpret_cast<uintptr_t>(values)) & 3u)
        return fail(VTMU_ERR_INVALID, "cache_write: pointers must be 4-byte aligned");
    if (overlaps(cache + offset * width, (size_t)(rows * width) * 4, values, (size_t)(rows * width) * 4))
        return fail(VTMU_ERR_INVALID, "cache_write: values overlap the destination rows");
    cudaError_t e = vtmu::launch_cache_write(cache, width, values, rows, offset, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cache_write launch");
    return ok();
}

void vtmu_mla_params_init(vtmu_mla_params* p) {
    if (!p) return;
    std::memset(p, 0, sizeof(*p));
    p->causal = 1;
    p->kv_rank = vtmu::kMlaKvRank;
    p->qk_rope = vtmu::kMlaRope;
}

vtmu_status vtmu_mla_workspace_size(const vtmu_mla_params* p, size_t* bytes) {
    if (!bytes) return fail(VTMU_ERR_INVALID, "bytes is NULL");
    vtmu::MlaDesc m;
    vtmu_status st = resolve_mla(p, &m);
    if (st != VTMU_OK) return st;
    *bytes = mla_workspace(m);
    return ok();
}

// mla_attention after resolve_mla(), with the decode step's cache write.
static vtmu_status run_mla(vtmu::MlaDesc& m, const float* q, const float* state, const float* k_b,
                           const float* v_b, float* out, void* workspace, size_t workspace_bytes,
                           const vtmu::MlaCacheWrite& cw, cudaStream_t stream) {
    if (m.T > 0) {
        if (!q || (m.N > 0 && !k_b) || !v_b || !out || (m.S > 0 && !state))
            return fail(VTMU_ERR_INVALID, "mla: q, state, k_b, v_b or out is NULL");
        if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 3u)
            return fail(VTMU_ERR_INVALID, "mla: q and out must be 4-byte aligned");
        if ((reinterpret_cast<uintptr_t>(state) | reinterpret_cast<uintptr_t>(k_b) | reinterpret_cast<uintptr_t>(v_b)) &
            15u)
            return fail(VTMU_ERR_INVALID, "mla: state, k_b and v_b must be 16-byte aligned");
        const size_t W = (size_t)vtmu::kMlaKvRank + vtmu::kMlaRope;
        const size_t out_b = (size_t)m.T * m.H * m.Dv * 4;
        if (overlaps(out, out_b, q, (size_t)m.T * m.H * (m.N + vtmu::kMlaRope) * 4) ||
            overlaps(out, out_b, state, (size_t)m.S * W * 4) ||
            overlaps(out, out_b, k_b, (size_t)m.H * m.N * vtmu::kMlaKvRank * 4) ||
            overlaps(out, out_b, v_b, (size_t)m.H * m.Dv * vtmu::kMlaKvRank * 4))
            return fail(VTMU_ERR_INVALID, "mla: out overlaps an input");
    }
    vtmu::MlaPlan plan;
    vtmu::mla_plan(m, device_sm_count(), &plan);
    const size_t need = mla_workspace(m);
    if (!workspace || workspace_bytes < need)
        return fail(VTMU_ERR_WORKSPACE, "mla needs a workspace of %zu bytes (got %zu)", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(VTMU_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    m.q = q;
    m.state = state;
    m.k_b = k_b;
    m.v_b = v_b;
    m.out = out;
    cudaError_t e = vtmu::launch_mla(m, plan, workspace, cw, stream);
    if (e != cudaSuccess) return cuda_fail(e, "mla launch");
    return ok();
}

vtmu_status vtmu_mla_attention(const float* q, const float* state, const float* k_b, const float* v_b, float* out,
                               const vtmu_mla_params* p, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
    vtmu::MlaDesc m;
    vtmu_status st = resolve_mla(p, &m);
    if (st != VTMU_OK) return st;
    if (m.T == 0) return ok();
    const vtmu::MlaCacheWrite none{nullptr, nullptr, 0, 0};
    return run_mla(m, q, state, k_b, v_b, out, workspace, workspace_bytes, none, stream);
}

vtmu_status vtmu_mla_decode_step(float* state, int64_t max_rows, const float* state_new, int64_t new_rows,
                                 int64_t offset, const float* q, const float* k_b, const float* v_b, float* out,
                                 const vtmu_mla_params* p, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
    vtmu::MlaDesc m;
    vtmu_status st = resolve_mla(p, &m);
    if (st != VTMU_OK) return st;
    if (max_rows < 0 || new_rows < 0)
        return fail(VTMU_ERR_INVALID, "mla_decode_step: negative size (max_rows %lld, new_rows %lld)",
                    (long long)max_rows, (long long)new_rows);
    if (offset < 0 || offset > max_rows || new_rows > max_rows - offset)
        return fail(VTMU_ERR_RANGE, "mla_decode_step: offset %lld + rows %lld exceeds maxRows %lld",
                    (long long)offset, (long long)new_rows, (long long)max_rows);
    if (m.S > max_rows)
        return fail(VTMU_ERR_INVALID, "mla_decode_step: S %lld exceeds the cache's %lld rows", (long long)m.S,
                    (long long)max_rows);
    const size_t W = (size_t)vtmu::kMlaKvRank + vtmu::kMlaRope;
    vtmu::MlaCacheWrite cw{nullptr, nullptr, 0, 0};
    if (new_rows > 0) {
        if (!state || !state_new) return fail(VTMU_ERR_INVALID, "mla_decode_step: state or state_new is NULL");
        if ((reinterpret_cast<uintptr_t>(state) | reinterpret_cast<uintptr_t>(state_new)) & 15u)
            return fail(VTMU_ERR_INVALID, "mla_decode_step: state and state_new must be 16-byte aligned");
        if (overlaps(state, (size_t)max_rows * W * 4, state_new, (size_t)new_rows * W * 4))
            return fail(VTMU_ERR_INVALID, "mla_decode_step: state_new overlaps the cache");
        if (out && overlaps(out, (size_t)m.T * m.H * m.Dv * 4, state, (size_t)max_rows * W * 4))
            return fail(VTMU_ERR_INVALID, "mla_decode_step: out overlaps the cache");
        cw = vtmu::MlaCacheWrite{state, state_new, new_rows, offset};
    }
    if (m.T == 0) {  // the cache write alone
        if (new_rows == 0) return ok();
        cudaError_t e = vtmu::launch_cache_write(state, (int64_t)W, state_new, new_rows, offset, stream);
        return e == cudaSuccess ? ok() : cuda_fail(e, "cache_write launch");
    }
    return run_mla(m, q, state, k_b, v_b, out, workspace, workspace_bytes, cw, stream);
}

// Staging areas of vtmu_mla_decode_step_host after the latent attention's
// own workspace: q, the new cache rows, the output.
struct MlaHostStaging {
    size_t q, q_b, sn, sn_b, out, out_b, total;
};
static MlaHostStaging mla_host_staging(const vtmu::MlaDesc& m, int64_t new_rows) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    MlaHostStaging h;
    h.q_b = (size_t)m.T * m.H * (m.N + vtmu::kMlaRope) * 4;
    h.sn_b = (size_t)new_rows * (vtmu::kMlaKvRank + vtmu::kMlaRope) * 4;
    h.out_b = (size_t)m.T * m.H * m.Dv * 4;
    h.q = up(mla_workspace(m));
    h.sn = h.q + up(h.q_b);
    h.out = h.sn + up(h.sn_b);
    h.total = h.out + up(h.out_b);
    return h;
}

vtmu_status vtmu_mla_decode_step_host_workspace_size(const vtmu_mla_params* p, int64_t new_rows, size_t* bytes) {
    if (!bytes) return fail(VTMU_ERR_INVALID, "bytes is NULL");
    if (new_rows < 0) return fail(VTMU_ERR_INVALID, "mla_decode_step_host: negative new_rows %lld", (long long)new_rows);
    vtmu::MlaDesc m;
    vtmu_status st = resolve_mla(p, &m);
    if (st != VTMU_OK) return st;
    *bytes = mla_host_staging(m, new_rows).total;
    return ok();
}

vtmu_status vtmu_mla_decode_step_host(float* state, int64_t max_rows, const float* state_new_host, int64_t new_rows,
                                      int64_t offset, const float* q_host, const float* k_b, const float* v_b,
                                      float* out_host, const vtmu_mla_params* p, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream) {
    vtmu::MlaDesc m;
    vtmu_status st = resolve_mla(p, &m);
    if (st != VTMU_OK) return st;
    if (new_rows < 0) return fail(VTMU_ERR_INVALID, "mla_decode_step_host: negative new_rows %lld", (long long)new_rows);
    const MlaHostStaging h = mla_host_staging(m, new_rows);
    if (!workspace || workspace_bytes < h.total)
        return fail(VTMU_ERR_WORKSPACE, "mla_decode_step_host: workspace of %zu bytes, %zu needed",
                    workspace ? workspace_bytes : (size_t)0, h.total);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(VTMU_ERR_INVALID, "mla_decode_step_host: workspace must be 256-byte aligned");
    if ((h.q_b && !q_host) || (h.out_b && !out_host) || (h.sn_b && !state_new_host))
        return fail(VTMU_ERR_INVALID, "mla_decode_step_host: a host buffer is NULL");
    // The checks of vtmu_mla_decode_step on the device buffers, before any copy.
    if (max_rows < 0) return fail(VTMU_ERR_INVALID, "mla_decode_step_host: negative max_rows %lld", (long long)max_rows);
    if (offset < 0 || offset > max_rows || new_rows > max_rows - offset)
        return fail(VTMU_ERR_RANGE, "mla_decode_step_host: offset %lld + rows %lld exceeds maxRows %lld",
                    (long long)offset, (long long)new_rows, (long long)max_rows);
    if (m.S > max_rows)
        return fail(VTMU_ERR_INVALID, "mla_decode_step_host: S %lld exceeds the cache's %lld rows", (long long)m.S,
                    (long long)max_rows);
    if ((new_rows > 0 || (m.T > 0 && m.S > 0)) && !state)
        return fail(VTMU_ERR_INVALID, "mla_decode_step_host: state is NULL");
    if (m.T > 0 && ((m.N > 0 && !k_b) || !v_b))
        return fail(VTMU_ERR_INVALID, "mla_decode_step_host: k_b or v_b is NULL");
    if ((reinterpret_cast<uintptr_t>(state) | reinterpret_cast<uintptr_t>(k_b) | reinterpret_cast<uintptr_t>(v_b)) & 15u)
        return fail(VTMU_ERR_INVALID, "mla_decode_step_host: state, k_b and v_b must be 16-byte aligned");
    char* w = static_cast<char*>(workspace);
    const size_t ws_attn = h.q;  // the latent attention's own part of the workspace
    // Page-locked, device-addressable buffers are used in place, as in
    // vtmu_decode_step_host: the absorb launch reads q and the new rows and
    // the projection writes the output row with plain loads and stores.
    // Buffers the launches could not take as they are (q or out not 4-byte
    // aligned, new rows not 16-byte aligned) go through the workspace.
    if (h.q_b && h.out_b) {
        void* q_d = device_view_of_host(q_host);
        void* out_d = device_view_of_host(out_host);
        void* sn_d = h.sn_b ? device_view_of_host(state_new_host) : nullptr;
        const bool aligned = ((reinterpret_cast<uintptr_t>(q_d) | reinterpret_cast<uintptr_t>(out_d)) & 3u) == 0 &&
                             (reinterpret_cast<uintptr_t>(sn_d) & 15u) == 0;
        if (q_d && out_d && (!h.sn_b || sn_d) && aligned) {
            st = vtmu_mla_decode_step(state, max_rows, static_cast<const float*>(sn_d), new_rows, offset,
                                      static_cast<const float*>(q_d), k_b, v_b, static_cast<float*>(out_d), p,
                                      workspace, ws_attn, stream);
            if (st != VTMU_OK) return st;
            const cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return cuda_fail(e, "mla_decode_step_host: stream synchronisation");
            return ok();
        }
    }
    cudaError_t e = cudaSuccess;
    if (h.q_b) e = cudaMemcpyAsync(w + h.q, q_host, h.q_b, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess && h.sn_b) e = cudaMemcpyAsync(w + h.sn, state_new_host, h.sn_b, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "mla_decode_step_host: host to device copy");
    st = vtmu_mla_decode_step(state, max_rows, h.sn_b ? reinterpret_cast<const float*>(w + h.sn) : nullptr,
                              new_rows, offset, h.q_b ? reinterpret_cast<const float*>(w + h.q) : nullptr, k_b, v_b,
                              h.out_b ? reinterpret_cast<float*>(w + h.out) : nullptr, p, workspace, ws_attn, stream);
    if (st != VTMU_OK) return st;
    if (h.out_b) {
        e = cudaMemcpyAsync(out_host, w + h.out, h.out_b, cudaMemcpyDeviceToHost, stream);
        if (e != cudaSuccess) return cuda_fail(e, "mla_decode_step_host: device to host copy");
    }
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "mla_decode_step_host: stream synchronisation");
    return ok();
}

const char* vtmu_features(void) {
    return "attention.alibi attention.bias attention.scale attention.softcap attention.window rope.interleaved "
           "rope.rotaryDim";
}

const char* vtmu_last_error(void) { return g_last_error.c_str(); }

vtmu_status vtmu_device_error(unsigned int* flags) {
    if (!flags) return fail(VTMU_ERR_INVALID, "flags is NULL");
    *flags = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "device_error: synchronize");
    *flags = vtmu::decode_take_device_error() | vtmu::decode_tc_take_device_error() | vtmu::tc_take_device_error() |
             vtmu::mla_take_device_error() |
             vtmu::mla_tc_take_device_error();
    return ok();
}

}  // extern "C"
