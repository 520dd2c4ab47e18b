/*
 * attention_oracle.c -- plain, slow CPU oracle for the f32 `attention`,
 * `cache_write` and `rope` ops of the volunteer-inference op catalog
 * (vtmu.mpakt.dev/api/ops, ops "attention", "cache_write" and "rope"), and
 * for the absorbed latent attention of the IR schema page
 * ($defs.op_mla_attention), at the end of this file.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (op catalog, op "attention"): for every query head h and
 * query row t, with G = heads / kvHeads and p = posOffset + t,
 *
 *   key s is visible  iff  (!causal || s <= p)  and
 *                          (window == 0 ||
 *                           (causal ? p - window < s : |p - s| <= window))
 *   x_s = scale * sum_d q[t, h*D + d] * k[s, (h/G)*D + d]
 *   x_s = softcap * tanh(x_s / softcap)               (if softcap > 0)
 *   x_s = x_s + slope_h * (s - p)                     (if ALiBi)
 *   x_s = x_s + bias[t, s]  or  bias[h, t, s]         (if bias)
 *   m   = max over visible s of x_s
 *   out[t, h*Dv + e] = sum_s exp(x_s - m) v[s, (h/G)*Dv + e] / sum_s exp(x_s - m)
 *
 * and zeros for a row with no visible key (or whose visible keys all have a
 * score of -inf).  Every sum and every score is kept in double; inputs are
 * the caller's f32 arrays, outputs are double.
 *
 * The order scale -> softcap -> ALiBi -> bias -> mask follows the catalog's
 * feature table (the cap comes ahead of masking) and its bias text
 * (-1e9 masks, which only works if the bias is added after the cap).
 *
 * ALiBi slopes follow the geometric sequences BLOOM and MPT use
 * (Press et al., "Train Short, Test Long", 2022), computed in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BIAS_NONE 0
#define ORACLE_BIAS_TS 1  /* bias [T, S], shared by every head */
#define ORACLE_BIAS_HTS 2 /* bias [heads, T, S] */

#define ORACLE_ALIBI_BLOOM 1
#define ORACLE_ALIBI_MPT 2

typedef struct {
    int64_t T, S;
    int heads, kv_heads, head_dim, v_head_dim;
    int causal;
    int64_t pos_offset;
    double scale;   /* already resolved: 1/sqrt(head_dim) unless overridden */
    double softcap; /* 0 = off */
    int64_t window; /* 0 = off */
    const double* slopes; /* [heads] or NULL */
    int bias_kind;
    int64_t sinks;  /* 0 = none */
} oracle_attn_desc;

/* op "attention", param "window": causal keys are visible when
 * pos - window < s <= pos, non-causal ones when |pos - s| <= window.
 * Attention sinks (the IR page's integer `sinks` beside `window`, read as
 * the sink tokens of streaming attention): with a window, keys s < sinks
 * stay visible wherever the window has moved (still subject to causality). */
static int key_visible(int causal, int64_t window, int64_t sinks, int64_t p, int64_t s)
{
    if (causal && s > p) return 0;
    if (window > 0) {
        if (s < sinks) return 1;
        if (causal) {
            if (!(p - window < s)) return 0;
        } else {
            int64_t dist = p > s ? p - s : s - p;
            if (dist > window) return 0;
        }
    }
    return 1;
}

/* One query row t of head h.  x is scratch of S doubles, o receives Dv values. */
static void attend_row(const oracle_attn_desc* a, const float* q, const float* k,
                       const float* v, const float* bias, int64_t t, int h,
                       double* x, char* vis, double* o)
{
    const int G = a->heads / a->kv_heads;
    const int kh = h / G;
    const int D = a->head_dim, Dv = a->v_head_dim;
    const int64_t p = a->pos_offset + t;
    const float* qrow = q + t * (int64_t)a->heads * D + (int64_t)h * D;
    double m = -INFINITY;

    for (int64_t s = 0; s < a->S; ++s) {
        vis[s] = (char)key_visible(a->causal, a->window, a->sinks, p, s);
        if (!vis[s]) continue;
        const float* krow = k + s * (int64_t)a->kv_heads * D + (int64_t)kh * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += (double)qrow[d] * (double)krow[d];
        double xs = a->scale * dot;
        if (a->softcap > 0.0) xs = a->softcap * tanh(xs / a->softcap);
        if (a->slopes) xs += a->slopes[h] * (double)(s - p);
        if (a->bias_kind == ORACLE_BIAS_TS)
            xs += (double)bias[t * a->S + s];
        else if (a->bias_kind == ORACLE_BIAS_HTS)
            xs += (double)bias[((int64_t)h * a->T + t) * a->S + s];
        x[s] = xs;
        if (xs > m) m = xs;
    }

    for (int e = 0; e < Dv; ++e) o[e] = 0.0;
    if (m == -INFINITY) return; /* nothing visible: the row is zero */

    /* op "softmax": the row maximum is subtracted first, which keeps exp finite. */
    double l = 0.0;
    for (int64_t s = 0; s < a->S; ++s) {
        if (!vis[s]) continue;
        double w = exp(x[s] - m);
        l += w;
        const float* vrow = v + s * (int64_t)a->kv_heads * Dv + (int64_t)kh * Dv;
        for (int e = 0; e < Dv; ++e) o[e] += w * (double)vrow[e];
    }
    for (int e = 0; e < Dv; ++e) o[e] /= l;
}

static int desc_ok(const oracle_attn_desc* a)
{
    if (!a || a->T < 0 || a->S < 0 || a->heads <= 0 || a->kv_heads <= 0) return 0;
    if (a->heads % a->kv_heads != 0) return 0;
    if (a->head_dim <= 0 || a->v_head_dim <= 0) return 0;
    if (a->window < 0 || a->softcap < 0.0) return 0;
    return 1;
}

/* Full output: out is [T, heads*Dv] doubles.  Returns 0 on success. */
int oracle_attention(const oracle_attn_desc* a, const float* q, const float* k,
                     const float* v, const float* bias, double* out)
{
    if (!desc_ok(a)) return 1;
    const int64_t rows = a->T * a->heads;
    int bad = 0;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)(a->S > 0 ? a->S : 1));
        char* vis = (char*)malloc((size_t)(a->S > 0 ? a->S : 1));
        if (!x || !vis) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < rows; ++r) {
                int64_t t = r / a->heads;
                int h = (int)(r % a->heads);
                attend_row(a, q, k, v, bias, t, h, x, vis,
                           out + t * (int64_t)a->heads * a->v_head_dim +
                               (int64_t)h * a->v_head_dim);
            }
        }
        free(x);
        free(vis);
    }
    return bad ? 2 : 0;
}

/* Selected rows only: for i < n, row (ts[i], hs[i]) goes to out[i*Dv ...]. */
int oracle_attention_rows(const oracle_attn_desc* a, const float* q, const float* k,
                          const float* v, const float* bias, const int64_t* ts,
                          const int32_t* hs, int64_t n, double* out)
{
    if (!desc_ok(a)) return 1;
    for (int64_t i = 0; i < n; ++i)
        if (ts[i] < 0 || ts[i] >= a->T || hs[i] < 0 || hs[i] >= a->heads) return 1;
    int bad = 0;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)(a->S > 0 ? a->S : 1));
        char* vis = (char*)malloc((size_t)(a->S > 0 ? a->S : 1));
        if (!x || !vis) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < n; ++i)
                attend_row(a, q, k, v, bias, ts[i], hs[i], x, vis,
                           out + i * (int64_t)a->v_head_dim);
        }
        free(x);
        free(vis);
    }
    return bad ? 2 : 0;
}

/*
 * ALiBi slopes, in double.
 *  BLOOM (op param `alibi: true`): with c the largest power of two <= heads,
 *    slope_i = 2^(-8 i / c) for i = 1..c, then, if heads > c,
 *    2^(-4 (2 j - 1) / c) for j = 1..heads-c.
 *  MPT (op param `alibiMax` = b): with n the smallest power of two >= heads,
 *    a_i = 2^(-b i / n) for i = 1..n; if n != heads the list is
 *    a_2, a_4, ..., a_n, a_1, a_3, ... cut to `heads` entries.
 */
int oracle_alibi_slopes(int heads, int kind, double alibi_max, double* out)
{
    if (heads <= 0 || !out) return 1;
    if (kind == ORACLE_ALIBI_BLOOM) {
        int c = 1;
        while (c * 2 <= heads) c *= 2;
        for (int i = 1; i <= c; ++i) out[i - 1] = pow(2.0, -8.0 * i / c);
        for (int j = 1; j <= heads - c; ++j)
            out[c + j - 1] = pow(2.0, -4.0 * (2.0 * j - 1.0) / c);
        return 0;
    }
    if (kind == ORACLE_ALIBI_MPT) {
        int n = 1;
        while (n < heads) n *= 2;
        double* a = (double*)malloc(sizeof(double) * (size_t)n);
        if (!a) return 2;
        for (int i = 1; i <= n; ++i) a[i - 1] = pow(2.0, -alibi_max * i / n);
        if (n == heads) {
            memcpy(out, a, sizeof(double) * (size_t)heads);
        } else {
            int w = 0;
            for (int i = 2; i <= n && w < heads; i += 2) out[w++] = a[i - 1];
            for (int i = 1; i <= n && w < heads; i += 2) out[w++] = a[i - 1];
        }
        free(a);
        return 0;
    }
    return 1;
}

/* op "cache_write": cache[offset + r, :] = values[r, :] for r < rows, in
 * place.  Rows outside [offset, offset+rows) are left alone.  Returns 0, or 1
 * when the rows would not fit. */
int oracle_cache_write(float* cache, int64_t max_rows, int64_t width,
                       const float* values, int64_t rows, int64_t offset)
{
    if (rows < 0 || width < 0 || offset < 0 || offset + rows > max_rows) return 1;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < width; ++c)
            cache[(offset + r) * width + c] = values[r * width + c];
    return 0;
}

/* Inverse frequencies of op "rope" (same page, param base = rope_theta,
 * default 10000): inv_freq[j] = base^(-2j / rotary_dim) for j < rotary_dim/2,
 * the geometric sequence of rotary position embeddings (Su et al.,
 * "RoFormer", 2021).  Returns 1 on a bad argument. */
int oracle_rope_inv_freq(int rotary_dim, double base, double* out)
{
    if (rotary_dim <= 0 || rotary_dim % 2 != 0 || !(base > 0.0)) return 1;
    for (int j = 0; j < rotary_dim / 2; ++j)
        out[j] = pow(base, -2.0 * (double)j / (double)rotary_dim);
    return 0;
}

/* op "rope": rotary position embedding of x [T, heads*head_dim].  Row t sits
 * at position (offset + t) / pos_divisor (pos_divisor is 1, or the factor of
 * a linear frequency scaling).  Pair j < rotary_dim/2 of every head turns by
 * theta = position * inv_freq[j]: channels (j, j + rotary_dim/2), or
 * (2j, 2j + 1) when interleaved, go
 *     (a, b) -> (a cos(theta) - b sin(theta), b cos(theta) + a sin(theta)),
 * with cos and sin multiplied by attention_factor; channels at or past
 * rotary_dim pass through.  Output in double.  Returns 1 on a bad argument. */
int oracle_rope(const float* x, int64_t T, int heads, int head_dim, int rotary_dim,
                int interleaved, int64_t offset, double pos_divisor,
                const double* inv_freq, double attention_factor, double* out)
{
    if (T < 0 || heads <= 0 || head_dim <= 0 || rotary_dim < 0 || rotary_dim > head_dim ||
        rotary_dim % 2 != 0 || offset < 0 || !(pos_divisor > 0.0))
        return 1;
    const int half = rotary_dim / 2;
    for (int64_t t = 0; t < T; ++t) {
        const double position = (double)(offset + t) / pos_divisor;
        for (int h = 0; h < heads; ++h) {
            const float* xr = x + (t * heads + h) * (int64_t)head_dim;
            double* orow = out + (t * heads + h) * (int64_t)head_dim;
            for (int d = rotary_dim; d < head_dim; ++d) orow[d] = xr[d];
            for (int j = 0; j < half; ++j) {
                const int ia = interleaved ? 2 * j : j;
                const int ib = interleaved ? 2 * j + 1 : j + half;
                const double theta = position * inv_freq[j];
                const double c = cos(theta) * attention_factor;
                const double s = sin(theta) * attention_factor;
                orow[ia] = (double)xr[ia] * c - (double)xr[ib] * s;
                orow[ib] = (double)xr[ib] * c + (double)xr[ia] * s;
            }
        }
    }
    return 0;
}

/*
 * Absorbed latent attention ("mla_attention" of the IR schema page,
 * $defs.op_mla_attention: heads, kv_rank, qk_nope, qk_rope, v_head_dim, the
 * up-projections k_b and v_b, scale, causal, window, sinks).  The oracle
 * computes its plain, un-absorbed definition (DeepSeek-V2's multi-head latent
 * attention, which the parameter names follow):
 *
 *   state [S, kv_rank + qk_rope]: row s = [c_s (kv_rank) | r_s (qk_rope)],
 *       the latent KV cache: the compressed latent and the shared rotary key;
 *   k_b [heads*qk_nope, kv_rank], v_b [heads*v_head_dim, kv_rank]: the
 *       up-projections as stored ([out, in]);
 *   q [T, heads*(qk_nope + qk_rope)]: per head the no-rope part, then the
 *       rotary part;
 *   key of head h at s:   [ sum_j k_b[h*qk_nope + i, j] c_s[j]  (i < qk_nope) | r_s ]
 *   value of head h at s: [ sum_j v_b[h*v_head_dim + e, j] c_s[j] (e < v_head_dim) ]
 *   out[t, h*v_head_dim + e] = the attention of q's head-h row over those keys
 *       and values: x_s = scale * q . key, visible keys as for op attention
 *       (causal, window, sinks), max-subtracted softmax, zeros when nothing is
 *       visible.
 *
 * Every head's keys and values are expanded in double first (the definition),
 * then each requested row attends to them.  The absorbed form that a GPU
 * kernel uses (queries through k_b into the latent space, one shared latent
 * head, the output through v_b) is the same sum in another order.
 */
typedef struct {
    int64_t T, S;
    int heads, kv_rank, qk_nope, qk_rope, v_head_dim;
    int causal;
    int64_t pos_offset;
    double scale;   /* resolved by the caller */
    int64_t window; /* 0 = off */
    int64_t sinks;  /* 0 = none */
} oracle_mla_desc;

static int mla_desc_ok(const oracle_mla_desc* a)
{
    if (!a || a->T < 0 || a->S < 0 || a->heads <= 0 || a->kv_rank <= 0 || a->qk_nope < 0 ||
        a->qk_rope < 0 || a->qk_nope + a->qk_rope <= 0 || a->v_head_dim <= 0)
        return 0;
    if (a->window < 0 || a->sinks < 0) return 0;
    return 1;
}

/* Keys and values of head h for every s: kh [S, qk_nope + qk_rope],
 * vh [S, v_head_dim], in double. */
static void mla_expand_head(const oracle_mla_desc* a, const float* state, const float* k_b,
                            const float* v_b, int h, double* kh, double* vh)
{
    const int R = a->kv_rank, N = a->qk_nope, P = a->qk_rope, Dv = a->v_head_dim;
    const int64_t W = (int64_t)R + P;
#pragma omp parallel for schedule(static)
    for (int64_t s = 0; s < a->S; ++s) {
        const float* c = state + s * W;
        double* krow = kh + s * (int64_t)(N + P);
        double* vrow = vh + s * (int64_t)Dv;
        for (int i = 0; i < N; ++i) {
            const float* w = k_b + ((int64_t)h * N + i) * R;
            double acc = 0.0;
            for (int j = 0; j < R; ++j) acc += (double)w[j] * (double)c[j];
            krow[i] = acc;
        }
        for (int i = 0; i < P; ++i) krow[N + i] = (double)c[R + i];
        for (int e = 0; e < Dv; ++e) {
            const float* w = v_b + ((int64_t)h * Dv + e) * R;
            double acc = 0.0;
            for (int j = 0; j < R; ++j) acc += (double)w[j] * (double)c[j];
            vrow[e] = acc;
        }
    }
}

/* Row t of head h against the expanded keys and values. */
static void mla_attend_row(const oracle_mla_desc* a, const float* q, const double* kh,
                           const double* vh, int64_t t, int h, double* x, char* vis, double* o)
{
    const int Dq = a->qk_nope + a->qk_rope, Dv = a->v_head_dim;
    const int64_t pos = a->pos_offset + t;
    const float* qrow = q + (t * (int64_t)a->heads + h) * Dq;
    double m = -INFINITY;
    for (int64_t s = 0; s < a->S; ++s) {
        vis[s] = (char)key_visible(a->causal, a->window, a->sinks, pos, s);
        if (!vis[s]) continue;
        const double* krow = kh + s * (int64_t)Dq;
        double dot = 0.0;
        for (int d = 0; d < Dq; ++d) dot += (double)qrow[d] * krow[d];
        x[s] = a->scale * dot;
        if (x[s] > m) m = x[s];
    }
    for (int e = 0; e < Dv; ++e) o[e] = 0.0;
    if (m == -INFINITY) return;
    double l = 0.0;
    for (int64_t s = 0; s < a->S; ++s) {
        if (!vis[s]) continue;
        const double wgt = exp(x[s] - m);
        l += wgt;
        const double* vrow = vh + s * (int64_t)Dv;
        for (int e = 0; e < Dv; ++e) o[e] += wgt * vrow[e];
    }
    for (int e = 0; e < Dv; ++e) o[e] /= l;
}

/* Selected rows: for i < n, row (ts[i], hs[i]) -> out[i * v_head_dim ...].
 * Returns 0 on success. */
int oracle_mla_attention_rows(const oracle_mla_desc* a, const float* q, const float* state,
                              const float* k_b, const float* v_b, const int64_t* ts,
                              const int32_t* hs, int64_t n, double* out)
{
    if (!mla_desc_ok(a)) return 1;
    for (int64_t i = 0; i < n; ++i)
        if (ts[i] < 0 || ts[i] >= a->T || hs[i] < 0 || hs[i] >= a->heads) return 1;
    const int Dq = a->qk_nope + a->qk_rope, Dv = a->v_head_dim;
    const size_t S1 = (size_t)(a->S > 0 ? a->S : 1);
    double* kh = (double*)malloc(sizeof(double) * S1 * (size_t)Dq);
    double* vh = (double*)malloc(sizeof(double) * S1 * (size_t)Dv);
    if (!kh || !vh) {
        free(kh);
        free(vh);
        return 2;
    }
    int bad = 0;
    for (int h = 0; h < a->heads && !bad; ++h) {
        int any = 0;
        for (int64_t i = 0; i < n && !any; ++i) any = hs[i] == h;
        if (!any) continue;
        mla_expand_head(a, state, k_b, v_b, h, kh, vh);
#pragma omp parallel
        {
            double* x = (double*)malloc(sizeof(double) * S1);
            char* vis = (char*)malloc(S1);
            if (!x || !vis) {
#pragma omp atomic write
                bad = 1;
            } else {
#pragma omp for schedule(dynamic, 1)
                for (int64_t i = 0; i < n; ++i)
                    if (hs[i] == h) mla_attend_row(a, q, kh, vh, ts[i], h, x, vis, out + i * (int64_t)Dv);
            }
            free(x);
            free(vis);
        }
    }
    free(kh);
    free(vh);
    return bad ? 2 : 0;
}

/* Full output: out [T, heads * v_head_dim] doubles.  Returns 0 on success. */
int oracle_mla_attention(const oracle_mla_desc* a, const float* q, const float* state,
                         const float* k_b, const float* v_b, double* out)
{
    if (!mla_desc_ok(a)) return 1;
    const int64_t n = a->T * a->heads;
    int64_t* ts = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    int32_t* hs = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    double* tmp = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)a->v_head_dim);
    if (!ts || !hs || !tmp) {
        free(ts);
        free(hs);
        free(tmp);
        return 2;
    }
    for (int64_t i = 0; i < n; ++i) {
        ts[i] = i / a->heads;
        hs[i] = (int32_t)(i % a->heads);
    }
    int rc = oracle_mla_attention_rows(a, q, state, k_b, v_b, ts, hs, n, tmp);
    if (rc == 0)
        for (int64_t i = 0; i < n; ++i)
            memcpy(out + (ts[i] * a->heads + hs[i]) * (int64_t)a->v_head_dim,
                   tmp + i * (int64_t)a->v_head_dim, sizeof(double) * (size_t)a->v_head_dim);
    free(ts);
    free(hs);
    free(tmp);
    return rc;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
