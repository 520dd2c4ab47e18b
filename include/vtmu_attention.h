/*
 * vtmu_attention.h -- C ABI of the GB300 (sm_103a) f32 attention library.
 *
 * Three ops of the volunteer-inference op catalog (vtmu.mpakt.dev/api/ops):
 *
 *   attention    op "attention": scaled dot-product attention with
 *                grouped-query heads on flat row-major f32 tensors
 *                  q    [T, heads*headDim]
 *                  k    [S, kvHeads*headDim]
 *                  v    [S, kvHeads*vHeadDim]
 *                  bias [T, S] or [heads, T, S]   (optional, additive)
 *                  out  [T, heads*vHeadDim]
 *                Query head h reads KV head h / (heads/kvHeads).  Query row
 *                t sits at absolute position p = posOffset + t and key row s
 *                at position s.  For each visible key (see `window` and
 *                `causal` below) the score is
 *                  x = scale * q.k ; x = softcap*tanh(x/softcap) (if set) ;
 *                  x += slope_h * (s - p) (ALiBi) ; x += bias ;
 *                and the output row is the max-subtracted softmax of the
 *                scores applied to the value rows.  A row with no visible key
 *                (or only keys whose score is -inf) is written as zeros.
 *                The score matrix never leaves the chip.
 *   cache_write  op "cache_write": cache[offset + r, :] = values[r, :] for
 *                r < rows, in place (the op mutates its first input).
 *   rope         op "rope": rotary position embedding of [T, heads*headDim]
 *                (vtmu_rope), also fused into a decode step
 *                (vtmu_decode_step_rope).
 *
 * Conventions shared by every entry point
 *  - Tensor pointers are DEVICE pointers (cudaMalloc / PyTorch allocations)
 *    owned by the caller; the library never allocates or frees, and never
 *    synchronises except in vtmu_decode_step_host and
 *    vtmu_mla_decode_step_host (host buffers), which wait for their stream.
 *    Work is enqueued on `stream` and the call returns at once.  Results are
 *    visible once the stream reaches that point.
 *  - Host pointers are marked HOST and are used during the call only.
 *  - Every check runs on the host before any launch.  A failed check
 *    launches nothing and returns a status; vtmu_last_error() then names the
 *    offending parameter or feature (the catalog, likewise, names the missing
 *    feature when it refuses a graph).
 *  - A CUDA launch error returns VTMU_ERR_CUDA with the CUDA error string.
 */
#ifndef VTMU_ATTENTION_H
#define VTMU_ATTENTION_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VTMU_API __attribute__((visibility("default")))
#else
#define VTMU_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cudaStream_t;

typedef enum vtmu_status {
    VTMU_OK = 0,
    VTMU_ERR_INVALID = 1,     /* null pointer, bad shape or parameter */
    VTMU_ERR_UNSUPPORTED = 2, /* a valid request this build does not serve */
    VTMU_ERR_RANGE = 3,       /* an offset or position outside its range */
    VTMU_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
    VTMU_ERR_CUDA = 5         /* a CUDA runtime error at launch */
} vtmu_status;

/* ALiBi slope source (op "attention" params alibi / alibiMax / alibiSlopes). */
typedef enum vtmu_alibi_kind {
    VTMU_ALIBI_NONE = 0,
    VTMU_ALIBI_BLOOM = 1,  /* alibi: true -> BLOOM geometric slopes */
    VTMU_ALIBI_MPT = 2,    /* alibiMax: b -> MPT slopes with alibi_bias_max b */
    VTMU_ALIBI_SLOPES = 3  /* alibiSlopes: explicit per-head slopes (HOST) */
} vtmu_alibi_kind;

/* Shape of the optional fourth input of op "attention". */
typedef enum vtmu_bias_kind {
    VTMU_BIAS_NONE = 0,
    VTMU_BIAS_TS = 1,  /* bias [T, S], shared by every head */
    VTMU_BIAS_HTS = 2  /* bias [heads, T, S] */
} vtmu_bias_kind;

/* Kernel choice.  AUTO takes the tensor-core decode kernel for T >= 2 when
 * it covers the call (T * group size <= 16, headDim == vHeadDim == 128,
 * no softcap, ALiBi or bias; 16-byte aligned q, k, v, out), else the split-KV
 * decode kernel for 1 <= T <= 8
 * (when its shape table covers headDim/vHeadDim/group size), the tcgen05 3xTF32
 * prefill for T >= 64 when it covers the shape (headDim == vHeadDim in
 * {32, 64, 96, 128, 256}, or headDim 192 with vHeadDim 128; 16-byte aligned q
 * and out), and the FFMA prefill otherwise.  The others force one kernel,
 * for tests and measurement. */
typedef enum vtmu_kernel {
    VTMU_KERNEL_AUTO = 0,
    VTMU_KERNEL_DECODE = 1,        /* 1 <= T <= 16: T query rows against a cache */
    VTMU_KERNEL_PREFILL_FFMA = 2,  /* tiled online-softmax kernel on FP32 FMA */
    VTMU_KERNEL_PREFILL_TF32X3 = 3, /* tcgen05 3xTF32 tensor-core prefill */
    VTMU_KERNEL_DECODE_TF32X3 = 4   /* T query rows against a cache, T * group
                                       size <= 16, headDim 128: scores and
                                       P.V on the tensor cores (3xTF32) */
} vtmu_kernel;

/*
 * Parameters of one attention call.  Fill with vtmu_attention_params_init()
 * (which writes the op's defaults), then set fields.  Names follow the op
 * catalog: heads, headDim, kvHeads, vHeadDim, causal, posOffset, scale,
 * softcap, window, alibi/alibiMax/alibiSlopes.
 */
typedef struct vtmu_attention_params {
    int64_t T;            /* query rows (0 is a no-op) */
    int64_t S;            /* key/value rows (0: every output row is zero) */
    int32_t heads;        /* query heads, > 0 */
    int32_t kv_heads;     /* KV heads; 0 means "= heads"; heads % kv_heads == 0 */
    int32_t head_dim;     /* query/key width per head, 1..256 */
    int32_t v_head_dim;   /* value width per head; 0 means "= head_dim"; 1..256 */
    int32_t causal;       /* default 1 */
    int32_t has_scale;    /* 0: scale = 1/sqrt(head_dim) */
    float scale;          /* used when has_scale != 0; must be finite */
    float softcap;        /* 0 = off; > 0: x = softcap * tanh(x / softcap) */
    int64_t pos_offset;   /* absolute position of query row 0, >= 0 */
    int64_t window;       /* 0 = off; causal: p - window < s <= p;
                             non-causal: |p - s| <= window */
    int32_t alibi;        /* vtmu_alibi_kind */
    float alibi_max;      /* MPT alibi_bias_max (> 0) for VTMU_ALIBI_MPT */
    const float* alibi_slopes; /* HOST [heads], for VTMU_ALIBI_SLOPES */
    int32_t bias_kind;    /* vtmu_bias_kind; bias pointer must agree */
    int32_t kernel;       /* vtmu_kernel */
    int32_t decode_splits; /* decode kernels: KV splits per KV head, 0 = auto */
    int64_t sinks;        /* attention sinks (the IR page's op_attention.sinks, not a
                             param of the op page): with a window, keys s < sinks
                             stay visible (causality still applies); 0 = none */
} vtmu_attention_params;

/* Writes the op's defaults: causal = 1, everything else 0 / off / AUTO. */
VTMU_API void vtmu_attention_params_init(vtmu_attention_params* p);

/*
 * Scratch bytes that vtmu_attention needs for `p` (0 for the FFMA prefill).
 * The decode kernel keeps per-split partial results (running max, sum and
 * unnormalised output) and one arrival counter per KV head there; the
 * tensor-core prefill keeps the tf32 hi/lo halves of K and of V transposed
 * (4 * S * kvHeads * headDim floats).
 * Returns VTMU_ERR_INVALID / VTMU_ERR_UNSUPPORTED for parameters that
 * vtmu_attention would refuse.
 */
VTMU_API vtmu_status vtmu_attention_workspace_size(const vtmu_attention_params* p, size_t* bytes);

/*
 * op "attention" (vtmu.mpakt.dev/api/ops).  q, k, v, out: DEVICE, layouts
 * above, 4-byte aligned.  bias: DEVICE or NULL, must be non-NULL exactly when
 * p->bias_kind != VTMU_BIAS_NONE.  out must not overlap an input.
 * workspace: DEVICE, at least vtmu_attention_workspace_size() bytes (may be
 * NULL when that is 0), 256-byte aligned.  Its first 64 KiB hold the decode
 * kernel's arrival counters and must be ZERO before the first decode call;
 * every call leaves them zero again and no kernel writes scratch there, so a
 * workspace is reused across calls of any kind and shape without clearing.
 * Calls that share a workspace must not overlap on the GPU (use one
 * workspace per concurrent stream).
 *
 * Errors: VTMU_ERR_INVALID (null pointer, T/S < 0, heads <= 0, heads not a
 * multiple of kv_heads, window < 0, softcap < 0 or not finite, scale not
 * finite, bias pointer and bias_kind disagree, alibi slopes missing, out
 * aliasing an input, T outside 1..16 with VTMU_KERNEL_DECODE), VTMU_ERR_RANGE
 * (pos_offset < 0), VTMU_ERR_UNSUPPORTED (head_dim or v_head_dim outside
 * 1..256, a forced kernel that does not cover the shape),
 * VTMU_ERR_WORKSPACE, VTMU_ERR_CUDA.
 */
VTMU_API vtmu_status vtmu_attention(const float* q, const float* k, const float* v,
                           const float* bias, float* out,
                           const vtmu_attention_params* p, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/*
 * A decode step of a KV-cached model: op "cache_write" of k_new into k_cache
 * and of v_new into v_cache at row `offset`, then op "attention" of q over the
 * updated caches (vtmu.mpakt.dev/api/ops: a whole decode step is meant to run
 * without leaving the worker).  The result equals vtmu_cache_write(k_cache,
 * ...), vtmu_cache_write(v_cache, ...), vtmu_attention(q, k_cache, v_cache,
 * bias, out, p, ...) in that order; when the decode kernel covers the call
 * (1 <= T <= 8 under AUTO, same shape table as VTMU_KERNEL_DECODE) all three run as one
 * launch: the CTA that reads a new row takes it from k_new / v_new and writes
 * it to the cache itself.
 *   k_cache [max_rows, kvHeads*headDim], v_cache [max_rows, kvHeads*vHeadDim]:
 *     DEVICE, updated in place; the attention reads their first p->S rows
 *     (p->S <= max_rows).
 *   k_new [new_rows, kvHeads*headDim], v_new [new_rows, kvHeads*vHeadDim]:
 *     DEVICE, must not overlap a cache; new_rows == 0 skips the writes.
 *   q, bias, out, p, workspace: as for vtmu_attention.
 * Errors: those of vtmu_attention, plus VTMU_ERR_RANGE (offset < 0 or
 * offset + new_rows > max_rows), VTMU_ERR_INVALID (p->S > max_rows, NULL or
 * overlapping cache / new-row buffers).
 */
VTMU_API vtmu_status vtmu_decode_step(float* k_cache, float* v_cache, int64_t max_rows,
                                      const float* k_new, const float* v_new, int64_t new_rows,
                                      int64_t offset, const float* q, const float* bias, float* out,
                                      const vtmu_attention_params* p, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream);

/*
 * Workspace bytes of vtmu_decode_step_host for these params and new_rows:
 * the workspace vtmu_attention needs for `p`, then device staging areas for
 * q, k_new, v_new, the bias and out, each starting on a 256-byte boundary.
 * Errors: those of vtmu_attention_workspace_size, VTMU_ERR_INVALID
 * (new_rows < 0).
 */
VTMU_API vtmu_status vtmu_decode_step_host_workspace_size(const vtmu_attention_params* p,
                                                          int64_t new_rows, size_t* bytes);

/*
 * A decode step whose inputs and output live in HOST memory: the call a
 * worker makes when a step's q and new K/V rows arrive over the network and
 * its output row goes back (vtmu.mpakt.dev/api/ops: the worker runs the
 * step and returns the result).  On `stream` it copies q_host, k_new_host,
 * v_new_host and bias_host into the staging areas of `workspace`, runs
 * vtmu_decode_step on those copies, copies out back to out_host and WAITS for
 * the stream: unlike every other entry point it returns only when out_host
 * holds the result (or an error occurred).  When the step runs on a decode
 * kernel (VTMU_KERNEL_DECODE or VTMU_KERNEL_DECODE_TF32X3), no bias is given,
 * and q_host, k_new_host, v_new_host and out_host are page-locked buffers the
 * device can address (cudaHostAlloc / cudaMallocHost / cudaHostRegister,
 * e.g. a pinned PyTorch tensor) that are, like the caches, 16-byte aligned,
 * the kernel reads q and the new rows and writes the output row in place over
 * the host link, with no staging copy (same result, bit for bit).
 *   k_cache, v_cache, max_rows, new_rows, offset, p: as for vtmu_decode_step
 *     (the caches are DEVICE memory, updated in place).
 *   q_host [T, heads*headDim], k_new_host / v_new_host [new_rows, kvHeads*
 *     headDim / vHeadDim], bias_host (as bias_kind says, or NULL), out_host
 *     [T, heads*vHeadDim]: HOST, row-major f32.  Page-locked memory lets the
 *     copies run asynchronously; pageable memory works with staged copies.
 *   workspace: DEVICE, at least vtmu_decode_step_host_workspace_size bytes,
 *     256-byte aligned; its first 64 KiB follow vtmu_attention's rule.
 * Errors: those of vtmu_decode_step, VTMU_ERR_WORKSPACE (workspace too
 * small), VTMU_ERR_INVALID (a host pointer NULL where data is needed),
 * VTMU_ERR_CUDA (a copy or the wait failed).  Checks run before any copy.
 */
VTMU_API vtmu_status vtmu_decode_step_host(float* k_cache, float* v_cache, int64_t max_rows,
                                           const float* k_new_host, const float* v_new_host,
                                           int64_t new_rows, int64_t offset, const float* q_host,
                                           const float* bias_host, float* out_host,
                                           const vtmu_attention_params* p, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream);

/*
 * op "cache_write" (vtmu.mpakt.dev/api/ops): cache[offset + r, :] =
 * values[r, :] for 0 <= r < rows, bit-exact, in place; rows outside
 * [offset, offset + rows) are untouched.  cache [max_rows, width] and values
 * [rows, width]: DEVICE, row-major f32, must not overlap.  rows == 0 is a
 * no-op.  Errors: VTMU_ERR_INVALID (null pointer with rows > 0, negative
 * sizes), VTMU_ERR_RANGE (offset < 0 or offset + rows > max_rows),
 * VTMU_ERR_CUDA.
 */
VTMU_API vtmu_status vtmu_cache_write(float* cache, int64_t max_rows, int64_t width,
                             const float* values, int64_t rows, int64_t offset,
                             cudaStream_t stream);

/*
 * Decode without allocation.  The op catalog has no counterpart: this entry
 * point exists for callers that cannot allocate device memory themselves --
 * a plug-in whose host process owns all device memory through its own pool,
 * or a latency-critical decode loop that must not call cudaMalloc (it can
 * synchronise the device).  It computes exactly what vtmu_attention does
 * with VTMU_KERNEL_DECODE (same arguments, same checks, T must be 1, the
 * decode kernel's shape table must cover the call and p->kernel must be
 * VTMU_KERNEL_AUTO or VTMU_KERNEL_DECODE) but takes no workspace: the
 * kernel's scratch (split partials and arrival counters) lives in a static
 * device array of VTMU_NOALLOC_SCRATCH_BYTES that every GPU loading this
 * library holds until the process exits.  The call itself allocates nothing.
 *  - Limit: a call whose decode scratch (vtmu_attention_workspace_size with
 *    kernel = VTMU_KERNEL_DECODE) exceeds VTMU_NOALLOC_SCRATCH_BYTES is
 *    refused with VTMU_ERR_WORKSPACE.  With 16384 or more visible keys at
 *    vHeadDim 128 the array holds 62 virtual heads: up to 62 query heads
 *    when heads/kvHeads >= 2, up to 31 when heads == kvHeads (the kernel
 *    pads each KV head to two virtual heads there).
 *  - Every call looks up the array's device address (cudaGetSymbolAddress,
 *    with the caller's device current), so the address stays right after
 *    cudaDeviceReset or under another context of the same device.  The first
 *    call in a context may load the library's device code: make it before
 *    any stream capture.
 *  - All calls share the one array.  Every host-side check runs before the
 *    array is touched; then its arrival counters are cleared on `stream`
 *    and the kernel launched.  Calls whose GPU work overlaps (several streams
 *    or host threads at once) race on the array: serialise them.
 */
#define VTMU_NOALLOC_SCRATCH_BYTES (8u << 20)
VTMU_API vtmu_status vtmu_attention_decode_noalloc(const float* q, const float* k, const float* v,
                                                   const float* bias, float* out,
                                                   const vtmu_attention_params* p,
                                                   cudaStream_t stream);

/* Frequency scaling of op "rope" (param scaling, config.json's rope_scaling).
 * Linear divides every position by the factor.  Other schemes (llama3, yarn,
 * longrope, dynamic) are served through explicit inverse frequencies and an
 * attention factor computed by the caller; requesting them by kind is
 * refused with "rope.scaling" named. */
typedef enum vtmu_rope_scaling {
    VTMU_ROPE_SCALING_NONE = 0,
    VTMU_ROPE_SCALING_LINEAR = 1
} vtmu_rope_scaling;

/*
 * Parameters of op "rope" (vtmu.mpakt.dev/api/ops): rotary position
 * embedding over x [T, heads*headDim].  Row t sits at position offset + t
 * (divided by scaling_factor with linear scaling).  Pair j < rotary_dim/2
 * of every head turns by theta = position * inv_freq[j]: channels
 * (j, j + rotary_dim/2) (Llama, Qwen, Mistral, NeoX) or, interleaved,
 * (2j, 2j + 1) (GPT-J), as (a, b) -> (a cos - b sin, b cos + a sin), with
 * cos and sin multiplied by attention_factor; channels at or past rotary_dim
 * pass through.  inv_freq[j] = base^(-2j / rotary_dim) unless given.
 * Fill with vtmu_rope_params_init(), then set fields.
 */
typedef struct vtmu_rope_params {
    int32_t head_dim;        /* per-head width, 1..4096 */
    int32_t rotary_dim;      /* 0 means head_dim; even, <= head_dim, <= 256 */
    int32_t interleaved;     /* 0: half-split pairs; 1: (2j, 2j + 1) */
    int32_t scaling;         /* vtmu_rope_scaling */
    float base;              /* rope_theta; 0 means 10000; > 0 */
    float scaling_factor;    /* VTMU_ROPE_SCALING_LINEAR: > 0 */
    float attention_factor;  /* 0 means 1; multiplies cos and sin */
    const float* inv_freq;   /* HOST [rotary_dim/2] explicit inverse frequencies, or NULL */
} vtmu_rope_params;

/* Writes the op's defaults: base 10000, rotary_dim = head_dim, half-split
 * pairs, no scaling, attention factor 1 (head_dim is left 0: set it). */
VTMU_API void vtmu_rope_params_init(vtmu_rope_params* r);

/*
 * op "rope": out = rope(x) for x, out [T, heads*head_dim], DEVICE, row-major
 * f32, 4-byte aligned; out == x turns x in place, otherwise they must not
 * overlap.  offset (param offset, >= 0): position of row 0.
 * Errors: VTMU_ERR_INVALID (NULL pointer with T > 0, T < 0, heads <= 0,
 * head_dim outside 1..4096, rotary_dim odd or above head_dim, base, factor
 * or attention factor not finite / not positive where required, inv_freq
 * not finite, partial overlap of x and out), VTMU_ERR_UNSUPPORTED
 * (rotary_dim above 256, a scaling kind other than none / linear:
 * "rope.scaling"), VTMU_ERR_RANGE (offset < 0), VTMU_ERR_CUDA.
 */
VTMU_API vtmu_status vtmu_rope(const float* x, float* out, int64_t T, int32_t heads, int64_t offset,
                               const vtmu_rope_params* r, cudaStream_t stream);

/*
 * A decode step with the rotary embedding fused in: what op "rope" on q
 * (row t at position p->pos_offset + t) and on k_new (row i at position
 * offset + i), then vtmu_decode_step with the turned q and k_new compute --
 * the caches receive turned keys, q is left as given -- in ONE launch of a
 * decode kernel (vtmu.mpakt.dev/api/ops: a whole decode step is meant to stay
 * on the worker).  Arguments as for vtmu_decode_step, plus `rope` with
 * rope->head_dim == p->head_dim.  Only the fused form is offered: the call
 * needs either a shape the tensor-core decode covers (VTMU_KERNEL_DECODE_TF32X3
 * chosen or picked by AUTO: T x group <= 16, headDim 128, with 16-byte
 * aligned q, caches, k_new, v_new and out), or T == 1 and a shape the CUDA-core
 * decode covers (same table and 16-byte alignment as VTMU_KERNEL_DECODE);
 * anything else, T == 0 included, is refused with VTMU_ERR_UNSUPPORTED --
 * compose vtmu_rope and vtmu_decode_step there.
 * Errors: those of vtmu_decode_step and vtmu_rope, VTMU_ERR_UNSUPPORTED.
 */
VTMU_API vtmu_status vtmu_decode_step_rope(float* k_cache, float* v_cache, int64_t max_rows,
                                           const float* k_new, const float* v_new, int64_t new_rows,
                                           int64_t offset, const float* q, const float* bias, float* out,
                                           const vtmu_attention_params* p, const vtmu_rope_params* rope,
                                           void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Absorbed latent attention: mla_attention of the IR schema page
 * (graph_ir_schema.h, $defs.op_mla_attention: heads, kv_rank, qk_nope,
 * qk_rope, v_head_dim, the up-projections k_b and v_b, scale, causal,
 * window, sinks), read as DeepSeek-V2's multi-head latent attention.
 *   state [max_rows, kv_rank + qk_rope]: latent KV cache; row s is
 *       [c_s (kv_rank) | r_s (qk_rope)], the compressed latent and the
 *       rotary key shared by every head (the first S rows are read)
 *   q     [T, heads*(qk_nope + qk_rope)]: per head the no-rope part, then
 *       the rotary part (already turned)
 *   k_b   [heads*qk_nope, kv_rank] (may be NULL when qk_nope is 0), v_b
 *       [heads*v_head_dim, kv_rank]: the
 *       up-projections as a checkpoint stores them ([out, in])
 *   out   [T, heads*v_head_dim]
 * Head h's key at s is [k_b_h c_s | r_s] and its value v_b_h c_s (k_b_h,
 * v_b_h: head h's rows); query row t at position pos_offset + t scores
 * x = scale * q . key over the visible keys (causal, window and sinks as for
 * op "attention"), and the output is the max-subtracted softmax of the scores
 * applied to the values (zeros when no key is visible).  The kernels compute
 * it in the absorbed order: every head's query is taken through k_b_h into
 * the latent space, so all heads read the same 576-wide cache rows once, and
 * the weighted latent is taken through v_b_h at the end.
 * This build serves kv_rank 512 with qk_rope 64 (DeepSeek-V2 and -V3),
 * qk_nope 0..512, v_head_dim 1..4096 and T * heads <= 65536 (the decode
 * form: it reads the cache once per 32 query rows x heads); other widths are
 * refused with VTMU_ERR_UNSUPPORTED.
 */
typedef struct vtmu_mla_params {
    int64_t T;            /* query rows (0 is a no-op) */
    int64_t S;            /* cache rows the attention reads */
    int32_t heads;        /* > 0 */
    int32_t kv_rank;      /* latent width (params_init: 512) */
    int32_t qk_nope;      /* no-rope query/key width per head */
    int32_t qk_rope;      /* rotary width, shared by the heads (params_init: 64) */
    int32_t v_head_dim;   /* value width per head, > 0 */
    int32_t causal;       /* default 1 */
    int32_t has_scale;    /* 0: scale = 1/sqrt(qk_nope + qk_rope) */
    float scale;          /* used when has_scale != 0; must be finite */
    int64_t pos_offset;   /* absolute position of query row 0, >= 0 */
    int64_t window;       /* 0 = off; as for op "attention" */
    int64_t sinks;        /* with a window: keys s < sinks stay visible */
    int32_t kernel;       /* 0 (auto): the CUDA-core kernel, the faster of the
                             two on the decode shapes measured; 1: the CUDA-core
                             kernel; 2: scores on the tensor cores (3xTF32),
                             values on the CUDA cores */
} vtmu_mla_params;

/* Writes the defaults: causal = 1, kv_rank 512, qk_rope 64, the rest 0. */
VTMU_API void vtmu_mla_params_init(vtmu_mla_params* p);

/* Scratch bytes vtmu_mla_attention / vtmu_mla_decode_step need for `p` (the
 * absorbed queries and the split partials), an upper bound over devices.
 * Errors: those of vtmu_mla_attention's parameter checks. */
VTMU_API vtmu_status vtmu_mla_workspace_size(const vtmu_mla_params* p, size_t* bytes);

/*
 * mla_attention (IR schema page, $defs.op_mla_attention).  q, out: DEVICE,
 * 4-byte aligned; state, k_b, v_b: DEVICE, 16-byte aligned; out must not
 * overlap an input.  workspace: DEVICE, at least vtmu_mla_workspace_size()
 * bytes, 256-byte aligned, no initial contents needed; calls that share a
 * workspace must not overlap on the GPU.  Four launches on `stream`.
 * Errors: VTMU_ERR_INVALID (null or misaligned pointer, negative sizes or
 * window/sinks, scale not finite, out overlapping an input), VTMU_ERR_RANGE
 * (pos_offset < 0), VTMU_ERR_UNSUPPORTED (kv_rank/qk_rope other than 512/64,
 * qk_nope above 512, v_head_dim above 4096, T * heads above 65536, S at or
 * above 2^31), VTMU_ERR_WORKSPACE, VTMU_ERR_CUDA.
 */
VTMU_API vtmu_status vtmu_mla_attention(const float* q, const float* state, const float* k_b,
                                        const float* v_b, float* out, const vtmu_mla_params* p,
                                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * A decode step of a latent-attention model: op "cache_write" of state_new
 * [new_rows, kv_rank + qk_rope] into state at row `offset`, then
 * vtmu_mla_attention over the updated cache (its first p->S rows).  The
 * rows are written by the first of the four launches, before any read.
 * state [max_rows, kv_rank + qk_rope] and state_new: DEVICE, 16-byte
 * aligned, not overlapping.  Errors: those of vtmu_mla_attention, plus
 * VTMU_ERR_RANGE (offset < 0 or offset + new_rows > max_rows) and
 * VTMU_ERR_INVALID (p->S > max_rows, NULL or overlapping buffers).
 */
VTMU_API vtmu_status vtmu_mla_decode_step(float* state, int64_t max_rows, const float* state_new,
                                          int64_t new_rows, int64_t offset, const float* q,
                                          const float* k_b, const float* v_b, float* out,
                                          const vtmu_mla_params* p, void* workspace,
                                          size_t workspace_bytes, cudaStream_t stream);

/*
 * Workspace bytes of vtmu_mla_decode_step_host for these params and new_rows:
 * the latent attention's workspace followed by staging areas for q, the new
 * cache rows and the output.  Errors: those of the parameter checks,
 * VTMU_ERR_INVALID (new_rows < 0, bytes NULL).
 */
VTMU_API vtmu_status vtmu_mla_decode_step_host_workspace_size(const vtmu_mla_params* p, int64_t new_rows,
                                                              size_t* bytes);

/*
 * vtmu_mla_decode_step with q, the new latent rows and the output in HOST
 * memory (as vtmu_decode_step_host is to vtmu_decode_step): q_host [T,
 * heads*(qk_nope + qk_rope)], state_new_host [new_rows, kv_rank + qk_rope],
 * out_host [T, heads*v_head_dim], row-major f32; state, k_b, v_b: DEVICE as
 * for vtmu_mla_decode_step.  Page-locked buffers the device can address
 * (state_new_host also 16-byte aligned) are read and written in place by the
 * launches (the absorb launch reads q and copies the new rows, the projection
 * writes the output row); other buffers are copied through the staging areas
 * of `workspace` (DEVICE, at least vtmu_mla_decode_step_host_workspace_size
 * bytes, 256-byte aligned).  The call WAITS for `stream` and returns when
 * out_host holds the result.  Every check runs before any copy.  Errors:
 * those of vtmu_mla_decode_step, VTMU_ERR_WORKSPACE, VTMU_ERR_INVALID (a host
 * buffer NULL where data is needed), VTMU_ERR_CUDA (a copy or the wait).
 */
VTMU_API vtmu_status vtmu_mla_decode_step_host(float* state, int64_t max_rows, const float* state_new_host,
                                               int64_t new_rows, int64_t offset, const float* q_host,
                                               const float* k_b, const float* v_b, float* out_host,
                                               const vtmu_mla_params* p, void* workspace,
                                               size_t workspace_bytes, cudaStream_t stream);

/*
 * Kernel-side failures.  Every wait inside a kernel (TMA stage arrival,
 * stage release) gives up after one second instead of hanging the GPU; the
 * kernel then sets a bit in a device flag, abandons its output and returns.
 * This call synchronises the current device, stores the OR of the flags of
 * every kernel in *flags (0: no wait gave up since the last call) and clears
 * them.  Decode bits: 1 = a consumer gave up on a loaded stage, 2 = the
 * producer gave up on a free stage, 4 = the producer gave up draining its
 * copies; tensor-core prefill bits: 0x100 stage load, 0x200 free stage,
 * 0x400 drain, 0x800 query load, 0x1000 score tile, 0x2000 probabilities,
 * 0x4000 P.V product; latent attention bits: 0x10000 stage load, 0x20000
 * free stage, 0x40000 drain (CUDA-core kernel), 0x100000 ring item,
 * 0x200000 free slot, 0x400000 split item, 0x800000 score tile, 0x1000000
 * free score buffer, 0x2000000 drain (tensor-core kernel); tensor-core
 * decode bits: 0x4000000 ring item or query tiles, 0x8000000 free slot,
 * 0x10000000 split item, 0x20000000 score tile, 0x40000000 free score
 * buffer, 0x80000000 drain.  Errors: VTMU_ERR_INVALID (NULL flags), VTMU_ERR_CUDA.
 */
VTMU_API vtmu_status vtmu_device_error(unsigned int* flags);

/* Space-separated optional features this build implements, named as the op
 * catalog's feature table names them.  rope.scaling is not listed: of the
 * schemes it covers only linear scaling, explicit inverse frequencies and
 * the attention factor are served. */
VTMU_API const char* vtmu_features(void);

/* Message of the last failed call on this host thread ("" after success). */
VTMU_API const char* vtmu_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* VTMU_ATTENTION_H */
