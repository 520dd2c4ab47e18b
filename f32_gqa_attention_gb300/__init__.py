"""Python binding of the GB300 f32 attention library (``libvtmu.so``).

Argument marshalling only: every step of the ops runs in the library's CUDA
kernels.  The binding exposes the C ABI of ``include/vtmu_attention.h`` under
the same names (``vtmu_attention``, ``vtmu_cache_write``, ...) plus two
conveniences for PyTorch CUDA tensors, ``attention`` and ``cache_write``,
whose keyword names follow the op catalog (vtmu.mpakt.dev/api/ops, ops
"attention" and "cache_write").  PyTorch only provides device memory and
streams.

There is no fallback: if ``libvtmu.so`` is not built, loading raises.
Build it with ``python -m f32_gqa_attention_gb300._build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libvtmu.so")

VTMU_OK = 0
VTMU_ERR_INVALID = 1
VTMU_ERR_UNSUPPORTED = 2
VTMU_ERR_RANGE = 3
VTMU_ERR_WORKSPACE = 4
VTMU_ERR_CUDA = 5

VTMU_ALIBI_NONE, VTMU_ALIBI_BLOOM, VTMU_ALIBI_MPT, VTMU_ALIBI_SLOPES = 0, 1, 2, 3
VTMU_BIAS_NONE, VTMU_BIAS_TS, VTMU_BIAS_HTS = 0, 1, 2
VTMU_KERNEL_AUTO, VTMU_KERNEL_DECODE, VTMU_KERNEL_PREFILL_FFMA, VTMU_KERNEL_PREFILL_TF32X3 = 0, 1, 2, 3
VTMU_KERNEL_DECODE_TF32X3 = 4

EXPORTED = ("vtmu_attention_params_init", "vtmu_attention_workspace_size", "vtmu_attention",
            "vtmu_cache_write", "vtmu_features", "vtmu_last_error", "vtmu_attention_decode_noalloc",
            "vtmu_device_error", "vtmu_decode_step", "vtmu_decode_step_host_workspace_size",
            "vtmu_decode_step_host", "vtmu_rope_params_init", "vtmu_rope", "vtmu_decode_step_rope",
            "vtmu_mla_params_init", "vtmu_mla_workspace_size", "vtmu_mla_attention", "vtmu_mla_decode_step",
            "vtmu_mla_decode_step_host_workspace_size", "vtmu_mla_decode_step_host")
NOALLOC_SCRATCH_BYTES = 8 << 20  # VTMU_NOALLOC_SCRATCH_BYTES


class VtmuError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"vtmu status {status}: {message}")
        self.status = status


class vtmu_attention_params(ctypes.Structure):
    """Mirror of ``vtmu_attention_params`` (include/vtmu_attention.h)."""
    _fields_ = [
        ("T", ctypes.c_int64),
        ("S", ctypes.c_int64),
        ("heads", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("v_head_dim", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("has_scale", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("softcap", ctypes.c_float),
        ("pos_offset", ctypes.c_int64),
        ("window", ctypes.c_int64),
        ("alibi", ctypes.c_int32),
        ("alibi_max", ctypes.c_float),
        ("alibi_slopes", ctypes.POINTER(ctypes.c_float)),
        ("bias_kind", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("decode_splits", ctypes.c_int32),
        ("sinks", ctypes.c_int64),
    ]


VTMU_ROPE_SCALING_NONE, VTMU_ROPE_SCALING_LINEAR = 0, 1


class vtmu_rope_params(ctypes.Structure):
    """Mirror of ``vtmu_rope_params`` (include/vtmu_attention.h)."""
    _fields_ = [
        ("head_dim", ctypes.c_int32),
        ("rotary_dim", ctypes.c_int32),
        ("interleaved", ctypes.c_int32),
        ("scaling", ctypes.c_int32),
        ("base", ctypes.c_float),
        ("scaling_factor", ctypes.c_float),
        ("attention_factor", ctypes.c_float),
        ("inv_freq", ctypes.POINTER(ctypes.c_float)),
    ]


class vtmu_mla_params(ctypes.Structure):
    """Mirror of ``vtmu_mla_params`` (include/vtmu_attention.h)."""
    _fields_ = [
        ("T", ctypes.c_int64),
        ("S", ctypes.c_int64),
        ("heads", ctypes.c_int32),
        ("kv_rank", ctypes.c_int32),
        ("qk_nope", ctypes.c_int32),
        ("qk_rope", ctypes.c_int32),
        ("v_head_dim", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("has_scale", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("pos_offset", ctypes.c_int64),
        ("window", ctypes.c_int64),
        ("sinks", ctypes.c_int64),
        ("kernel", ctypes.c_int32),
    ]


MLA_KERNEL_AUTO, MLA_KERNEL_CUDA_CORES, MLA_KERNEL_TENSOR_CORES = 0, 1, 2

_lib = None
_lib_lock = threading.Lock()


def load_library():
    """Load libvtmu.so (raises if it has not been built)."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run `python -m f32_gqa_attention_gb300._build`")
        lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(vtmu_attention_params)
        vp = ctypes.c_void_p
        lib.vtmu_attention_params_init.argtypes = [P]
        lib.vtmu_attention_params_init.restype = None
        lib.vtmu_attention_workspace_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
        lib.vtmu_attention_workspace_size.restype = ctypes.c_int
        lib.vtmu_attention.argtypes = [vp, vp, vp, vp, vp, P, vp, ctypes.c_size_t, vp]
        lib.vtmu_attention.restype = ctypes.c_int
        lib.vtmu_cache_write.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, vp, ctypes.c_int64,
                                         ctypes.c_int64, vp]
        lib.vtmu_cache_write.restype = ctypes.c_int
        lib.vtmu_features.argtypes = []
        lib.vtmu_features.restype = ctypes.c_char_p
        lib.vtmu_last_error.argtypes = []
        lib.vtmu_last_error.restype = ctypes.c_char_p
        lib.vtmu_decode_step.argtypes = [vp, vp, ctypes.c_int64, vp, vp, ctypes.c_int64, ctypes.c_int64,
                                         vp, vp, vp, P, vp, ctypes.c_size_t, vp]
        lib.vtmu_decode_step.restype = ctypes.c_int
        lib.vtmu_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.vtmu_device_error.restype = ctypes.c_int
        lib.vtmu_attention_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, P, vp]
        lib.vtmu_attention_decode_noalloc.restype = ctypes.c_int
        R = ctypes.POINTER(vtmu_rope_params)
        lib.vtmu_rope_params_init.argtypes = [R]
        lib.vtmu_rope_params_init.restype = None
        lib.vtmu_rope.argtypes = [vp, vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, R, vp]
        lib.vtmu_rope.restype = ctypes.c_int
        lib.vtmu_decode_step_rope.argtypes = [vp, vp, ctypes.c_int64, vp, vp, ctypes.c_int64, ctypes.c_int64,
                                              vp, vp, vp, P, R, vp, ctypes.c_size_t, vp]
        lib.vtmu_decode_step_rope.restype = ctypes.c_int
        lib.vtmu_decode_step_host_workspace_size.argtypes = [P, ctypes.c_int64, ctypes.POINTER(ctypes.c_size_t)]
        lib.vtmu_decode_step_host_workspace_size.restype = ctypes.c_int
        lib.vtmu_decode_step_host.argtypes = [vp, vp, ctypes.c_int64, vp, vp, ctypes.c_int64, ctypes.c_int64,
                                              vp, vp, vp, P, vp, ctypes.c_size_t, vp]
        lib.vtmu_decode_step_host.restype = ctypes.c_int
        M = ctypes.POINTER(vtmu_mla_params)
        lib.vtmu_mla_params_init.argtypes = [M]
        lib.vtmu_mla_params_init.restype = None
        lib.vtmu_mla_workspace_size.argtypes = [M, ctypes.POINTER(ctypes.c_size_t)]
        lib.vtmu_mla_workspace_size.restype = ctypes.c_int
        lib.vtmu_mla_attention.argtypes = [vp, vp, vp, vp, vp, M, vp, ctypes.c_size_t, vp]
        lib.vtmu_mla_attention.restype = ctypes.c_int
        lib.vtmu_mla_decode_step.argtypes = [vp, ctypes.c_int64, vp, ctypes.c_int64, ctypes.c_int64, vp, vp, vp, vp,
                                             M, vp, ctypes.c_size_t, vp]
        lib.vtmu_mla_decode_step.restype = ctypes.c_int
        lib.vtmu_mla_decode_step_host_workspace_size.argtypes = [M, ctypes.c_int64, ctypes.POINTER(ctypes.c_size_t)]
        lib.vtmu_mla_decode_step_host_workspace_size.restype = ctypes.c_int
        lib.vtmu_mla_decode_step_host.argtypes = [vp, ctypes.c_int64, vp, ctypes.c_int64, ctypes.c_int64, vp, vp,
                                                  vp, vp, M, vp, ctypes.c_size_t, vp]
        lib.vtmu_mla_decode_step_host.restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int):
    if status != VTMU_OK:
        raise VtmuError(status, load_library().vtmu_last_error().decode())


def _addr(x):
    """Device address of a torch tensor, or an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _haddr(x):
    """Host address of a contiguous f32 numpy array or CPU tensor, an int, or None."""
    if x is None or isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if x.device.type != "cpu" or not x.is_contiguous() or x.element_size() != 4:
            raise ValueError("host buffer: expected a contiguous f32 CPU tensor")
        return x.data_ptr()
    if x.dtype.itemsize != 4 or x.dtype.kind != "f" or not x.flags["C_CONTIGUOUS"]:
        raise ValueError("host buffer: expected a C-contiguous float32 array")
    return x.ctypes.data


# ---------------------------------------------------------------- C ABI names
def vtmu_attention_params_init() -> vtmu_attention_params:
    p = vtmu_attention_params()
    load_library().vtmu_attention_params_init(ctypes.byref(p))
    return p


def vtmu_attention_workspace_size(p: vtmu_attention_params) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().vtmu_attention_workspace_size(ctypes.byref(p), ctypes.byref(n)))
    return int(n.value)


def vtmu_attention(q, k, v, bias, out, p: vtmu_attention_params, workspace, workspace_bytes: int,
                   stream: int = 0) -> None:
    _check(load_library().vtmu_attention(_addr(q), _addr(k), _addr(v), _addr(bias), _addr(out),
                                         ctypes.byref(p), _addr(workspace), int(workspace_bytes),
                                         stream or None))


def vtmu_decode_step(k_cache, v_cache, max_rows: int, k_new, v_new, new_rows: int, offset: int, q, bias, out,
                     p: vtmu_attention_params, workspace, workspace_bytes: int, stream: int = 0) -> None:
    _check(load_library().vtmu_decode_step(_addr(k_cache), _addr(v_cache), int(max_rows), _addr(k_new),
                                           _addr(v_new), int(new_rows), int(offset), _addr(q), _addr(bias),
                                           _addr(out), ctypes.byref(p), _addr(workspace), int(workspace_bytes),
                                           stream or None))


def vtmu_decode_step_host_workspace_size(p: vtmu_attention_params, new_rows: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().vtmu_decode_step_host_workspace_size(ctypes.byref(p), int(new_rows), ctypes.byref(n)))
    return int(n.value)


def vtmu_decode_step_host(k_cache, v_cache, max_rows: int, k_new_host, v_new_host, new_rows: int, offset: int,
                          q_host, bias_host, out_host, p: vtmu_attention_params, workspace, workspace_bytes: int,
                          stream: int = 0) -> None:
    """vtmu_decode_step with q / new rows / bias / out in host memory (numpy
    arrays or CPU tensors, f32, contiguous; pinned memory copies
    asynchronously).  Returns once out_host holds the result."""
    _check(load_library().vtmu_decode_step_host(_addr(k_cache), _addr(v_cache), int(max_rows), _haddr(k_new_host),
                                                _haddr(v_new_host), int(new_rows), int(offset), _haddr(q_host),
                                                _haddr(bias_host), _haddr(out_host), ctypes.byref(p),
                                                _addr(workspace), int(workspace_bytes), stream or None))


def vtmu_rope_params_init() -> vtmu_rope_params:
    r = vtmu_rope_params()
    load_library().vtmu_rope_params_init(ctypes.byref(r))
    return r


def vtmu_rope(x, out, T: int, heads: int, offset: int, r: vtmu_rope_params, stream: int = 0) -> None:
    _check(load_library().vtmu_rope(_addr(x), _addr(out), int(T), int(heads), int(offset), ctypes.byref(r),
                                    stream or None))


def vtmu_decode_step_rope(k_cache, v_cache, max_rows: int, k_new, v_new, new_rows: int, offset: int, q, bias, out,
                          p: vtmu_attention_params, r: vtmu_rope_params, workspace, workspace_bytes: int,
                          stream: int = 0) -> None:
    _check(load_library().vtmu_decode_step_rope(_addr(k_cache), _addr(v_cache), int(max_rows), _addr(k_new),
                                                _addr(v_new), int(new_rows), int(offset), _addr(q), _addr(bias),
                                                _addr(out), ctypes.byref(p), ctypes.byref(r), _addr(workspace),
                                                int(workspace_bytes), stream or None))


def vtmu_cache_write(cache, max_rows: int, width: int, values, rows: int, offset: int, stream: int = 0) -> None:
    _check(load_library().vtmu_cache_write(_addr(cache), int(max_rows), int(width), _addr(values),
                                           int(rows), int(offset), stream or None))


def vtmu_attention_decode_noalloc(q, k, v, bias, out, p: vtmu_attention_params, stream: int = 0) -> None:
    """Decode (T == 1) with the library's static scratch: no workspace, no
    allocation, for callers that cannot allocate device memory.  The first
    call on a device looks up the scratch address (do it before any stream
    capture); calls that overlap on the GPU race on the shared scratch."""
    _check(load_library().vtmu_attention_decode_noalloc(_addr(q), _addr(k), _addr(v), _addr(bias), _addr(out),
                                                        ctypes.byref(p), stream or None))


def vtmu_mla_params_init() -> vtmu_mla_params:
    p = vtmu_mla_params()
    load_library().vtmu_mla_params_init(ctypes.byref(p))
    return p


def vtmu_mla_workspace_size(p: vtmu_mla_params) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().vtmu_mla_workspace_size(ctypes.byref(p), ctypes.byref(n)))
    return int(n.value)


def vtmu_mla_attention(q, state, k_b, v_b, out, p: vtmu_mla_params, workspace, workspace_bytes: int,
                       stream: int = 0) -> None:
    _check(load_library().vtmu_mla_attention(_addr(q), _addr(state), _addr(k_b), _addr(v_b), _addr(out),
                                             ctypes.byref(p), _addr(workspace), int(workspace_bytes),
                                             stream or None))


def vtmu_mla_decode_step(state, max_rows: int, state_new, new_rows: int, offset: int, q, k_b, v_b, out,
                         p: vtmu_mla_params, workspace, workspace_bytes: int, stream: int = 0) -> None:
    _check(load_library().vtmu_mla_decode_step(_addr(state), int(max_rows), _addr(state_new), int(new_rows),
                                               int(offset), _addr(q), _addr(k_b), _addr(v_b), _addr(out),
                                               ctypes.byref(p), _addr(workspace), int(workspace_bytes),
                                               stream or None))


def vtmu_mla_decode_step_host_workspace_size(p: vtmu_mla_params, new_rows: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().vtmu_mla_decode_step_host_workspace_size(ctypes.byref(p), int(new_rows), ctypes.byref(n)))
    return int(n.value)


def vtmu_mla_decode_step_host(state, max_rows: int, state_new_host, new_rows: int, offset: int, q_host, k_b, v_b,
                              out_host, p: vtmu_mla_params, workspace, workspace_bytes: int, stream: int = 0) -> None:
    """vtmu_mla_decode_step with q / new latent rows / out in host memory
    (numpy arrays or CPU tensors, f32, contiguous; pinned buffers are used in
    place).  Returns once out_host holds the result."""
    _check(load_library().vtmu_mla_decode_step_host(_addr(state), int(max_rows), _haddr(state_new_host),
                                                    int(new_rows), int(offset), _haddr(q_host), _addr(k_b),
                                                    _addr(v_b), _haddr(out_host), ctypes.byref(p), _addr(workspace),
                                                    int(workspace_bytes), stream or None))


def vtmu_device_error() -> int:
    """Synchronises the device; returns and clears the kernels' wait-timeout
    flags (0 when no bounded wait gave up)."""
    v = ctypes.c_uint(0)
    _check(load_library().vtmu_device_error(ctypes.byref(v)))
    return int(v.value)


def vtmu_features() -> str:
    return load_library().vtmu_features().decode()


def vtmu_last_error() -> str:
    return load_library().vtmu_last_error().decode()


# ------------------------------------------------------------ torch helpers
def make_params(T, S, *, heads, headDim, kvHeads=None, vHeadDim=None, causal=True, posOffset=0,
                scale=None, softcap=None, window=None, alibi=False, alibiMax=None, alibiSlopes=None,
                bias_kind=VTMU_BIAS_NONE, kernel=VTMU_KERNEL_AUTO, decode_splits=0, sinks=None):
    """A params struct from the op catalog's parameter names.  ALiBi
    precedence: alibiSlopes, then alibiMax, then alibi.  The returned struct
    keeps any slope array alive as ``_slopes``."""
    p = vtmu_attention_params_init()
    p.T, p.S = int(T), int(S)
    p.heads = int(heads)
    p.kv_heads = 0 if kvHeads is None else int(kvHeads)
    p.head_dim = int(headDim)
    p.v_head_dim = 0 if vHeadDim is None else int(vHeadDim)
    p.causal = 1 if causal else 0
    p.pos_offset = int(posOffset)
    if scale is not None:
        p.has_scale, p.scale = 1, float(scale)
    p.softcap = 0.0 if softcap is None else float(softcap)
    p.window = 0 if window is None else int(window)
    if alibiSlopes is not None:
        arr = (ctypes.c_float * len(alibiSlopes))(*[float(s) for s in alibiSlopes])
        p.alibi, p.alibi_slopes = VTMU_ALIBI_SLOPES, ctypes.cast(arr, ctypes.POINTER(ctypes.c_float))
        p._slopes = arr
    elif alibiMax is not None:
        p.alibi, p.alibi_max = VTMU_ALIBI_MPT, float(alibiMax)
    elif alibi:
        p.alibi = VTMU_ALIBI_BLOOM
    p.bias_kind = int(bias_kind)
    p.kernel = int(kernel)
    p.decode_splits = int(decode_splits)
    p.sinks = 0 if sinks is None else int(sinks)
    return p


def make_rope_params(*, headDim, base=None, rotaryDim=None, interleaved=False, scaling=None, invFreq=None,
                     attentionFactor=None):
    """A rope params struct from op "rope"'s parameter names.  ``scaling`` is
    config.json's rope_scaling object; "linear" maps to the library's linear
    scaling and any other kind is passed on so that the library refuses it
    with "rope.scaling" named.  Keeps an invFreq array alive as ``_inv``."""
    r = vtmu_rope_params_init()
    r.head_dim = int(headDim)
    r.rotary_dim = 0 if rotaryDim is None else int(rotaryDim)
    r.interleaved = 1 if interleaved else 0
    r.base = 0.0 if base is None else float(base)
    if scaling is not None:
        kind = scaling.get("rope_type", scaling.get("type"))
        r.scaling = VTMU_ROPE_SCALING_LINEAR if kind == "linear" else 100
        r.scaling_factor = float(scaling.get("factor", 0.0))
    r.attention_factor = 0.0 if attentionFactor is None else float(attentionFactor)
    if invFreq is not None:
        arr = (ctypes.c_float * len(invFreq))(*[float(f) for f in invFreq])
        r.inv_freq = ctypes.cast(arr, ctypes.POINTER(ctypes.c_float))
        r._inv = arr
    return r


class Workspace:
    """A zero-initialised device scratch buffer (torch-allocated) that grows
    on demand.  One per concurrent stream."""

    def __init__(self, device=None):
        import torch
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.buf = None

    def get(self, nbytes: int):
        import torch
        if nbytes == 0:
            return None, 0
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf, self.buf.numel()


_ws = {}


def _default_workspace(device):
    key = (device.type, device.index)
    if key not in _ws:
        _ws[key] = Workspace(device)
    return _ws[key]


def attention(q, k, v, bias=None, *, heads, headDim, out=None, workspace=None, stream=None, **params):
    """op "attention" on CUDA tensors: q [T, heads*headDim], k [S, kvHeads*headDim],
    v [S, kvHeads*vHeadDim], optional bias [T, S] or [heads, T, S]; returns
    out [T, heads*vHeadDim] (float32).  Keyword names as in the op catalog."""
    import torch
    T, S = q.shape[0], k.shape[0]
    vhd = params.get("vHeadDim") or headDim
    bias_kind = VTMU_BIAS_NONE
    if bias is not None:
        bias_kind = VTMU_BIAS_TS if bias.dim() == 2 else VTMU_BIAS_HTS
    p = make_params(T, S, heads=heads, headDim=headDim, bias_kind=bias_kind, **params)
    for name, t in (("q", q), ("k", k), ("v", v), ("bias", bias)):
        if t is not None and (not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    if out is None:
        out = torch.empty((T, heads * vhd), dtype=torch.float32, device=q.device)
    nbytes = vtmu_attention_workspace_size(p)
    ws = workspace if workspace is not None else _default_workspace(q.device)
    buf, cap = ws.get(nbytes)
    st = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    vtmu_attention(q, k, v, bias, out, p, buf, cap, st)
    return out


def decode_step(k_cache, v_cache, k_new, v_new, offset: int, q, bias=None, *, heads, headDim, out=None,
                workspace=None, stream=None, **params):
    """A decode step on CUDA tensors: cache_write of k_new / v_new into the
    caches at row ``offset``, then attention of q over the updated caches
    (all of their rows, posOffset defaulting to the last new row).  One launch
    when the decode kernel covers the shape.  Returns out."""
    import torch
    T, S = q.shape[0], k_cache.shape[0]
    vhd = params.get("vHeadDim") or headDim
    params.setdefault("posOffset", offset + k_new.shape[0] - T)
    bias_kind = VTMU_BIAS_NONE
    if bias is not None:
        bias_kind = VTMU_BIAS_TS if bias.dim() == 2 else VTMU_BIAS_HTS
    p = make_params(T, S, heads=heads, headDim=headDim, bias_kind=bias_kind, **params)
    if out is None:
        out = torch.empty((T, heads * vhd), dtype=torch.float32, device=q.device)
    nbytes = vtmu_attention_workspace_size(p)
    ws = workspace if workspace is not None else _default_workspace(q.device)
    buf, cap = ws.get(nbytes)
    st = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    vtmu_decode_step(k_cache, v_cache, S, k_new, v_new, k_new.shape[0], offset, q, bias, out, p, buf, cap, st)
    return out


def rope(x, *, headDim, offset=0, out=None, stream=None, **params):
    """op "rope" on a CUDA tensor x [T, heads*headDim]; ``out=x`` turns it in
    place.  Params as make_rope_params.  Returns out."""
    import torch
    T, width = x.shape
    if out is None:
        out = torch.empty_like(x)
    r = make_rope_params(headDim=headDim, **params)
    st = stream if stream is not None else torch.cuda.current_stream(x.device).cuda_stream
    vtmu_rope(x, out, T, width // headDim, offset, r, st)
    return out


def decode_step_rope(k_cache, v_cache, k_new, v_new, offset: int, q, bias=None, *, heads, headDim, rope: dict,
                     out=None, workspace=None, stream=None, **params):
    """decode_step with the rotary embedding ``rope`` (make_rope_params
    names, headDim taken from the call) fused in: q and the new keys are
    turned inside the one decode launch, the caches receive turned keys."""
    import torch
    T, S = q.shape[0], k_cache.shape[0]
    vhd = params.get("vHeadDim") or headDim
    params.setdefault("posOffset", offset + k_new.shape[0] - T)
    bias_kind = VTMU_BIAS_NONE
    if bias is not None:
        bias_kind = VTMU_BIAS_TS if bias.dim() == 2 else VTMU_BIAS_HTS
    p = make_params(T, S, heads=heads, headDim=headDim, bias_kind=bias_kind, **params)
    r = make_rope_params(headDim=headDim, **rope)
    if out is None:
        out = torch.empty((T, heads * vhd), dtype=torch.float32, device=q.device)
    nbytes = vtmu_attention_workspace_size(p)
    ws = workspace if workspace is not None else _default_workspace(q.device)
    buf, cap = ws.get(nbytes)
    st = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    vtmu_decode_step_rope(k_cache, v_cache, S, k_new, v_new, k_new.shape[0], offset, q, bias, out, p, r, buf, cap,
                          st)
    return out


def cache_write(cache, values, offset: int, stream=None):
    """op "cache_write" on CUDA tensors: cache [maxRows, width] is updated in
    place with values [rows, width] at row ``offset``; returns cache."""
    import torch
    for name, t in (("cache", cache), ("values", values)):
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or t.dim() != 2:
            raise ValueError(f"{name} must be a contiguous 2-D float32 CUDA tensor")
    if values.shape[1] != cache.shape[1]:
        raise ValueError("values must be as wide as the cache")
    st = stream if stream is not None else torch.cuda.current_stream(cache.device).cuda_stream
    vtmu_cache_write(cache, cache.shape[0], cache.shape[1], values, values.shape[0], offset, st)
    return cache


def make_mla_params(T, S, *, heads, kv_rank=512, qk_nope, qk_rope=64, v_head_dim, scale=None, causal=True,
                    posOffset=0, window=None, sinks=None, kernel=0):
    """An mla params struct from the IR page's parameter names (mla_attention)."""
    p = vtmu_mla_params_init()
    p.T, p.S = int(T), int(S)
    p.heads, p.kv_rank, p.qk_nope, p.qk_rope, p.v_head_dim = (int(heads), int(kv_rank), int(qk_nope), int(qk_rope),
                                                              int(v_head_dim))
    p.causal = 1 if causal else 0
    if scale is not None:
        p.has_scale, p.scale = 1, float(scale)
    p.pos_offset = int(posOffset)
    p.window = 0 if window is None else int(window)
    p.sinks = 0 if sinks is None else int(sinks)
    p.kernel = int(kernel)
    return p


def mla_attention(q, state, k_b, v_b, *, heads, qk_nope, v_head_dim, out=None, workspace=None, stream=None,
                  S=None, **params):
    """mla_attention on CUDA tensors: q [T, heads*(qk_nope+qk_rope)], state
    [rows, kv_rank+qk_rope] (its first S rows are read; all by default),
    k_b [heads*qk_nope, kv_rank], v_b [heads*v_head_dim, kv_rank]; returns
    out [T, heads*v_head_dim] (float32)."""
    import torch
    T = q.shape[0]
    p = make_mla_params(T, state.shape[0] if S is None else S, heads=heads, qk_nope=qk_nope,
                        v_head_dim=v_head_dim, **params)
    for name, t in (("q", q), ("state", state), ("k_b", k_b), ("v_b", v_b)):
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    if out is None:
        out = torch.empty((T, heads * v_head_dim), dtype=torch.float32, device=q.device)
    nbytes = vtmu_mla_workspace_size(p)
    ws = workspace if workspace is not None else _default_workspace(q.device)
    buf, cap = ws.get(nbytes)
    st = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    vtmu_mla_attention(q, state, k_b, v_b, out, p, buf, cap, st)
    return out


def mla_decode_step(state, state_new, offset: int, q, k_b, v_b, *, heads, qk_nope, v_head_dim, out=None,
                    workspace=None, stream=None, **params):
    """A latent-attention decode step on CUDA tensors: cache_write of
    state_new into state at row ``offset``, then mla_attention over the
    first offset + new rows of the cache (posOffset defaulting to the last
    new row).  Returns out."""
    import torch
    T, R = q.shape[0], state_new.shape[0]
    params.setdefault("posOffset", offset + R - T)
    p = make_mla_params(T, offset + R, heads=heads, qk_nope=qk_nope, v_head_dim=v_head_dim, **params)
    if out is None:
        out = torch.empty((T, heads * v_head_dim), dtype=torch.float32, device=q.device)
    nbytes = vtmu_mla_workspace_size(p)
    ws = workspace if workspace is not None else _default_workspace(q.device)
    buf, cap = ws.get(nbytes)
    st = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    vtmu_mla_decode_step(state, state.shape[0], state_new, R, offset, q, k_b, v_b, out, p, buf, cap, st)
    return out
