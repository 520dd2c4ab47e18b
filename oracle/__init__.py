"""CPU oracle for the f32 ``attention``, ``cache_write`` and ``rope`` ops, and
for absorbed latent attention (``mla_attention``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product path (the
``f32_gqa_attention_gb300`` package and its CUDA library) never imports this
module, and this module never imports the product.

The arithmetic lives in ``attention_oracle.c`` (plain C, every sum in double,
OpenMP over query rows).  This wrapper only resolves the op's parameter
defaults as the op catalog states them (vtmu.mpakt.dev/api/ops, op
"attention"):

* ``kvHeads`` defaults to ``heads``;
* ``vHeadDim`` defaults to ``headDim`` (the page gives it only for a value
  width that is not headDim);
* ``causal`` defaults to true, ``posOffset`` to 0;
* ``scale`` replaces 1/sqrt(headDim);
* ``softcap`` and ``window`` are off when absent (or 0);
* ALiBi: ``alibiSlopes`` wins over ``alibiMax``, which wins over ``alibi``;
* ``sinks`` (the IR page's attention sinks, not a param of the op page):
  with a window, keys before ``sinks`` stay visible; 0 or absent = none.

``mla_attention`` (the IR schema page's ``$defs.op_mla_attention``) takes
q [T, heads*(qk_nope + qk_rope)], the latent cache state [S, kv_rank +
qk_rope], k_b [heads*qk_nope, kv_rank] and v_b [heads*v_head_dim, kv_rank]
(the page's parameter names); ``scale`` defaults to 1/sqrt(qk_nope +
qk_rope), the query/key width per head, as op "attention"'s scale defaults
to 1/sqrt(headDim); causal, window and sinks as for ``attention``.

``Oracle(path)`` wraps one compiled build; the module-level functions use the
default build of ``attention_oracle.c``.  The tests also compile copies with a
planted mistake and check that the pins catch each one.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "attention_oracle.c")
_LIB = os.path.join(HERE, "liboracle.so")

BIAS_NONE, BIAS_TS, BIAS_HTS = 0, 1, 2
ALIBI_BLOOM, ALIBI_MPT = 1, 2

_lock = threading.Lock()
_default = None


class _Desc(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int64),
        ("S", ctypes.c_int64),
        ("heads", ctypes.c_int),
        ("kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int),
        ("v_head_dim", ctypes.c_int),
        ("causal", ctypes.c_int),
        ("pos_offset", ctypes.c_int64),
        ("scale", ctypes.c_double),
        ("softcap", ctypes.c_double),
        ("window", ctypes.c_int64),
        ("slopes", ctypes.POINTER(ctypes.c_double)),
        ("bias_kind", ctypes.c_int),
        ("sinks", ctypes.c_int64),
    ]


class _MlaDesc(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int64),
        ("S", ctypes.c_int64),
        ("heads", ctypes.c_int),
        ("kv_rank", ctypes.c_int),
        ("qk_nope", ctypes.c_int),
        ("qk_rope", ctypes.c_int),
        ("v_head_dim", ctypes.c_int),
        ("causal", ctypes.c_int),
        ("pos_offset", ctypes.c_int64),
        ("scale", ctypes.c_double),
        ("window", ctypes.c_int64),
        ("sinks", ctypes.c_int64),
    ]


def compile_source(src: str, out: str) -> str:
    """gcc -O2 -fopenmp a C file of the oracle into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle (no CUDA involved).  Returns the .so path."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(SOURCE)):
            return _LIB
        return compile_source(SOURCE, _LIB)


def _f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """One compiled build of the oracle."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        lib.oracle_attention.argtypes = [ctypes.POINTER(_Desc), p, p, p, p, p]
        lib.oracle_attention_rows.argtypes = [ctypes.POINTER(_Desc), p, p, p,
                                              p, p, p, ctypes.c_int64, p]
        lib.oracle_alibi_slopes.argtypes = [ctypes.c_int, ctypes.c_int,
                                            ctypes.c_double, p]
        lib.oracle_cache_write.argtypes = [p, ctypes.c_int64, ctypes.c_int64,
                                           p, ctypes.c_int64, ctypes.c_int64]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_mla_attention.argtypes = [ctypes.POINTER(_MlaDesc), p, p, p, p, p]
        lib.oracle_mla_attention_rows.argtypes = [ctypes.POINTER(_MlaDesc), p, p, p, p, p, p,
                                                  ctypes.c_int64, p]
        lib.oracle_rope_inv_freq.argtypes = [ctypes.c_int, ctypes.c_double, p]
        lib.oracle_rope.argtypes = [p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                    ctypes.c_double, p, ctypes.c_double, p]
        self.lib = lib
        self.path = path

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def alibi_slopes(self, heads: int, alibi: bool = False, alibiMax=None,
                     alibiSlopes=None):
        """Per-head ALiBi slopes in double, or None when ALiBi is off."""
        if alibiSlopes is not None:
            s = np.ascontiguousarray(np.asarray(alibiSlopes, dtype=np.float64))
            if s.shape != (heads,):
                raise ValueError("alibiSlopes needs one slope per head")
            return s
        if alibiMax is not None:
            kind, bmax = ALIBI_MPT, float(alibiMax)
        elif alibi:
            kind, bmax = ALIBI_BLOOM, 0.0
        else:
            return None
        out = np.zeros(heads, dtype=np.float64)
        if self.lib.oracle_alibi_slopes(int(heads), kind, bmax, _ptr(out)):
            raise ValueError("oracle_alibi_slopes failed")
        return out

    def _prepare(self, q, k, v, bias, heads, headDim, kvHeads, vHeadDim,
                 causal, posOffset, scale, softcap, window, alibi, alibiMax,
                 alibiSlopes, sinks=None):
        q, k, v = _f32(q), _f32(k), _f32(v)
        kvHeads = heads if kvHeads is None else int(kvHeads)
        vHeadDim = headDim if vHeadDim is None else int(vHeadDim)
        if q.ndim != 2 or q.shape[1] != heads * headDim:
            raise ValueError("q must be [T, heads*headDim]")
        if k.ndim != 2 or k.shape[1] != kvHeads * headDim:
            raise ValueError("k must be [S, kvHeads*headDim]")
        if (v.ndim != 2 or v.shape[1] != kvHeads * vHeadDim
                or v.shape[0] != k.shape[0]):
            raise ValueError("v must be [S, kvHeads*vHeadDim]")
        T, S = q.shape[0], k.shape[0]
        bias_kind = BIAS_NONE
        if bias is not None:
            bias = _f32(bias)
            if bias.shape == (T, S):
                bias_kind = BIAS_TS
            elif bias.shape == (heads, T, S):
                bias_kind = BIAS_HTS
            else:
                raise ValueError("bias must be [T, S] or [heads, T, S]")
        slopes = self.alibi_slopes(heads, alibi, alibiMax, alibiSlopes)
        d = _Desc()
        d.T, d.S = T, S
        d.heads, d.kv_heads = heads, kvHeads
        d.head_dim, d.v_head_dim = headDim, vHeadDim
        d.causal = 1 if causal else 0
        d.pos_offset = int(posOffset)
        d.scale = (1.0 / math.sqrt(headDim)) if scale is None else float(scale)
        d.softcap = 0.0 if softcap is None else float(softcap)
        d.window = 0 if window is None else int(window)
        d.slopes = (slopes.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
                    if slopes is not None else None)
        d.bias_kind = bias_kind
        d.sinks = 0 if sinks is None else int(sinks)
        if d.sinks < 0:
            raise ValueError("sinks must be >= 0")
        return d, (q, k, v, bias, slopes)

    def attention(self, q, k, v, bias=None, *, heads, headDim, kvHeads=None,
                  vHeadDim=None, causal=True, posOffset=0, scale=None,
                  softcap=None, window=None, alibi=False, alibiMax=None,
                  alibiSlopes=None, sinks=None):
        """The whole op: returns out [T, heads*vHeadDim] as float64."""
        d, keep = self._prepare(q, k, v, bias, heads, headDim, kvHeads,
                                vHeadDim, causal, posOffset, scale, softcap,
                                window, alibi, alibiMax, alibiSlopes, sinks)
        q, k, v, bias, _ = keep
        out = np.zeros((d.T, d.heads * d.v_head_dim), dtype=np.float64)
        rc = self.lib.oracle_attention(ctypes.byref(d), _ptr(q), _ptr(k),
                                       _ptr(v), _ptr(bias), _ptr(out))
        if rc:
            raise ValueError(f"oracle_attention failed ({rc})")
        return out

    def attention_rows(self, q, k, v, bias=None, *, rows, heads, headDim,
                       kvHeads=None, vHeadDim=None, causal=True, posOffset=0,
                       scale=None, softcap=None, window=None, alibi=False,
                       alibiMax=None, alibiSlopes=None, sinks=None):
        """Selected (t, h) rows only: returns [len(rows), vHeadDim] float64."""
        d, keep = self._prepare(q, k, v, bias, heads, headDim, kvHeads,
                                vHeadDim, causal, posOffset, scale, softcap,
                                window, alibi, alibiMax, alibiSlopes, sinks)
        q, k, v, bias, _ = keep
        rows = list(rows)
        ts = np.ascontiguousarray([int(t) for t, _ in rows], dtype=np.int64)
        hs = np.ascontiguousarray([int(h) for _, h in rows], dtype=np.int32)
        out = np.zeros((len(rows), d.v_head_dim), dtype=np.float64)
        rc = self.lib.oracle_attention_rows(ctypes.byref(d), _ptr(q), _ptr(k),
                                            _ptr(v), _ptr(bias), _ptr(ts),
                                            _ptr(hs), len(rows), _ptr(out))
        if rc:
            raise ValueError(f"oracle_attention_rows failed ({rc})")
        return out

    def cache_write(self, cache, values, offset):
        """In place on the numpy array ``cache`` [maxRows, width]; returns it."""
        if not (isinstance(cache, np.ndarray) and cache.dtype == np.float32
                and cache.flags.c_contiguous and cache.ndim == 2):
            raise ValueError("cache must be a C-contiguous float32 [maxRows, width]")
        values = _f32(values)
        if values.ndim != 2 or values.shape[1] != cache.shape[1]:
            raise ValueError("values must be [rows, width]")
        rc = self.lib.oracle_cache_write(_ptr(cache), cache.shape[0],
                                         cache.shape[1], _ptr(values),
                                         values.shape[0], int(offset))
        if rc:
            raise ValueError("cache_write: rows do not fit the cache at offset")
        return cache

    def rope_inv_freq(self, rotaryDim, base=None):
        """base^(-2j / rotaryDim) for j < rotaryDim / 2, in double."""
        out = np.zeros(int(rotaryDim) // 2, dtype=np.float64)
        if self.lib.oracle_rope_inv_freq(int(rotaryDim), 10000.0 if base is None else float(base), _ptr(out)):
            raise ValueError("rope: rotaryDim must be positive and even, base positive")
        return out

    def rope(self, x, *, headDim, offset=0, base=None, rotaryDim=None,
             interleaved=False, scaling=None, invFreq=None,
             attentionFactor=None):
        """op "rope" (vtmu.mpakt.dev/api/ops): x [T, heads*headDim] -> the
        same shape, float64.  Defaults as the catalog states them: base
        (rope_theta) 10000, offset 0, rotaryDim = headDim, half-split pairs.
        ``scaling`` is config.json's rope_scaling object; the linear scheme
        (positions divided by ``factor``) is the one implemented here.
        ``invFreq`` replaces the base-derived frequencies; ``attentionFactor``
        multiplies cos and sin (default 1)."""
        x = _f32(x)
        headDim = int(headDim)
        if x.ndim != 2 or headDim <= 0 or x.shape[1] % headDim:
            raise ValueError("x must be [T, heads*headDim]")
        heads = x.shape[1] // headDim
        rd = headDim if rotaryDim is None else int(rotaryDim)
        if rd <= 0 or rd % 2 or rd > headDim:
            raise ValueError("rotaryDim must be even and at most headDim")
        if invFreq is not None:
            inv = np.ascontiguousarray(np.asarray(invFreq, dtype=np.float64))
            if inv.shape != (rd // 2,):
                raise ValueError("invFreq needs rotaryDim / 2 values")
        else:
            inv = self.rope_inv_freq(rd, base)
        divisor = 1.0
        if scaling is not None:
            kind = scaling.get("rope_type", scaling.get("type"))
            if kind != "linear":
                raise ValueError(f"rope.scaling: {kind!r} is not implemented")
            divisor = float(scaling["factor"])
        af = 1.0 if attentionFactor is None else float(attentionFactor)
        out = np.zeros(x.shape, dtype=np.float64)
        if x.shape[0] and self.lib.oracle_rope(_ptr(x), x.shape[0], heads, headDim, rd,
                                               1 if interleaved else 0, int(offset), divisor,
                                               _ptr(inv), af, _ptr(out)):
            raise ValueError("oracle_rope failed")
        return out

    def _mla_prepare(self, q, state, k_b, v_b, heads, kv_rank, qk_nope, qk_rope,
                     v_head_dim, scale, causal, posOffset, window, sinks):
        q, state, k_b, v_b = _f32(q), _f32(state), _f32(k_b), _f32(v_b)
        H, R, N, P, Dv = int(heads), int(kv_rank), int(qk_nope), int(qk_rope), int(v_head_dim)
        if q.ndim != 2 or q.shape[1] != H * (N + P):
            raise ValueError("q must be [T, heads*(qk_nope + qk_rope)]")
        if state.ndim != 2 or state.shape[1] != R + P:
            raise ValueError("state must be [S, kv_rank + qk_rope]")
        if k_b.shape != (H * N, R):
            raise ValueError("k_b must be [heads*qk_nope, kv_rank]")
        if v_b.shape != (H * Dv, R):
            raise ValueError("v_b must be [heads*v_head_dim, kv_rank]")
        d = _MlaDesc()
        d.T, d.S = q.shape[0], state.shape[0]
        d.heads, d.kv_rank, d.qk_nope, d.qk_rope, d.v_head_dim = H, R, N, P, Dv
        d.causal = 1 if causal else 0
        d.pos_offset = int(posOffset)
        d.scale = (1.0 / math.sqrt(N + P)) if scale is None else float(scale)
        d.window = 0 if window is None else int(window)
        d.sinks = 0 if sinks is None else int(sinks)
        if d.window < 0 or d.sinks < 0:
            raise ValueError("window and sinks must be >= 0")
        return d, (q, state, k_b, v_b)

    def mla_attention(self, q, state, k_b, v_b, *, heads, kv_rank, qk_nope, qk_rope,
                      v_head_dim, scale=None, causal=True, posOffset=0, window=None,
                      sinks=None):
        """Absorbed latent attention by its un-absorbed definition: returns
        out [T, heads*v_head_dim] as float64."""
        d, keep = self._mla_prepare(q, state, k_b, v_b, heads, kv_rank, qk_nope, qk_rope,
                                    v_head_dim, scale, causal, posOffset, window, sinks)
        q, state, k_b, v_b = keep
        out = np.zeros((d.T, d.heads * d.v_head_dim), dtype=np.float64)
        rc = self.lib.oracle_mla_attention(ctypes.byref(d), _ptr(q), _ptr(state), _ptr(k_b),
                                           _ptr(v_b), _ptr(out))
        if rc:
            raise ValueError(f"oracle_mla_attention failed ({rc})")
        return out

    def mla_attention_rows(self, q, state, k_b, v_b, *, rows, heads, kv_rank, qk_nope,
                           qk_rope, v_head_dim, scale=None, causal=True, posOffset=0,
                           window=None, sinks=None):
        """Selected (t, h) rows only: returns [len(rows), v_head_dim] float64."""
        d, keep = self._mla_prepare(q, state, k_b, v_b, heads, kv_rank, qk_nope, qk_rope,
                                    v_head_dim, scale, causal, posOffset, window, sinks)
        q, state, k_b, v_b = keep
        rows = list(rows)
        ts = np.ascontiguousarray([int(t) for t, _ in rows], dtype=np.int64)
        hs = np.ascontiguousarray([int(h) for _, h in rows], dtype=np.int32)
        out = np.zeros((len(rows), d.v_head_dim), dtype=np.float64)
        rc = self.lib.oracle_mla_attention_rows(ctypes.byref(d), _ptr(q), _ptr(state), _ptr(k_b),
                                                _ptr(v_b), _ptr(ts), _ptr(hs), len(rows), _ptr(out))
        if rc:
            raise ValueError(f"oracle_mla_attention_rows failed ({rc})")
        return out


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def num_threads() -> int:
    return default().num_threads()


def alibi_slopes(heads, alibi=False, alibiMax=None, alibiSlopes=None):
    return default().alibi_slopes(heads, alibi, alibiMax, alibiSlopes)


def attention(q, k, v, bias=None, **params):
    return default().attention(q, k, v, bias, **params)


def attention_rows(q, k, v, bias=None, **params):
    return default().attention_rows(q, k, v, bias, **params)


def cache_write(cache, values, offset):
    return default().cache_write(cache, values, offset)


def rope(x, **params):
    return default().rope(x, **params)


def rope_inv_freq(rotaryDim, base=None):
    return default().rope_inv_freq(rotaryDim, base)


def mla_attention(q, state, k_b, v_b, **params):
    return default().mla_attention(q, state, k_b, v_b, **params)


def mla_attention_rows(q, state, k_b, v_b, **params):
    return default().mla_attention_rows(q, state, k_b, v_b, **params)
