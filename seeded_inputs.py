"""Seeded synthetic inputs for the attention tests and the benchmark.

This module is shared by both sides of every parity check (the CPU oracle and
the CUDA library) and so holds none of the attention arithmetic: only random
numbers, shapes and the workload catalogue.

Random numbers: a counter-based SplitMix64 stream (Steele, Lea & Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014).  Word i of the
stream with seed s is mix64(s + (i + 1) * 0x9E3779B97F4A7C15) mod 2^64, with
mix64 the published SplitMix64 finaliser.  Uniforms take the top 53 bits;
normals come from the Box-Muller transform on consecutive word pairs.  The
stream does not depend on the numpy or torch version: the same seed gives the
same float32 arrays on every machine (up to last-ulp differences of the host's
log/cos/sin, which the f32 cast almost always hides).

Draw order inside one workload: q, k, v, then the bias values, then the bias
mask uniforms, then the new K/V rows of a decode step (latent attention: q,
the latent cache, k_b, v_b, the new cache rows).
"""
from __future__ import annotations

import math

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


class Stream:
    """A SplitMix64 word stream; every draw advances a counter."""

    def __init__(self, seed: int):
        self.seed = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
        self.counter = 0

    def words(self, n: int) -> np.ndarray:
        i = np.arange(self.counter + 1, self.counter + 1 + n, dtype=np.uint64)
        self.counter += n
        with np.errstate(over="ignore"):
            return _mix64(self.seed + i * _GAMMA)

    def uniform(self, n: int) -> np.ndarray:
        """n doubles in [0, 1)."""
        out = np.empty(n, dtype=np.float64)
        for lo in range(0, n, _CHUNK):
            m = min(_CHUNK, n - lo)
            out[lo:lo + m] = (self.words(m) >> np.uint64(11)).astype(np.float64) * 2.0**-53
        return out

    def normal_f32(self, n: int, sigma: float = 1.0) -> np.ndarray:
        """n float32 draws of N(0, sigma^2) (Box-Muller, pairs of words)."""
        out = np.empty(n, dtype=np.float32)
        for lo in range(0, n, 2 * _CHUNK):
            m = min(2 * _CHUNK, n - lo)
            pairs = (m + 1) // 2
            u = self.uniform(2 * pairs).reshape(pairs, 2)
            r = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
            th = 2.0 * math.pi * u[:, 1]
            z = np.empty((pairs, 2), dtype=np.float64)
            z[:, 0] = r * np.cos(th)
            z[:, 1] = r * np.sin(th)
            out[lo:lo + m] = (z.reshape(-1)[:m] * sigma).astype(np.float32)
        return out


def attention_inputs(T, S, heads, kvHeads, headDim, vHeadDim, seed, *,
                     sigma=1.0, bias=None, bias_mask_p=0.0):
    """q [T, heads*headDim], k [S, kvHeads*headDim], v [S, kvHeads*vHeadDim]
    (float32, N(0, sigma^2)) and an optional bias ("ts" -> [T, S],
    "hts" -> [heads, T, S]) of N(0, 1) values with a Bernoulli(bias_mask_p)
    share set to -1e9."""
    st = Stream(seed)
    out = {
        "q": st.normal_f32(T * heads * headDim, sigma).reshape(T, heads * headDim),
        "k": st.normal_f32(S * kvHeads * headDim, sigma).reshape(S, kvHeads * headDim),
        "v": st.normal_f32(S * kvHeads * vHeadDim, sigma).reshape(S, kvHeads * vHeadDim),
    }
    if bias is not None:
        shape = (T, S) if bias == "ts" else (heads, T, S)
        n = int(np.prod(shape))
        b = st.normal_f32(n)
        if bias_mask_p > 0.0:
            b[st.uniform(n) < bias_mask_p] = np.float32(-1e9)
        out["bias"] = b.reshape(shape)
    return out


def decode_inputs(max_rows, heads, kvHeads, headDim, vHeadDim, seed, *, sigma=1.0, rows=1):
    """A decode step: caches kc [max_rows, kvHeads*headDim] and
    vc [max_rows, kvHeads*vHeadDim] already filled, the step's query rows
    q [rows, heads*headDim] and the new rows k_new / v_new [rows, ...]."""
    st = Stream(seed)
    return {
        "q": st.normal_f32(rows * heads * headDim, sigma).reshape(rows, heads * headDim),
        "kc": st.normal_f32(max_rows * kvHeads * headDim, sigma).reshape(max_rows, kvHeads * headDim),
        "vc": st.normal_f32(max_rows * kvHeads * vHeadDim, sigma).reshape(max_rows, kvHeads * vHeadDim),
        "k_new": st.normal_f32(rows * kvHeads * headDim, sigma).reshape(rows, kvHeads * headDim),
        "v_new": st.normal_f32(rows * kvHeads * vHeadDim, sigma).reshape(rows, kvHeads * vHeadDim),
    }


def mla_inputs(rows, T, heads, kv_rank, qk_nope, qk_rope, v_head_dim, seed, *, new_rows=0):
    """Absorbed latent attention: q [T, heads*(qk_nope+qk_rope)] and the
    latent cache state [rows, kv_rank+qk_rope] of N(0, 1) values; the
    up-projections k_b [heads*qk_nope, kv_rank] and v_b [heads*v_head_dim,
    kv_rank] of N(0, 1/kv_rank) values (so keys and values have unit
    variance); and state_new [new_rows, kv_rank+qk_rope] of N(0, 1) values.
    Draw order: q, state, k_b, v_b, state_new."""
    st = Stream(seed)
    W = kv_rank + qk_rope
    sw = 1.0 / math.sqrt(kv_rank)
    return {
        "q": st.normal_f32(T * heads * (qk_nope + qk_rope)).reshape(T, heads * (qk_nope + qk_rope)),
        "state": st.normal_f32(rows * W).reshape(rows, W),
        "k_b": st.normal_f32(heads * qk_nope * kv_rank, sw).reshape(heads * qk_nope, kv_rank),
        "v_b": st.normal_f32(heads * v_head_dim * kv_rank, sw).reshape(heads * v_head_dim, kv_rank),
        "state_new": st.normal_f32(new_rows * W).reshape(new_rows, W),
    }


# The workloads: shapes, op parameters (named as the op catalog names them),
# seeds and input scale.  Parameters left out take the op's defaults.
WORKLOADS = {
    "tiny_prefill": dict(
        kind="prefill", T=16, S=16, heads=4, kvHeads=4, headDim=32, seed=0,
        params=dict(causal=True, posOffset=0)),
    "gqa_decode": dict(
        kind="decode", max_rows=32768, offset=32767, heads=32, kvHeads=8,
        headDim=128, seed=1, params=dict(causal=True, posOffset=32767)),
    "gqa_decode_rope": dict(
        kind="decode", max_rows=32768, offset=32767, heads=32, kvHeads=8,
        headDim=128, seed=1, params=dict(causal=True, posOffset=32767),
        rope=dict(base=500000.0)),
    "gqa_spec_decode": dict(
        kind="decode", rows=4, max_rows=32768, offset=32764, heads=32, kvHeads=8,
        headDim=128, seed=6, params=dict(causal=True, posOffset=32764)),
    "gqa_decode_sinks": dict(
        kind="decode", max_rows=32768, offset=32767, heads=32, kvHeads=8,
        headDim=128, seed=1, params=dict(causal=True, posOffset=32767, window=8188, sinks=4)),
    "gqa_prefill": dict(
        kind="prefill", T=4096, S=4096, heads=32, kvHeads=8, headDim=128,
        seed=2, params=dict(causal=True, posOffset=0)),
    "swa_softcap_prefill": dict(
        kind="prefill", T=8192, S=8192, heads=16, kvHeads=8, headDim=256,
        seed=3, sigma=2.0,
        params=dict(causal=True, scale=1.0 / 16, softcap=50.0, window=4096)),
    "swa_sinks_prefill": dict(
        kind="prefill", T=8192, S=8192, heads=16, kvHeads=8, headDim=256,
        seed=3, sigma=2.0,
        params=dict(causal=True, scale=1.0 / 16, softcap=50.0, window=4096, sinks=4)),
    "latent_bias_prefill": dict(
        kind="prefill", T=2048, S=2048, heads=128, kvHeads=128, headDim=192,
        vHeadDim=128, seed=4, bias="ts", bias_mask_p=0.1,
        params=dict(causal=False)),
    "alibi_prefill": dict(
        kind="prefill", T=2048, S=2048, heads=32, kvHeads=32, headDim=128,
        seed=5, params=dict(causal=True, alibi=True)),
    # Absorbed latent attention (the IR page's mla_attention), decode steps:
    # cache_write of one latent row at 32767, then one query row over 32768
    # cache rows.  DeepSeek-V2-Lite's shape (16 heads) and DeepSeek-V3's (128).
    "mla_decode": dict(
        kind="mla_decode", max_rows=32768, offset=32767, heads=16, kv_rank=512, qk_nope=128,
        qk_rope=64, v_head_dim=128, seed=7, params=dict(causal=True, posOffset=32767)),
    "mla_decode_v3": dict(
        kind="mla_decode", max_rows=32768, offset=32767, heads=128, kv_rank=512, qk_nope=128,
        qk_rope=64, v_head_dim=128, seed=8, params=dict(causal=True, posOffset=32767)),
}


def workload_inputs(name):
    """Inputs of a catalogue workload (see WORKLOADS)."""
    w = WORKLOADS[name]
    if w["kind"] == "mla_decode":
        R = w.get("rows", 1)
        return mla_inputs(w["max_rows"], R, w["heads"], w["kv_rank"], w["qk_nope"], w["qk_rope"],
                          w["v_head_dim"], w["seed"], new_rows=R)
    vhd = w.get("vHeadDim", w["headDim"])
    if w["kind"] == "decode":
        return decode_inputs(w["max_rows"], w["heads"], w["kvHeads"],
                             w["headDim"], vhd, w["seed"], sigma=w.get("sigma", 1.0),
                             rows=w.get("rows", 1))
    return attention_inputs(w["T"], w["S"], w["heads"], w["kvHeads"],
                            w["headDim"], vhd, w["seed"],
                            sigma=w.get("sigma", 1.0), bias=w.get("bias"),
                            bias_mask_p=w.get("bias_mask_p", 0.0))
