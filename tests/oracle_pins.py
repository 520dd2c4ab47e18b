"""Pins of the CPU oracle to facts fixed outside it.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with something the op catalog (vtmu.mpakt.dev/api/ops, ops
"attention", "softcap", "softmax", "cache_write", "rope"), the IR schema page
($defs.op_mla_attention, absorbed latent attention) or plain mathematics fixes:
hand-worked examples, closed forms, limits, invariants, a library routine
(PyTorch's float64 ``scaled_dot_product_attention``) on the cases it can
express, and exact rational brute force.  ``test_oracle_pins.py`` runs them on
the oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle with a
planted mistake and expects each copy to fail at least one pin.
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_SYMBOLS = {"L3": math.log(3.0), "L2": math.log(2.0), "L3m1": math.log(3.0) - 1.0}


def _sym(x):
    if isinstance(x, list):
        return [_sym(e) for e in x]
    if isinstance(x, str):
        return _SYMBOLS[x]
    return x


def visible(causal, window, p, s, sinks=0):
    """The op catalog's visibility rule, written from its `window` text, with
    the IR page's attention sinks (keys before `sinks` escape the window)."""
    if causal and s > p:
        return False
    if window:
        if s < sinks:
            return True
        if causal:
            return p - window < s
        return abs(p - s) <= window
    return True


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- hand examples
def pin_hand_examples(orc):
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        params = {k: _sym(v) for k, v in c["params"].items()}
        bias = None if "bias" not in c else np.asarray(_sym(c["bias"]), np.float32)
        out = orc.attention(np.asarray(_sym(c["q"]), np.float32),
                            np.asarray(_sym(c["k"]), np.float32),
                            np.asarray(_sym(c["v"]), np.float32), bias, **params)
        want = np.asarray(c["expected"], np.float64)
        err = np.max(np.abs(out - want))
        assert err <= c["tol"], f"{c['name']}: err {err} > {c['tol']} ({out} vs {want})"


# ---------------------------------------------------------------------- slopes
def pin_bloom_slopes(orc):
    got8 = orc.alibi_slopes(8, alibi=True)
    assert np.array_equal(got8, [2.0 ** -i for i in range(1, 9)]), got8
    want12 = [2.0 ** -i for i in range(1, 9)] + [2.0 ** -0.5, 2.0 ** -1.5,
                                                 2.0 ** -2.5, 2.0 ** -3.5]
    assert np.allclose(orc.alibi_slopes(12, alibi=True), want12, rtol=0, atol=1e-15)
    assert np.allclose(orc.alibi_slopes(3, alibi=True), [1 / 16, 1 / 256, 1 / 4],
                       rtol=0, atol=1e-15)
    assert np.allclose(orc.alibi_slopes(1, alibi=True), [1 / 256], rtol=0, atol=1e-15)


def pin_mpt_slopes(orc):
    # A power-of-two head count takes 2^(-b i / n) directly.
    assert np.allclose(orc.alibi_slopes(4, alibiMax=16.0),
                       [2.0 ** -4, 2.0 ** -8, 2.0 ** -12, 2.0 ** -16], rtol=0, atol=1e-18)
    # With b = 8 the MPT sequence (evens then odds of a 2^ceil grid) is the
    # BLOOM sequence for every head count: a_{2i} = 2^(-8i/c), a_{2j-1} =
    # 2^(-4(2j-1)/c) when n = 2c.
    for h in (1, 2, 3, 5, 6, 7, 8, 12, 20, 40, 96):
        a = orc.alibi_slopes(h, alibiMax=8.0)
        b = orc.alibi_slopes(h, alibi=True)
        assert np.allclose(a, b, rtol=1e-14, atol=0), (h, a, b)
    # A non-power-of-two count with b != 8: n = 4, a = 2^-1, 2^-2, 2^-3, 2^-4,
    # reordered to a2, a4, a1.
    assert np.allclose(orc.alibi_slopes(3, alibiMax=4.0), [2.0 ** -2, 2.0 ** -4, 2.0 ** -1],
                       rtol=0, atol=1e-18)


# ----------------------------------------------------------------- closed forms
def pin_zero_query_is_mean_of_visible(orc):
    g = _rng(11)
    for causal, window, T, S, pos in ((True, None, 5, 9, 4), (True, 3, 6, 12, 5),
                                      (False, 2, 4, 10, 3), (False, None, 3, 7, 0),
                                      (True, 1, 3, 8, 2)):
        H, Hk, D, Dv = 2, 1, 3, 5
        q = np.zeros((T, H * D), np.float32)
        k = g.standard_normal((S, Hk * D)).astype(np.float32)
        v = g.standard_normal((S, Hk * Dv)).astype(np.float32)
        out = orc.attention(q, k, v, heads=H, headDim=D, kvHeads=Hk, vHeadDim=Dv,
                            causal=causal, window=window, posOffset=pos)
        for t in range(T):
            vis = [s for s in range(S) if visible(causal, window or 0, pos + t, s)]
            want = v[vis].astype(np.float64).mean(axis=0) if vis else np.zeros(Dv)
            for h in range(H):
                got = out[t, h * Dv:(h + 1) * Dv]
                assert np.max(np.abs(got - want)) < 1e-12, (causal, window, t, got, want)


def pin_single_visible_key(orc):
    g = _rng(12)
    T, S, H, D = 6, 6, 2, 4
    q = g.standard_normal((T, H * D)).astype(np.float32) * 3
    k = g.standard_normal((S, H * D)).astype(np.float32) * 3
    v = g.standard_normal((S, H * D)).astype(np.float32)
    out = orc.attention(q, k, v, heads=H, headDim=D, window=1)
    for t in range(T):
        for h in range(H):
            assert np.array_equal(out[t, h * D:(h + 1) * D], v[t, h * D:(h + 1) * D].astype(np.float64))


def pin_identical_keys(orc):
    g = _rng(13)
    T, S, H, D = 4, 7, 3, 4
    q = g.standard_normal((T, H * D)).astype(np.float32)
    krow = g.standard_normal((1, H * D)).astype(np.float32)
    k = np.repeat(krow, S, axis=0)
    v = g.standard_normal((S, H * D)).astype(np.float32)
    out = orc.attention(q, k, v, heads=H, headDim=D, causal=False)
    want = np.tile(v.astype(np.float64).mean(axis=0), (T, 1))
    assert np.max(np.abs(out - want)) < 1e-12


def pin_nothing_visible_gives_zeros(orc):
    q = np.ones((2, 4), np.float32)
    k = np.ones((2, 4), np.float32)
    v = np.ones((2, 4), np.float32)
    # positions 10 and 11 with window 3 see keys 8..11, none of which exist.
    out = orc.attention(q, k, v, heads=1, headDim=4, posOffset=10, window=3)
    assert np.array_equal(out, np.zeros((2, 4))), out
    out = orc.attention(q, np.zeros((0, 4), np.float32), np.zeros((0, 4), np.float32),
                        heads=1, headDim=4, causal=False)
    assert np.array_equal(out, np.zeros((2, 4))), out
    # A -inf bias on every key masks the row too.
    b = np.full((2, 2), -np.inf, np.float32)
    out = orc.attention(q, k, v, b, heads=1, headDim=4, causal=False)
    assert np.array_equal(out, np.zeros((2, 4))), out


def pin_large_logits_do_not_overflow(orc):
    # Scores near 1e4: a softmax that is not max-subtracted overflows.
    q = np.full((1, 2), 100.0, np.float32)
    k = np.array([[100.0, 100.0], [99.0, 100.0], [-100.0, 0.0]], np.float32)
    v = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0]], np.float32)
    out = orc.attention(q, k, v, heads=1, headDim=2, scale=1.0, causal=False)
    # key 0 beats key 1 by 100 in the score -> weight ratio e^-100.
    assert np.all(np.isfinite(out)) and np.max(np.abs(out - [[1.0, 2.0]])) < 1e-30


# ---------------------------------------------------------------------- softcap
def pin_softcap_limits(orc):
    g = _rng(14)
    T, S, H, D = 5, 5, 2, 8
    q = g.standard_normal((T, H * D)).astype(np.float32)
    k = g.standard_normal((S, H * D)).astype(np.float32)
    v = g.standard_normal((S, H * D)).astype(np.float32)
    # cap >> |x|: c tanh(x/c) = x - x^3/(3c^2) + ... -> no cap to O(1/c^2).
    a = orc.attention(q, k, v, heads=H, headDim=D, softcap=1e6)
    b = orc.attention(q, k, v, heads=H, headDim=D)
    assert np.max(np.abs(a - b)) < 1e-9
    # |x| >> cap: every score becomes cap * sign(x).
    qb, kb = q * 300.0, k * 300.0
    cap = 2.0
    out = orc.attention(qb, kb, v, heads=H, headDim=D, softcap=cap, causal=False)
    x = np.einsum("thd,shd->hts", qb.astype(np.float64).reshape(T, H, D),
                  kb.astype(np.float64).reshape(S, H, D))
    w = np.exp(cap * np.sign(x))
    want = np.einsum("hts,shd->thd", w / w.sum(-1, keepdims=True),
                     v.astype(np.float64).reshape(S, H, D)).reshape(T, H * D)
    assert np.max(np.abs(out - want)) < 1e-9


# --------------------------------------------------------------- torch library
def _sdpa(q, k, v, bias, *, heads, headDim, kvHeads, vHeadDim, causal, posOffset,
          scale, window, slopes, sinks=0):
    """PyTorch float64 scaled_dot_product_attention with the masks, the ALiBi
    term (absolute form slope * s) and the bias folded into an additive mask."""
    import torch
    T, S = q.shape[0], k.shape[0]
    tq = torch.from_numpy(q.astype(np.float64)).reshape(T, heads, headDim).transpose(0, 1)[None]
    tk = torch.from_numpy(k.astype(np.float64)).reshape(S, kvHeads, headDim).transpose(0, 1)[None]
    tv = torch.from_numpy(v.astype(np.float64)).reshape(S, kvHeads, vHeadDim).transpose(0, 1)[None]
    mask = np.zeros((heads, T, S), np.float64)
    for t in range(T):
        for s in range(S):
            if not visible(causal, window or 0, posOffset + t, s, sinks or 0):
                mask[:, t, s] = -np.inf
    if slopes is not None:
        mask += np.asarray(slopes, np.float64)[:, None, None] * np.arange(S)[None, None, :]
    if bias is not None:
        mask += bias.astype(np.float64) if bias.ndim == 3 else bias.astype(np.float64)[None]
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=torch.from_numpy(mask)[None], scale=scale,
        enable_gqa=(heads != kvHeads))
    return o[0].transpose(0, 1).reshape(T, heads * vHeadDim).numpy()


def pin_torch_sdpa(orc):
    g = _rng(15)
    cases = [
        dict(T=7, S=7, heads=4, kvHeads=2, headDim=8, vHeadDim=8, causal=True, posOffset=0),
        dict(T=3, S=11, heads=6, kvHeads=3, headDim=5, vHeadDim=9, causal=True, posOffset=8),
        dict(T=5, S=9, heads=4, kvHeads=1, headDim=16, vHeadDim=16, causal=False, posOffset=2,
             window=2),
        dict(T=6, S=13, heads=2, kvHeads=2, headDim=4, vHeadDim=4, causal=True, posOffset=7,
             window=4, scale=0.3),
        dict(T=4, S=6, heads=3, kvHeads=3, headDim=6, vHeadDim=2, causal=False, posOffset=0,
             bias="ts"),
        dict(T=4, S=8, heads=4, kvHeads=2, headDim=8, vHeadDim=12, causal=True, posOffset=4,
             bias="hts", slopes=True),
        dict(T=9, S=9, heads=8, kvHeads=8, headDim=4, vHeadDim=4, causal=True, posOffset=0,
             slopes=True),
        dict(T=6, S=20, heads=4, kvHeads=2, headDim=8, vHeadDim=8, causal=True, posOffset=12,
             window=3, sinks=4),
        dict(T=5, S=16, heads=2, kvHeads=1, headDim=4, vHeadDim=6, causal=False, posOffset=9,
             window=2, sinks=3, bias="ts"),
        dict(T=8, S=8, heads=2, kvHeads=2, headDim=4, vHeadDim=4, causal=True, posOffset=0,
             window=2, sinks=5),
    ]
    for c in cases:
        T, S, H, Hk = c["T"], c["S"], c["heads"], c["kvHeads"]
        D, Dv = c["headDim"], c["vHeadDim"]
        q = g.standard_normal((T, H * D)).astype(np.float32)
        k = g.standard_normal((S, Hk * D)).astype(np.float32)
        v = g.standard_normal((S, Hk * Dv)).astype(np.float32)
        bias = None
        if c.get("bias") == "ts":
            bias = g.standard_normal((T, S)).astype(np.float32)
        elif c.get("bias") == "hts":
            bias = g.standard_normal((H, T, S)).astype(np.float32)
        slopes = g.uniform(0.01, 0.7, H) if c.get("slopes") else None
        scale = c.get("scale")
        out = orc.attention(q, k, v, bias, heads=H, headDim=D, kvHeads=Hk, vHeadDim=Dv,
                            causal=c["causal"], posOffset=c["posOffset"], scale=scale,
                            window=c.get("window"), alibiSlopes=slopes, sinks=c.get("sinks"))
        want = _sdpa(q, k, v, bias, heads=H, headDim=D, kvHeads=Hk, vHeadDim=Dv,
                     causal=c["causal"], posOffset=c["posOffset"],
                     scale=(1.0 / math.sqrt(D)) if scale is None else scale,
                     window=c.get("window"), slopes=slopes, sinks=c.get("sinks"))
        err = np.max(np.abs(out - want))
        assert err < 1e-10, (c, err)


# ------------------------------------------------------------------- invariants
def pin_gqa_equals_repeated_kv(orc):
    g = _rng(16)
    T, S, H, Hk, D, Dv = 5, 8, 6, 2, 4, 6
    G = H // Hk
    q = g.standard_normal((T, H * D)).astype(np.float32)
    k = g.standard_normal((S, Hk * D)).astype(np.float32)
    v = g.standard_normal((S, Hk * Dv)).astype(np.float32)
    gqa = orc.attention(q, k, v, heads=H, headDim=D, kvHeads=Hk, vHeadDim=Dv, posOffset=3)
    kr = np.repeat(k.reshape(S, Hk, D), G, axis=1).reshape(S, H * D)
    vr = np.repeat(v.reshape(S, Hk, Dv), G, axis=1).reshape(S, H * Dv)
    mha = orc.attention(q, kr, vr, heads=H, headDim=D, vHeadDim=Dv, posOffset=3)
    assert np.max(np.abs(gqa - mha)) < 1e-13


def pin_bias_mask_drops_key(orc):
    g = _rng(17)
    T, S, H, D = 4, 9, 2, 4
    q = g.standard_normal((T, H * D)).astype(np.float32)
    k = g.standard_normal((S, H * D)).astype(np.float32)
    v = g.standard_normal((S, H * D)).astype(np.float32)
    drop = [1, 4, 5]
    bias = np.zeros((T, S), np.float32)
    bias[:, drop] = -1e9
    a = orc.attention(q, k, v, bias, heads=H, headDim=D, causal=False)
    keep = [s for s in range(S) if s not in drop]
    b = orc.attention(q, k[keep], v[keep], heads=H, headDim=D, causal=False)
    assert np.max(np.abs(a - b)) < 1e-12


def pin_decode_is_last_prefill_row(orc):
    g = _rng(18)
    H, Hk, D = 4, 2, 8
    p = 12
    Smax = 20  # cache longer than the position: keys beyond it are future ones
    q = g.standard_normal((p + 1, H * D)).astype(np.float32)
    k = g.standard_normal((Smax, Hk * D)).astype(np.float32)
    v = g.standard_normal((Smax, Hk * D)).astype(np.float32)
    full = orc.attention(q, k[:p + 1], v[:p + 1], heads=H, headDim=D, kvHeads=Hk)
    for window in (None, 5):
        full = orc.attention(q, k[:p + 1], v[:p + 1], heads=H, headDim=D, kvHeads=Hk,
                             window=window)
        dec = orc.attention(q[p:p + 1], k, v, heads=H, headDim=D, kvHeads=Hk,
                            posOffset=p, window=window)
        assert np.max(np.abs(dec[0] - full[p])) < 1e-13


def pin_alibi_shift_invariance(orc):
    # slope*(s - p) and the BLOOM absolute form slope*s differ by a per-row
    # constant; the softmax removes it.  Here the absolute form is supplied
    # as an explicit bias.
    g = _rng(19)
    T, S, H, D = 5, 9, 4, 4
    q = g.standard_normal((T, H * D)).astype(np.float32)
    k = g.standard_normal((S, H * D)).astype(np.float32)
    v = g.standard_normal((S, H * D)).astype(np.float32)
    slopes = orc.alibi_slopes(H, alibi=True)
    a = orc.attention(q, k, v, heads=H, headDim=D, alibi=True, posOffset=4)
    bias = (slopes[:, None, None] * np.arange(S)[None, None, :]).repeat(T, axis=1)
    b = orc.attention(q, k, v, bias.astype(np.float32), heads=H, headDim=D, posOffset=4)
    # the bias is rounded to f32 (|slope*s| < 4.5, error < 3e-7 in a score)
    assert np.max(np.abs(a - b)) < 2e-6


# ---------------------------------------------------------- rational brute force
def pin_rational_brute_force(orc):
    """D = 1, q = 1, scale = 1 and k_s = ln(n_s): exp(score) = n_s, so every
    output is the rational sum(n_s v_s) / sum(n_s) over the visible keys."""
    g = _rng(20)
    for trial in range(12):
        T = int(g.integers(1, 6))
        S = int(g.integers(1, 7))
        causal = bool(trial % 2)
        window = int(g.integers(0, 4))
        pos = int(g.integers(0, 4))
        n = g.integers(1, 10, size=S)
        vint = g.integers(-9, 10, size=S)
        q = np.ones((T, 1), np.float32)
        k = np.log(n.astype(np.float64)).astype(np.float32).reshape(S, 1)
        v = vint.astype(np.float32).reshape(S, 1)
        out = orc.attention(q, k, v, heads=1, headDim=1, scale=1.0, causal=causal,
                            window=window, posOffset=pos)
        for t in range(T):
            vis = [s for s in range(S) if visible(causal, window, pos + t, s)]
            if vis:
                want = Fraction(sum(int(n[s]) * int(vint[s]) for s in vis),
                                sum(int(n[s]) for s in vis))
            else:
                want = Fraction(0)
            assert abs(out[t, 0] - float(want)) < 2e-6, (trial, t, out[t, 0], want)


# ------------------------------------------------------------------ cache_write
def pin_cache_write(orc):
    cache = np.full((6, 3), 7.5, np.float32)
    vals = np.arange(6, dtype=np.float32).reshape(2, 3)
    orc.cache_write(cache, vals, 3)
    want = np.full((6, 3), 7.5, np.float32)
    want[3:5] = vals
    assert np.array_equal(cache, want)
    for bad in (5, -1):
        try:
            orc.cache_write(cache, vals, bad)
        except ValueError:
            pass
        else:
            raise AssertionError(f"offset {bad} must be refused")
    orc.cache_write(cache, np.zeros((0, 3), np.float32), 6)  # empty write at the end
    assert np.array_equal(cache, want)


# ------------------------------------------------------------------------ rope
# op "rope" of the same page: rotary position embedding over [T, heads*headDim].
def pin_rope_hand_examples(orc):
    with open(os.path.join(GOLDEN, "rope_hand_examples.json")) as f:
        doc = json.load(f)
    for c in doc["cases"]:
        out = orc.rope(np.asarray(c["x"], np.float32), **c["params"])
        want = np.asarray(c["expected"], np.float64)
        err = np.max(np.abs(out - want))
        assert err <= doc["tol"], f"{c['name']}: err {err} ({out} vs {want})"


def _pairs(headDim, rd, interleaved):
    half = rd // 2
    return [((2 * j, 2 * j + 1) if interleaved else (j, j + half)) for j in range(half)]


def pin_rope_relative_position(orc):
    """The defining property of rotary embeddings: the dot product of a query
    at position m with a key at position n depends on m - n only (per head, on
    the rotated channels; the pass-through channels add a constant)."""
    g = _rng(41)
    D, H = 10, 2
    for interleaved in (False, True):
        q = g.standard_normal((1, H * D)).astype(np.float32)
        k = g.standard_normal((1, H * D)).astype(np.float32)
        kw = dict(headDim=D, rotaryDim=8, interleaved=interleaved, base=500.0)
        dots = []
        for m, n in ((7, 3), (40, 36), (1004, 1000)):
            a = orc.rope(q, offset=m, **kw).reshape(H, D)
            b = orc.rope(k, offset=n, **kw).reshape(H, D)
            dots.append(np.sum(a * b, axis=1))
        assert np.allclose(dots[0], dots[1], rtol=0, atol=1e-9), dots
        assert np.allclose(dots[0], dots[2], rtol=0, atol=1e-9), dots
        # and a different offset changes it
        c = orc.rope(q, offset=8, **kw).reshape(H, D)
        assert not np.allclose(np.sum(c * orc.rope(k, offset=3, **kw).reshape(H, D), axis=1), dots[0])


def pin_rope_norm_and_pass_through(orc):
    """Each pair is rotated (its norm times attentionFactor); channels past
    rotaryDim come out unchanged."""
    g = _rng(42)
    D, H, rd, af = 12, 3, 8, 1.5
    x = g.standard_normal((5, H * D)).astype(np.float32)
    for interleaved in (False, True):
        out = orc.rope(x, headDim=D, rotaryDim=rd, interleaved=interleaved, offset=17,
                       attentionFactor=af).reshape(5, H, D)
        xr = x.astype(np.float64).reshape(5, H, D)
        assert np.array_equal(out[:, :, rd:], xr[:, :, rd:])
        for a, b in _pairs(D, rd, interleaved):
            n_in = np.hypot(xr[:, :, a], xr[:, :, b])
            n_out = np.hypot(out[:, :, a], out[:, :, b])
            assert np.allclose(n_out, af * n_in, rtol=1e-12, atol=1e-12)
        assert not np.allclose(out[:, :, :rd], af * xr[:, :, :rd])  # it does turn


def pin_rope_interleaved_is_permuted_half_split(orc):
    """Interleaved pairing is half-split pairing on permuted channels: the
    permutation sending channel 2j -> j and 2j+1 -> j + rd/2 conjugates one
    into the other."""
    g = _rng(43)
    D, H, rd = 8, 2, 8
    perm = np.array([2 * j for j in range(rd // 2)] + [2 * j + 1 for j in range(rd // 2)])
    x = g.standard_normal((3, H * D)).astype(np.float32)
    xi = x.reshape(3, H, D)
    xh = xi[:, :, perm].reshape(3, H * D)  # half-split order
    a = orc.rope(x, headDim=D, interleaved=True, offset=9).reshape(3, H, D)
    b = orc.rope(xh, headDim=D, interleaved=False, offset=9).reshape(3, H, D)
    assert np.allclose(a[:, :, perm], b, rtol=0, atol=1e-12)


def pin_rope_linear_scaling_and_inv_freq(orc):
    """Linear scaling by f at position f*p equals no scaling at p; explicit
    inverse frequencies equal to the base-derived ones change nothing."""
    g = _rng(44)
    x = g.standard_normal((3, 2 * 16)).astype(np.float32)
    plain = orc.rope(x, headDim=16, offset=6)
    lin = orc.rope(x, headDim=16, offset=18, scaling={"rope_type": "linear", "factor": 3.0})
    assert np.allclose(plain[0], lin[0], rtol=0, atol=1e-12)  # row 0: 18 / 3 = 6
    inv = [10000.0 ** (-2.0 * j / 16) for j in range(8)]
    assert np.allclose(orc.rope(x, headDim=16, offset=6, invFreq=inv), plain, rtol=0, atol=1e-12)


# ------------------------------------------------------- absorbed latent attention
def _mla_inputs(g, T, S, H, R, N, P, Dv):
    q = g.standard_normal((T, H * (N + P))).astype(np.float32)
    state = g.standard_normal((S, R + P)).astype(np.float32)
    k_b = (g.standard_normal((H * N, R)) / math.sqrt(R)).astype(np.float32)
    v_b = (g.standard_normal((H * Dv, R)) / math.sqrt(R)).astype(np.float32)
    return q, state, k_b, v_b


def pin_mla_hand_examples(orc):
    with open(os.path.join(GOLDEN, "mla_hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        out = orc.mla_attention(*(np.asarray(_sym(c[n]), np.float32) for n in ("q", "state", "k_b", "v_b")),
                                **c["params"])
        err = np.max(np.abs(out - np.asarray(c["expected"], np.float64)))
        assert err <= c["tol"], f"{c['name']}: err {err} > {c['tol']} ({out})"


def _mla_absorbed(q, state, k_b, v_b, *, heads, kv_rank, qk_nope, qk_rope, v_head_dim, scale,
                  causal, posOffset, window, sinks):
    """The absorbed order of the same sums, in float64: queries through k_b
    into the latent space, one score against [latent | rotary key] shared by
    every head, the softmax-weighted latent, then v_b."""
    H, R, N, P, Dv = heads, kv_rank, qk_nope, qk_rope, v_head_dim
    T, S = q.shape[0], state.shape[0]
    q64 = q.astype(np.float64).reshape(T, H, N + P)
    c = state[:, :R].astype(np.float64)
    r = state[:, R:].astype(np.float64)
    kb = k_b.astype(np.float64).reshape(H, N, R)
    vb = v_b.astype(np.float64).reshape(H, Dv, R)
    q_lat = np.einsum("thn,hnr->thr", q64[:, :, :N], kb)
    x = scale * (np.einsum("thr,sr->ths", q_lat, c) + np.einsum("thp,sp->ths", q64[:, :, N:], r))
    vis = np.array([[visible(causal, window or 0, posOffset + t, s, sinks or 0) for s in range(S)]
                    for t in range(T)])
    x = np.where(vis[:, None, :], x, -np.inf)
    out = np.zeros((T, H, Dv))
    for t in range(T):
        if not vis[t].any():
            continue
        w = np.exp(x[t] - x[t].max(axis=1, keepdims=True))
        o_lat = (w @ c) / w.sum(axis=1, keepdims=True)
        out[t] = np.einsum("hr,her->he", o_lat, vb)
    return out.reshape(T, H * Dv)


MLA_CASES = [
    dict(T=5, S=9, H=3, R=7, N=4, P=2, Dv=5, causal=True, posOffset=4),
    dict(T=3, S=12, H=2, R=6, N=3, P=4, Dv=2, causal=False, posOffset=0, scale=0.4),
    dict(T=4, S=16, H=4, R=8, N=2, P=2, Dv=3, causal=True, posOffset=12, window=3, sinks=2),
    dict(T=2, S=10, H=1, R=5, N=5, P=1, Dv=6, causal=False, posOffset=5, window=2),
    dict(T=6, S=6, H=2, R=4, N=3, P=3, Dv=4, causal=True, posOffset=0, window=2, sinks=3),
]


def _mla_params(c):
    return dict(heads=c["H"], kv_rank=c["R"], qk_nope=c["N"], qk_rope=c["P"], v_head_dim=c["Dv"],
                causal=c["causal"], posOffset=c["posOffset"], window=c.get("window"), sinks=c.get("sinks"))


def pin_mla_absorbed_equals_unabsorbed(orc):
    """The oracle expands keys and values per head; the absorbed order (the
    GPU's) of the same sums must give the same rows in float64."""
    g = _rng(41)
    for c in MLA_CASES:
        q, state, k_b, v_b = _mla_inputs(g, c["T"], c["S"], c["H"], c["R"], c["N"], c["P"], c["Dv"])
        params = _mla_params(c)
        out = orc.mla_attention(q, state, k_b, v_b, scale=c.get("scale"), **params)
        scale = c.get("scale") or 1.0 / math.sqrt(c["N"] + c["P"])
        want = _mla_absorbed(q, state, k_b, v_b, scale=scale, **params)
        err = np.max(np.abs(out - want))
        assert err < 1e-10, (c, err)


def pin_mla_torch_sdpa(orc):
    """Keys and values expanded with torch (float64), then PyTorch's
    scaled_dot_product_attention with the visibility mask."""
    import torch
    g = _rng(43)
    for c in MLA_CASES:
        T, S, H, R, N, P, Dv = (c[k] for k in ("T", "S", "H", "R", "N", "P", "Dv"))
        q, state, k_b, v_b = _mla_inputs(g, T, S, H, R, N, P, Dv)
        st = torch.from_numpy(state.astype(np.float64))
        lat, rope = st[:, :R], st[:, R:]
        kn = torch.einsum("sr,hnr->hsn", lat, torch.from_numpy(k_b.astype(np.float64)).reshape(H, N, R))
        keys = torch.cat([kn, rope[None].expand(H, S, P)], dim=2)
        vals = torch.einsum("sr,her->hse", lat, torch.from_numpy(v_b.astype(np.float64)).reshape(H, Dv, R))
        tq = torch.from_numpy(q.astype(np.float64)).reshape(T, H, N + P).transpose(0, 1)
        mask = torch.zeros((T, S), dtype=torch.float64)
        for t in range(T):
            for s in range(S):
                if not visible(c["causal"], c.get("window") or 0, c["posOffset"] + t, s, c.get("sinks") or 0):
                    mask[t, s] = -math.inf
        scale = c.get("scale") or 1.0 / math.sqrt(N + P)
        o = torch.nn.functional.scaled_dot_product_attention(tq[None], keys[None], vals[None],
                                                             attn_mask=mask[None, None], scale=scale)
        want = o[0].transpose(0, 1).reshape(T, H * Dv).numpy()
        out = orc.mla_attention(q, state, k_b, v_b, scale=c.get("scale"), **_mla_params(c))
        err = np.max(np.abs(out - want))
        assert err < 1e-10, (c, err)


def pin_mla_identity_up_projections_are_mqa(orc):
    """With k_b and v_b the identity for every head (qk_nope = v_head_dim =
    kv_rank), each head attends to [latent | rotary key] with the latent as
    value: op attention with one KV head (kvHeads 1), which the attention
    pins fix."""
    g = _rng(47)
    for T, S, H, R, P, causal, pos, window in ((4, 9, 3, 5, 2, True, 5, None), (3, 7, 2, 4, 3, False, 0, 3)):
        q = g.standard_normal((T, H * (R + P))).astype(np.float32)
        state = g.standard_normal((S, R + P)).astype(np.float32)
        eye = np.tile(np.eye(R, dtype=np.float32), (H, 1))
        out = orc.mla_attention(q, state, eye, eye, heads=H, kv_rank=R, qk_nope=R, qk_rope=P, v_head_dim=R,
                                causal=causal, posOffset=pos, window=window)
        want = orc.attention(q, state, np.ascontiguousarray(state[:, :R]), heads=H, headDim=R + P, kvHeads=1,
                             vHeadDim=R, causal=causal, posOffset=pos, window=window)
        err = np.max(np.abs(out - want))
        assert err < 1e-12, err


def pin_mla_latent_rotation_invariance(orc):
    """An orthogonal change of the latent basis (c -> c Q, k_b -> k_b Q,
    v_b -> v_b Q) leaves every key and value, and so the output, unchanged;
    permuting the heads (query blocks with their k_b and v_b blocks) permutes
    the output blocks."""
    g = _rng(53)
    T, S, H, R, N, P, Dv = 3, 10, 3, 6, 4, 2, 5
    q, state, k_b, v_b = _mla_inputs(g, T, S, H, R, N, P, Dv)
    params = dict(heads=H, kv_rank=R, qk_nope=N, qk_rope=P, v_head_dim=Dv, causal=True, posOffset=7)
    base = orc.mla_attention(q, state, k_b, v_b, **params)
    Q, _ = np.linalg.qr(g.standard_normal((R, R)))
    st2 = state.astype(np.float64).copy()
    st2[:, :R] = st2[:, :R] @ Q
    rot = orc.mla_attention(q, st2, k_b.astype(np.float64) @ Q, v_b.astype(np.float64) @ Q, **params)
    assert np.max(np.abs(rot - base)) < 1e-5  # the rotated inputs are rounded to f32
    perm = [2, 0, 1]
    qp = q.reshape(T, H, N + P)[:, perm].reshape(T, -1)
    kbp = k_b.reshape(H, N, R)[perm].reshape(H * N, R)
    vbp = v_b.reshape(H, Dv, R)[perm].reshape(H * Dv, R)
    outp = orc.mla_attention(qp, state, kbp, vbp, **params)
    assert np.array_equal(outp.reshape(T, H, Dv), base.reshape(T, H, Dv)[:, perm])


def pin_mla_decode_is_last_prefill_row(orc):
    g = _rng(59)
    T, H, R, N, P, Dv = 6, 2, 5, 3, 2, 4
    q, state, k_b, v_b = _mla_inputs(g, T, T, H, R, N, P, Dv)
    params = dict(heads=H, kv_rank=R, qk_nope=N, qk_rope=P, v_head_dim=Dv)
    full = orc.mla_attention(q, state, k_b, v_b, causal=True, posOffset=0, **params)
    last = orc.mla_attention(q[-1:], state, k_b, v_b, causal=True, posOffset=T - 1, **params)
    assert np.array_equal(last[0], full[-1])
    rows = orc.mla_attention_rows(q, state, k_b, v_b, rows=[(T - 1, 1), (2, 0)], causal=True, posOffset=0,
                                  **params)
    assert np.array_equal(rows[0], full[-1, Dv:]) and np.array_equal(rows[1], full[2, :Dv])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
