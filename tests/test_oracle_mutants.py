"""The oracle's pins are strong enough: a copy of the oracle with one plausible
mistake planted (on the CPU, in a temporary copy of its C source) must fail
at least one pin.  Each mutation names the statement of the op catalog
(vtmu.mpakt.dev/api/ops) that it breaks."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import oracle  # noqa: E402
import oracle_pins  # noqa: E402

# (name, original text, planted text)
MUTANTS = [
    ("kv head by modulo instead of by group (grouped-query mapping)",
     "const int kh = h / G;", "const int kh = h % a->kv_heads;"),
    ("causal window boundary inclusive (pos - window < s)",
     "if (!(p - window < s)) return 0;", "if (!(p - window <= s)) return 0;"),
    ("non-causal window boundary exclusive (|pos - s| <= window)",
     "if (dist > window) return 0;", "if (dist >= window) return 0;"),
    ("causal mask hides the diagonal (s <= pos visible)",
     "if (causal && s > p) return 0;", "if (causal && s >= p) return 0;"),
    ("scale dropped (scale replaces 1/sqrt(headDim))",
     "double xs = a->scale * dot;", "double xs = dot;"),
    ("ALiBi sign flipped",
     "xs += a->slopes[h] * (double)(s - p);", "xs += a->slopes[h] * (double)(p - s);"),
    ("ALiBi dropped",
     "xs += a->slopes[h] * (double)(s - p);", "xs += 0.0;"),
    ("per-head bias indexed [T, heads, S]",
     "bias[((int64_t)h * a->T + t) * a->S + s]", "bias[((int64_t)t * a->heads + h) * a->S + s]"),
    ("bias dropped",
     "xs += (double)bias[t * a->S + s];", "xs += 0.0;"),
    ("softcap applied after the bias (softcap before the mask)", None, None),
    ("softcap without the cap factor",
     "xs = a->softcap * tanh(xs / a->softcap);", "xs = tanh(xs / a->softcap);"),
    ("softmax not max-subtracted",
     "double w = exp(x[s] - m);", "double w = exp(x[s]);"),
    ("value rows strided by headDim",
     "(int64_t)kh * Dv;", "(int64_t)kh * D;"),
    ("posOffset ignored",
     "const int64_t p = a->pos_offset + t;", "const int64_t p = t;"),
    ("no-visible-key row not zeroed",
     "if (m == -INFINITY) return; /* nothing visible: the row is zero */", ""),
    ("BLOOM extra slopes on the wrong grid",
     "out[c + j - 1] = pow(2.0, -4.0 * (2.0 * j - 1.0) / c);",
     "out[c + j - 1] = pow(2.0, -4.0 * (2.0 * j) / c);"),
    ("MPT odd slopes before the even ones",
     "for (int i = 2; i <= n && w < heads; i += 2) out[w++] = a[i - 1];\n"
     "            for (int i = 1; i <= n && w < heads; i += 2) out[w++] = a[i - 1];",
     "for (int i = 1; i <= n && w < heads; i += 2) out[w++] = a[i - 1];\n"
     "            for (int i = 2; i <= n && w < heads; i += 2) out[w++] = a[i - 1];"),
    ("cache_write copies the first row everywhere",
     "= values[r * width + c];", "= values[c];"),
    ("sinks escape causality (sinks keep keys the window drops, not future keys)",
     "    if (causal && s > p) return 0;\n    if (window > 0) {\n        if (s < sinks) return 1;",
     "    if (s < sinks) return 1;\n    if (causal && s > p) return 0;\n    if (window > 0) {"),
    ("sinks ignored",
     "        if (s < sinks) return 1;\n", ""),
    ("rope turns the wrong way (op rope: rotary embedding)",
     "orow[ia] = (double)xr[ia] * c - (double)xr[ib] * s;", "orow[ia] = (double)xr[ia] * c + (double)xr[ib] * s;"),
    ("rope half-split partner i + 1 instead of i + rotaryDim/2",
     "const int ib = interleaved ? 2 * j + 1 : j + half;", "const int ib = interleaved ? 2 * j + 1 : j + 1;"),
    ("rope interleaved flag ignored for the partner",
     "const int ib = interleaved ? 2 * j + 1 : j + half;", "const int ib = interleaved ? j + half : j + half;"),
    ("rope frequencies base^(-j/rotaryDim)",
     "pow(base, -2.0 * (double)j / (double)rotary_dim)", "pow(base, -1.0 * (double)j / (double)rotary_dim)"),
    ("rope attentionFactor on cos only (it multiplies cos and sin)",
     "const double s = sin(theta) * attention_factor;", "const double s = sin(theta);"),
    ("rope pass-through channels dropped (rotaryDim: the rest pass through)",
     "for (int d = rotary_dim; d < head_dim; ++d) orow[d] = xr[d];", ""),
    ("rope offset ignored (offset: position of the first row)",
     "const double position = (double)(offset + t) / pos_divisor;", "const double position = (double)t / pos_divisor;"),
    ("rope linear scaling ignored",
     "const double position = (double)(offset + t) / pos_divisor;", "const double position = (double)(offset + t);"),
    # absorbed latent attention (IR schema page, $defs.op_mla_attention)
    ("mla: rotary key dropped from the keys (qk_rope)",
     "for (int i = 0; i < P; ++i) krow[N + i] = (double)c[R + i];",
     "for (int i = 0; i < P; ++i) krow[N + i] = 0.0;"),
    ("mla: rotary key read from the start of the latent row",
     "for (int i = 0; i < P; ++i) krow[N + i] = (double)c[R + i];",
     "for (int i = 0; i < P; ++i) krow[N + i] = (double)c[i];"),
    ("mla: every head uses head 0's k_b block",
     "const float* w = k_b + ((int64_t)h * N + i) * R;", "const float* w = k_b + ((int64_t)0 * N + i) * R;"),
    ("mla: v_b read as [v_head_dim, heads] rows",
     "const float* w = v_b + ((int64_t)h * Dv + e) * R;", "const float* w = v_b + ((int64_t)e * a->heads + h) * R;"),
    ("mla: query heads strided by qk_nope (q is [T, heads*(qk_nope+qk_rope)])",
     "const float* qrow = q + (t * (int64_t)a->heads + h) * Dq;",
     "const float* qrow = q + (t * (int64_t)a->heads + h) * a->qk_nope;"),
    ("mla: scale dropped",
     "x[s] = a->scale * dot;", "x[s] = dot;"),
    ("mla: posOffset ignored",
     "const int64_t pos = a->pos_offset + t;", "const int64_t pos = t;"),
]


def _plant_softcap_after_bias(src):
    """Move the softcap line after the bias lines."""
    line = "        if (a->softcap > 0.0) xs = a->softcap * tanh(xs / a->softcap);\n"
    assert line in src
    src = src.replace(line, "")
    anchor = "        x[s] = xs;\n"
    assert anchor in src
    return src.replace(anchor, line + anchor)


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    with open(oracle.SOURCE) as f:
        src = f.read()
    if old is None:
        mutated = _plant_softcap_after_bias(src)
    else:
        assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
        mutated = src.replace(old, new)
    assert mutated != src
    c_path = tmp_path / "mutant.c"
    c_path.write_text(mutated)
    so = oracle.compile_source(str(c_path), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(so)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, FloatingPointError) as e:
            failed.append((pin.__name__, str(e)[:80]))
    assert failed, f"no pin caught the planted mistake: {name}"
