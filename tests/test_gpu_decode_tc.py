"""The tensor-core decode kernel (several query rows against a KV cache,
headDim 128, scores and P.V on tcgen05 in 3xTF32) against the CPU oracle: op "attention" of the
op catalog (vtmu.mpakt.dev/api/ops) with GQA, causal masking per query row,
window and attention sinks.  Tolerance 1e-4 absolute (outputs of order 1);
the cache rows a decode step writes are compared bit for bit."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import TOL, gpu_attention, max_err, oracle_params, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import f32_gqa_attention_gb300 as vtmu  # noqa: E402

DECODE_TC = vtmu.VTMU_KERNEL_DECODE_TF32X3


def check(x, params, tol=TOL):
    out = gpu_attention(x["q"], x["k"], x["v"], x.get("bias"), **params)
    ref = oracle.attention(x["q"], x["k"], x["v"], x.get("bias"), **oracle_params(params))
    assert out.shape == ref.shape and np.all(np.isfinite(out))
    err = max_err(out, ref)
    assert err <= tol, f"max |err| {err:.3e} > {tol} for {params}"
    assert vtmu.vtmu_device_error() == 0
    return out, ref


@pytest.mark.parametrize("G,T", [(1, 1), (1, 2), (1, 16), (2, 3), (2, 8), (4, 2), (4, 4), (4, 3), (8, 2),
                                 (16, 1)])
@pytest.mark.parametrize("feat", ["plain", "window", "noncausal", "sinks", "scale"])
def test_decode_tc_query_rows(G, T, feat):
    """Query rows x group heads as the MMA's N side (up to 16 virtual heads
    per KV head, padded heads masked); S ragged against the 128-row tiles;
    each row masks the keys of the shared range it cannot see."""
    Hk = 3 if G <= 4 else 2
    H = G * Hk
    D = 128
    S = 700 + 29 * T + 13 * G
    pos = S - T - 30 + (17 if feat == "noncausal" else 0)
    x = si.attention_inputs(T, S, H, Hk, D, D, 3000 + 17 * G + T)
    params = dict(heads=H, headDim=D, kvHeads=Hk, posOffset=pos, kernel=DECODE_TC)
    if feat == "window":
        params["window"] = 1 + 3 * T + 200
    elif feat == "noncausal":
        params.update(causal=False, window=150)
    elif feat == "sinks":
        params.update(window=300, sinks=20)
    elif feat == "scale":
        params["scale"] = 0.3
    check(x, params)


@pytest.mark.parametrize("T,S,pos,extra", [
    (4, 1, 0, {}),                                # one key
    (4, 100, 96, {}),                             # a single partial tile
    (2, 129, 127, {}),                            # two tiles, the second one row long
    (3, 256, 253, {}),                            # exactly two tiles
    (4, 2000, 1996, dict(window=64, sinks=300)),  # the sink range overlaps the window's
    (4, 5000, 4990, dict(window=700, sinks=64)),  # sinks as splits of their own
    (2, 300, 296, dict(window=50, sinks=500)),    # sinks past every key
])
def test_decode_tc_tile_and_split_edges(T, S, pos, extra):
    H, Hk, D = 16, 4, 128
    x = si.attention_inputs(T, S, H, Hk, D, D, 3100 + S + T)
    check(x, dict(heads=H, headDim=D, kvHeads=Hk, posOffset=pos, kernel=DECODE_TC, **extra))


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 47])
def test_decode_tc_forced_splits(splits):
    """Long runs of tiles per CTA (47 tiles in one split: 23 and 24 per
    softmax group) down to one tile per split."""
    T, S, H, Hk, D = 4, 6000, 16, 4, 128
    x = si.attention_inputs(T, S, H, Hk, D, D, 3150 + splits)
    check(x, dict(heads=H, headDim=D, kvHeads=Hk, posOffset=S - T, kernel=DECODE_TC, decode_splits=splits))


def test_decode_tc_nothing_visible_gives_zeros():
    """Rows whose window ends before the cache starts see no key: zeros."""
    T, S, H, Hk, D = 3, 400, 8, 2, 128
    x = si.attention_inputs(T, S, H, Hk, D, D, 3201)
    out = gpu_attention(x["q"], x["k"], x["v"], heads=H, headDim=D, kvHeads=Hk, posOffset=S + 500,
                        causal=False, window=20, kernel=DECODE_TC)
    assert np.array_equal(out, np.zeros((T, H * D), np.float32))


def test_decode_tc_large_magnitudes():
    """Scores spread over about a thousand (inputs x 4, scale 1): the lazy
    reference max and the split merge keep every weight finite.  The bound
    comes from f32 itself: a score of magnitude s (in log2 units) carries a
    rounding error of order s 2^-24, which moves a weight by that fraction
    and the output by that times max |v|; the test allows 2^-23 s_max v_max."""
    T, S, H, Hk, D = 4, 3000, 16, 4, 128
    x = si.attention_inputs(T, S, H, Hk, D, D, 3202)
    x = {k: v * 4.0 for k, v in x.items()}
    q = x["q"].astype(np.float64).reshape(T, Hk, H // Hk, D)
    k = x["k"].astype(np.float64).reshape(S, Hk, D)
    s_max = float(np.max(np.abs(np.einsum("tkgd,skd->tkgs", q, k)))) / np.log(2.0)
    tol = 2.0 ** -23 * s_max * float(np.max(np.abs(x["v"])))
    check(x, dict(heads=H, headDim=D, kvHeads=Hk, posOffset=S - T, scale=1.0, kernel=DECODE_TC), tol=tol)


def test_decode_tc_agrees_with_cuda_core_decode():
    """The same 4-row step on both decode kernels."""
    T, S, H, Hk, D = 4, 6000, 32, 8, 128
    x = si.attention_inputs(T, S, H, Hk, D, D, 3203)
    p = dict(heads=H, headDim=D, kvHeads=Hk, posOffset=S - T)
    o1 = gpu_attention(x["q"], x["k"], x["v"], kernel=DECODE_TC, **p)
    o2 = gpu_attention(x["q"], x["k"], x["v"], kernel=vtmu.VTMU_KERNEL_DECODE, **p)
    assert max_err(o1, o2) <= TOL


def _step(S, H, Hk, D, T, offset, seed, shift=0, **params):
    """A decode step (cache_write of T rows at `offset`, attention of T rows);
    `shift` floats of offset make the new-row buffers 4- but not 16-byte
    aligned (the rows then go in by the cache_write kernel)."""
    g = si.Stream(seed)
    q = g.normal_f32(T * H * D).reshape(T, H * D)
    kc = g.normal_f32(S * Hk * D).reshape(S, Hk * D)
    vc = g.normal_f32(S * Hk * D).reshape(S, Hk * D)
    kn = g.normal_f32(T * Hk * D).reshape(T, Hk * D)
    vn = g.normal_f32(T * Hk * D).reshape(T, Hk * D)

    def dev_shifted(a):
        buf = torch.zeros(a.size + shift, dtype=torch.float32, device="cuda")
        buf[shift:] = torch.from_numpy(a.ravel()).cuda()
        return buf[shift:].view(a.shape)

    Kc, Vc = to_dev(kc), to_dev(vc)
    out = vtmu.decode_step(Kc, Vc, dev_shifted(kn), dev_shifted(vn), offset, to_dev(q), heads=H, headDim=D,
                           kvHeads=Hk, kernel=DECODE_TC, **params)
    torch.cuda.synchronize()
    oracle.cache_write(kc, kn, offset)
    oracle.cache_write(vc, vn, offset)
    assert Kc.cpu().numpy().tobytes() == kc.tobytes() and Vc.cpu().numpy().tobytes() == vc.tobytes()
    pos = params.pop("posOffset", offset)
    ref = oracle.attention(q, kc, vc, heads=H, headDim=D, kvHeads=Hk, posOffset=pos, **params)
    assert max_err(out.cpu().numpy(), ref) <= TOL
    assert vtmu.vtmu_device_error() == 0


@pytest.mark.parametrize("shift", [0, 1])
def test_decode_tc_step_writes_rows(shift):
    """The step's new rows (fused into the query split when 16-byte aligned)."""
    _step(3000, 32, 8, 128, 4, 2996, 3210 + shift, shift=shift)
    _step(900, 8, 4, 128, 2, 500, 3212 + shift, shift=shift, posOffset=898)


def test_decode_tc_refuses_what_it_does_not_cover():
    x = si.attention_inputs(4, 300, 32, 4, 128, 128, 3220)  # group 8 x 4 rows = 32 virtual heads
    with pytest.raises(vtmu.VtmuError) as e:
        gpu_attention(x["q"], x["k"], x["v"], heads=32, headDim=128, kvHeads=4, posOffset=296, kernel=DECODE_TC)
    assert e.value.status == vtmu.VTMU_ERR_UNSUPPORTED
    x = si.attention_inputs(2, 300, 4, 2, 128, 128, 3221)
    with pytest.raises(vtmu.VtmuError) as e:
        gpu_attention(x["q"], x["k"], x["v"], heads=4, headDim=128, kvHeads=2, posOffset=298, softcap=30.0,
                      kernel=DECODE_TC)
    assert e.value.status == vtmu.VTMU_ERR_UNSUPPORTED


def test_decode_kernels_share_a_workspace():
    """The CUDA-core decode and the tensor-core decode keep their arrival
    counters in the same workspace header, each leaving them at zero: calls of
    both kinds and of different shapes in a row on one workspace all stay
    correct."""
    ws = vtmu.Workspace()
    cases = [
        (4, 3000, 32, 8, DECODE_TC),
        (1, 3000, 32, 8, vtmu.VTMU_KERNEL_DECODE),
        (2, 1500, 16, 4, DECODE_TC),
        (3, 2000, 8, 8, vtmu.VTMU_KERNEL_DECODE),
        (4, 3000, 32, 8, DECODE_TC),
    ]
    # One buffer for all of them (a workspace that grows is a new, zeroed one).
    ws.get(max(vtmu.vtmu_attention_workspace_size(
        vtmu.make_params(T, S, heads=H, headDim=128, kvHeads=Hk, posOffset=S - T, kernel=kern))
        for T, S, H, Hk, kern in cases))
    first = ws.buf
    for i, (T, S, H, Hk, kern) in enumerate(cases):
        x = si.attention_inputs(T, S, H, Hk, 128, 128, 3300 + i)
        check(x, dict(heads=H, headDim=128, kvHeads=Hk, posOffset=S - T, kernel=kern, workspace=ws))
    assert ws.buf is first
