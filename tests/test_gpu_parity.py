"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.  Floating-point outputs must agree within 1e-4
(absolute); cache_write must be bit-exact."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import TOL, gpu_attention, max_err, oracle_params, sample_rows, sample_tile_rows, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import f32_gqa_attention_gb300 as vtmu  # noqa: E402

DECODE = vtmu.VTMU_KERNEL_DECODE
FFMA = vtmu.VTMU_KERNEL_PREFILL_FFMA


def check(inputs, params, tol=TOL):
    out = gpu_attention(inputs["q"], inputs["k"], inputs["v"], inputs.get("bias"), **params)
    ref = oracle.attention(inputs["q"], inputs["k"], inputs["v"], inputs.get("bias"), **oracle_params(params))
    err = max_err(out, ref)
    assert out.shape == ref.shape
    assert np.all(np.isfinite(out))
    assert err <= tol, f"max |err| {err:.3e} > {tol} for {params}"
    return out, ref


# ------------------------------------------------------------------ workloads
def test_tiny_prefill_workload():
    w = si.WORKLOADS["tiny_prefill"]
    check(si.workload_inputs("tiny_prefill"),
          dict(heads=w["heads"], headDim=w["headDim"], kvHeads=w["kvHeads"], **w["params"]))


def test_gqa_decode_workload():
    """cache_write one row at 32767 into [32768, 1024] K/V caches, then T=1
    attention over all 32768 keys (32 heads, 8 KV heads, headDim 128)."""
    w = si.WORKLOADS["gqa_decode"]
    x = si.workload_inputs("gqa_decode")
    H, Hk, D, off = w["heads"], w["kvHeads"], w["headDim"], w["offset"]
    Kc, Vc = to_dev(x["kc"]), to_dev(x["vc"])
    vtmu.cache_write(Kc, to_dev(x["k_new"]), off)
    vtmu.cache_write(Vc, to_dev(x["v_new"]), off)
    out = vtmu.attention(to_dev(x["q"]), Kc, Vc, heads=H, headDim=D, kvHeads=Hk, **w["params"])
    torch.cuda.synchronize()
    oracle.cache_write(x["kc"], x["k_new"], off)
    oracle.cache_write(x["vc"], x["v_new"], off)
    assert torch.equal(Kc.cpu(), torch.from_numpy(x["kc"]))
    assert torch.equal(Vc.cpu(), torch.from_numpy(x["vc"]))
    ref = oracle.attention(x["q"], x["kc"], x["vc"], heads=H, headDim=D, kvHeads=Hk, **w["params"])
    err = max_err(out.cpu().numpy(), ref)
    assert err <= TOL, err


@pytest.mark.parametrize("name", ["gqa_spec_decode", "gqa_decode_sinks"])
def test_decode_step_workloads(name):
    """The 4-row speculative step and the windowed step with sinks at full size, as the
    bench runs them: one fused vtmu_decode_step (cache_write of the new rows + attention)."""
    w = si.WORKLOADS[name]
    x = si.workload_inputs(name)
    H, Hk, D, off, R = w["heads"], w["kvHeads"], w["headDim"], w["offset"], w.get("rows", 1)
    Kc, Vc = to_dev(x["kc"]), to_dev(x["vc"])
    out = vtmu.decode_step(Kc, Vc, to_dev(x["k_new"]), to_dev(x["v_new"]), off, to_dev(x["q"]), heads=H,
                           headDim=D, kvHeads=Hk, **w["params"])
    torch.cuda.synchronize()
    oracle.cache_write(x["kc"], x["k_new"], off)
    oracle.cache_write(x["vc"], x["v_new"], off)
    assert torch.equal(Kc.cpu(), torch.from_numpy(x["kc"]))
    assert torch.equal(Vc.cpu(), torch.from_numpy(x["vc"]))
    assert out.shape == (R, H * D)
    ref = oracle.attention(x["q"], x["kc"], x["vc"], heads=H, headDim=D, kvHeads=Hk, **w["params"])
    err = max_err(out.cpu().numpy(), ref)
    assert err <= TOL, err
    assert vtmu.vtmu_device_error() == 0


@pytest.mark.parametrize("name", ["gqa_prefill", "swa_softcap_prefill", "latent_bias_prefill",
                                  "alibi_prefill", "swa_sinks_prefill"])
def test_prefill_workload_sampled_rows(name):
    """Full-size prefill on the GPU; the oracle recomputes sampled (t, h) rows:
    the first and last rows, tile edges and random rows, plus one row of
    every 128-row query tile for four heads (every output column of a row is
    compared, so both vHeadDim halves of a headDim-256 launch are covered)."""
    w = si.WORKLOADS[name]
    x = si.workload_inputs(name)
    params = dict(heads=w["heads"], headDim=w["headDim"], kvHeads=w["kvHeads"],
                  vHeadDim=w.get("vHeadDim"), **w["params"])
    out = gpu_attention(x["q"], x["k"], x["v"], x.get("bias"), **params)
    assert np.all(np.isfinite(out))
    H, Dv = w["heads"], w.get("vHeadDim") or w["headDim"]
    G = H // w["kvHeads"]
    rows = sample_rows(w["T"], H, G, seed=1) + sample_tile_rows(w["T"], H, G, seed=2)
    ref = oracle.attention_rows(x["q"], x["k"], x["v"], x.get("bias"), rows=rows, **params)
    got = np.stack([out[t, h * Dv:(h + 1) * Dv] for t, h in rows])
    err = max_err(got, ref)
    assert err <= TOL, f"{name}: max |err| {err:.3e}"


# --------------------------------------------------------------- random sweep
def _case(seed):
    g = np.random.default_rng(1000 + seed)
    H, Hk = [(1, 1), (4, 1), (4, 2), (6, 3), (8, 8), (8, 2)][seed % 6]
    D = int(g.choice([1, 4, 8, 32, 64, 96, 128, 192, 256]))
    Dv = int(g.choice([D, D, 3, 16, 64, 128, 256]))
    T = int(g.integers(1, 71))
    S = int(g.integers(1, 200))
    params = dict(heads=H, headDim=D, kvHeads=Hk, vHeadDim=Dv, causal=bool(g.integers(0, 4) > 0),
                  posOffset=int(g.choice([0, 3, max(S - T, 0), S + 5])))
    if g.random() < 0.4:
        params["window"] = int(g.integers(1, 40))
    if g.random() < 0.3:
        params["softcap"] = float(g.choice([5.0, 30.0, 50.0]))
    if g.random() < 0.3:
        params["scale"] = float(g.uniform(0.02, 0.5))
    r = g.random()
    if r < 0.15:
        params["alibi"] = True
    elif r < 0.25:
        params["alibiMax"] = float(g.choice([4.0, 8.0]))
    elif r < 0.3:
        params["alibiSlopes"] = [float(s) for s in g.uniform(0.0, 0.5, H)]
    bias = None if g.random() < 0.6 else str(g.choice(["ts", "hts"]))
    x = si.attention_inputs(T, S, H, Hk, D, Dv, seed, sigma=float(g.choice([1.0, 2.0])), bias=bias,
                            bias_mask_p=0.1 if bias else 0.0)
    if bias is not None:
        # keep at least one unmasked visible key per row (rows whose only
        # visible keys all carry -1e9 are implementation-defined)
        b = x["bias"]
        b[b == np.float32(-1e9)] = np.float32(-30.0)
    return x, params


@pytest.mark.parametrize("seed", range(48))
def test_random_sweep(seed):
    x, params = _case(seed)
    check(x, params)


@pytest.mark.parametrize("seed", range(6))
def test_random_sweep_forced_ffma(seed):
    x, params = _case(seed)
    check(x, dict(params, kernel=FFMA))


# -------------------------------------------------------------------- decode
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("G", [2, 4, 8])
@pytest.mark.parametrize("feat", ["plain", "window", "softcap_alibi", "bias_hts", "noncausal"])
def test_decode_kernel(D, G, feat):
    Hk = 2
    H = G * Hk
    S = 1000 + 37 * G + D  # ragged against the 64-row stages
    pos = S - 120
    x = si.attention_inputs(1, S, H, Hk, D, D, 10 * G + D, bias="hts" if feat == "bias_hts" else None)
    params = dict(heads=H, headDim=D, kvHeads=Hk, posOffset=pos, kernel=DECODE)
    if feat == "window":
        params["window"] = 333
    elif feat == "softcap_alibi":
        params.update(softcap=20.0, alibi=True)
    elif feat == "noncausal":
        params.update(causal=False, window=150)
    check(x, params)


@pytest.mark.parametrize("G,T", [(1, 1), (1, 3), (1, 9), (2, 2), (2, 5), (4, 2), (4, 4), (4, 7), (8, 3),
                                 (4, 16), (8, 16)])
@pytest.mark.parametrize("feat", ["plain", "window", "bias_ts", "softcap_alibi", "noncausal", "bias_hts"])
def test_decode_kernel_query_rows(G, T, feat):
    """Several query rows against a cache (speculative or chunked decode): the
    kernel's virtual heads are query rows x group heads, in row groups of at
    most 8; each row masks the keys of the shared range it cannot see."""
    Hk = 2
    H = G * Hk
    D = (32, 64, 128)[(G + T) % 3]
    S = 900 + 13 * T + D
    pos = S - T - 40 + (17 if feat == "noncausal" else 0)
    bias = {"bias_ts": "ts", "bias_hts": "hts"}.get(feat)
    x = si.attention_inputs(T, S, H, Hk, D, D, 1000 + 10 * G + T, bias=bias)
    params = dict(heads=H, headDim=D, kvHeads=Hk, posOffset=pos, kernel=DECODE)
    if feat == "window":
        params["window"] = 1 + 3 * T + 41  # rows see different key ranges
    elif feat == "softcap_alibi":
        params.update(softcap=20.0, alibi=True)
    elif feat == "noncausal":
        params.update(causal=False, window=150)
    check(x, params)


def test_decode_query_rows_forced_splits_and_auto():
    """Forced splits over row groups, and AUTO choosing the decode kernel for
    T <= 8 (a row past S - 1 sees every key)."""
    x = si.attention_inputs(6, 5000, 32, 8, 128, 128, 78)
    for splits in (1, 5, 64):
        check(x, dict(heads=32, headDim=128, kvHeads=8, posOffset=4996, kernel=DECODE, decode_splits=splits))
    check(x, dict(heads=32, headDim=128, kvHeads=8, posOffset=4996))
    x = si.attention_inputs(8, 3000, 8, 8, 64, 64, 79)
    check(x, dict(heads=8, headDim=64, posOffset=2995))  # MHA, rows at 2995..3002


# ------------------------------------------------------------ attention sinks
SINK_CASES = [
    # (T, S, posOffset, window, sinks, causal)
    (200, 900, 700, 150, 4, True),      # sinks far below the window (a tile of their own)
    (130, 700, 0, 100, 37, True),       # sinks inside the first window tiles of early rows
    (64, 3000, 2900, 64, 130, True),    # sink range of several tiles
    (96, 500, 100, 20, 300, False),     # non-causal: sinks past the window's far end
    (1, 5000, 4999, 1000, 4, True),     # decode step with sinks
    (4, 5000, 4990, 700, 64, True),     # speculative step with sinks
    (3, 300, 296, 50, 500, True),       # sinks beyond every key: only causality limits them
]


@pytest.mark.parametrize("kernel", ["auto", "ffma", "tc", "decode"])
@pytest.mark.parametrize("case", SINK_CASES, ids=[str(i) for i in range(len(SINK_CASES))])
def test_attention_sinks(case, kernel):
    """The IR page's attention sinks (keys before `sinks` escape the window)
    on every kernel that covers the shape."""
    T, S, pos, window, sinks, causal = case
    H, Hk, D = 8, 2, 64
    if kernel == "decode" and T > 16:
        pytest.skip("decode kernel: T <= 16")
    if kernel == "tc" and T < 64:
        pytest.skip("tensor-core prefill case list uses T >= 64")
    x = si.attention_inputs(T, S, H, Hk, D, D, 700 + T + sinks)
    params = dict(heads=H, headDim=D, kvHeads=Hk, posOffset=pos, window=window, sinks=sinks, causal=causal)
    if kernel != "auto":
        params["kernel"] = {"ffma": FFMA, "tc": vtmu.VTMU_KERNEL_PREFILL_TF32X3, "decode": DECODE}[kernel]
    check(x, params)


def test_attention_sinks_decode_splits():
    x = si.attention_inputs(1, 6000, 16, 4, 128, 128, 777)
    for splits in (1, 3, 255, 256):
        check(x, dict(heads=16, headDim=128, kvHeads=4, posOffset=5999, window=2048, sinks=100, kernel=DECODE,
                      decode_splits=splits))


def test_attention_sinks_softcap_alibi_bias_tc():
    x = si.attention_inputs(256, 1200, 4, 2, 128, 128, 778, bias="hts")
    check(x, dict(heads=4, headDim=128, kvHeads=2, posOffset=900, window=300, sinks=70, softcap=20.0, alibi=True,
                  kernel=vtmu.VTMU_KERNEL_PREFILL_TF32X3))
    x = si.attention_inputs(256, 1200, 4, 4, 256, 256, 779)
    check(x, dict(heads=4, headDim=256, posOffset=900, window=300, sinks=9, scale=1 / 16, softcap=50.0,
                  kernel=vtmu.VTMU_KERNEL_PREFILL_TF32X3))


@pytest.mark.parametrize("splits", [1, 2, 7, 64, 256])
def test_decode_forced_splits(splits):
    x = si.attention_inputs(1, 5000, 16, 4, 128, 128, 77)
    check(x, dict(heads=16, headDim=128, kvHeads=4, posOffset=4999, kernel=DECODE, decode_splits=splits))


def test_decode_workspace_reused_across_shapes():
    """Arrival counters return to zero: calls of different shapes in a row on
    one workspace stay correct."""
    ws = vtmu.Workspace()
    # (T, S, H, Hk, D): decode calls interleaved with tensor-core prefills,
    # whose scratch shares the workspace.
    for i, (T, S, H, Hk, D) in enumerate([(1, 3000, 16, 4, 128), (256, 700, 8, 4, 64), (1, 700, 8, 4, 64),
                                           (1, 3000, 16, 4, 128), (128, 3000, 16, 4, 128), (1, 64, 8, 1, 32)]):
        x = si.attention_inputs(T, S, H, Hk, D, D, 300 + i)
        params = dict(heads=H, headDim=D, kvHeads=Hk, posOffset=S - T)
        out = vtmu.attention(to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"]), workspace=ws, **params)
        torch.cuda.synchronize()
        ref = oracle.attention(x["q"], x["k"], x["v"], **params)
        assert max_err(out.cpu().numpy(), ref) <= TOL, (T, S, H, Hk, D)
    assert torch.count_nonzero(ws.buf[:65536]).item() == 0  # counters back at zero


def test_decode_equals_last_prefill_row():
    S, H, Hk, D = 513, 8, 2, 128
    x = si.attention_inputs(S, S, H, Hk, D, D, 55)
    full = gpu_attention(x["q"], x["k"], x["v"], heads=H, headDim=D, kvHeads=Hk)
    dec = gpu_attention(x["q"][-1:], x["k"], x["v"], heads=H, headDim=D, kvHeads=Hk, posOffset=S - 1,
                        kernel=DECODE)
    assert max_err(dec[0], full[-1]) <= 1e-5
    ref = oracle.attention_rows(x["q"], x["k"], x["v"], rows=[(S - 1, h) for h in range(H)], heads=H,
                                headDim=D, kvHeads=Hk)
    assert max_err(dec[0].reshape(H, D), ref) <= TOL


# --------------------------------------------------------------------- edges
def test_no_keys_gives_zeros():
    x = si.attention_inputs(5, 0, 4, 2, 32, 32, 1)
    out = gpu_attention(x["q"], np.zeros((0, 64), np.float32), np.zeros((0, 64), np.float32),
                        heads=4, headDim=32, kvHeads=2)
    assert np.array_equal(out, np.zeros((5, 128), np.float32))


@pytest.mark.parametrize("T", [1, 7])
def test_nothing_visible_gives_zeros(T):
    x = si.attention_inputs(T, 40, 4, 2, 64, 64, 2)
    params = dict(heads=4, headDim=64, kvHeads=2, posOffset=500, window=10)
    out, _ = check(x, params)
    assert np.array_equal(out, np.zeros_like(out))


def test_minus_inf_bias_masks_without_nan():
    x = si.attention_inputs(9, 33, 2, 1, 32, 32, 3, bias="ts")
    x["bias"][:, ::3] = -np.inf
    x["bias"][4, :] = -np.inf  # a row with every key masked -> zeros
    out, _ = check(x, dict(heads=2, headDim=32, kvHeads=1, causal=False))
    assert np.array_equal(out[4], np.zeros_like(out[4]))


def test_minus_1e9_bias_equals_explicit_mask():
    x = si.attention_inputs(17, 17, 4, 4, 64, 64, 4, bias="ts")
    mask = np.random.default_rng(0).random((17, 17)) < 0.3
    np.fill_diagonal(mask, False)
    b1 = np.where(mask, np.float32(-1e9), np.float32(0))
    b2 = np.where(mask, np.float32(-np.inf), np.float32(0))
    o1 = gpu_attention(x["q"], x["k"], x["v"], b1, heads=4, headDim=64, causal=False)
    o2 = gpu_attention(x["q"], x["k"], x["v"], b2, heads=4, headDim=64, causal=False)
    assert max_err(o1, o2) <= 1e-6


def test_unaligned_views_take_the_scalar_path():
    """Tensors that start 4 bytes past a 16-byte boundary."""
    T, S, H, D = 20, 45, 4, 64
    x = si.attention_inputs(T, S, H, H, D, D, 9)
    def shifted(a):
        buf = torch.zeros(a.size + 1, dtype=torch.float32, device="cuda")
        buf[1:] = torch.from_numpy(a.ravel()).cuda()
        return buf[1:].view(a.shape)
    out_buf = torch.zeros(T * H * D + 1, dtype=torch.float32, device="cuda")
    out = out_buf[1:].view(T, H * D)
    vtmu.attention(shifted(x["q"]), shifted(x["k"]), shifted(x["v"]), heads=H, headDim=D, out=out)
    torch.cuda.synchronize()
    ref = oracle.attention(x["q"], x["k"], x["v"], heads=H, headDim=D)
    assert max_err(out.cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("T", [1, 300])
def test_long_positions_with_alibi(T):
    """Positions near 32767: the relative ALiBi form keeps scores small."""
    S = 32768
    x = si.attention_inputs(T, S, 4, 4, 32, 32, 12)
    check(x, dict(heads=4, headDim=32, posOffset=S - T, alibi=True))


# --------------------------------------------------------------- cache_write
@pytest.mark.parametrize("width,rows,offset,max_rows", [
    (1024, 1, 32767, 32768), (1024, 7, 0, 100), (33, 5, 10, 20), (3, 1, 0, 1), (256, 100, 155, 255)])
def test_cache_write_bit_exact(width, rows, offset, max_rows):
    g = si.Stream(width + rows)
    cache = g.normal_f32(max_rows * width).reshape(max_rows, width)
    vals = g.normal_f32(rows * width).reshape(rows, width)
    vals.ravel()[::7] = np.float32(-0.0)
    dc = to_dev(cache)
    vtmu.cache_write(dc, to_dev(vals), offset)
    torch.cuda.synchronize()
    oracle.cache_write(cache, vals, offset)
    got = dc.cpu().numpy()
    assert got.tobytes() == cache.tobytes()


def test_cache_write_out_of_range_launches_nothing():
    dc = torch.zeros((8, 4), device="cuda")
    with pytest.raises(vtmu.VtmuError):
        vtmu.cache_write(dc, torch.ones((2, 4), device="cuda"), 7)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dc).item() == 0


def test_no_bounded_wait_gave_up():
    """After all the launches above, no kernel wait hit its time limit."""
    x = si.attention_inputs(1, 4096, 16, 4, 128, 128, 91)
    check(x, dict(heads=16, headDim=128, kvHeads=4, posOffset=4095, kernel=DECODE))
    assert vtmu.vtmu_device_error() == 0


# ----------------------------------------------------------- fused decode step
def _decode_step_case(S, H, Hk, D, new_rows, offset, seed, T=1, **params):
    g = si.Stream(seed)
    x = {
        "q": g.normal_f32(T * H * D).reshape(T, H * D),
        "kc": g.normal_f32(S * Hk * D).reshape(S, Hk * D),
        "vc": g.normal_f32(S * Hk * D).reshape(S, Hk * D),
        "kn": g.normal_f32(new_rows * Hk * D).reshape(new_rows, Hk * D),
        "vn": g.normal_f32(new_rows * Hk * D).reshape(new_rows, Hk * D),
    }
    Kc, Vc = to_dev(x["kc"]), to_dev(x["vc"])
    out = vtmu.decode_step(Kc, Vc, to_dev(x["kn"]), to_dev(x["vn"]), offset, to_dev(x["q"]), heads=H,
                           headDim=D, kvHeads=Hk, **params)
    torch.cuda.synchronize()
    oracle.cache_write(x["kc"], x["kn"], offset)
    oracle.cache_write(x["vc"], x["vn"], offset)
    assert Kc.cpu().numpy().tobytes() == x["kc"].tobytes(), "K cache differs"
    assert Vc.cpu().numpy().tobytes() == x["vc"].tobytes(), "V cache differs"
    pos = params.get("posOffset", offset + new_rows - T)
    ref = oracle.attention(x["q"], x["kc"], x["vc"], heads=H, headDim=D, kvHeads=Hk,
                           **dict(oracle_params(params), posOffset=pos))
    err = max_err(out.cpu().numpy(), ref)
    assert err <= TOL, err


def test_decode_step_workload():
    """The decode workload as one fused launch: cache_write of one row at 32767
    into both [32768, 1024] caches, then attention over all 32768 keys."""
    _decode_step_case(32768, 32, 8, 128, 1, 32767, 1)


@pytest.mark.parametrize("case", [
    dict(S=4000, H=16, Hk=4, D=128, new_rows=1, offset=2222),                  # mid-split row
    dict(S=4000, H=16, Hk=4, D=128, new_rows=5, offset=1278, decode_splits=7),  # rows across a split edge
    dict(S=3000, H=8, Hk=4, D=64, new_rows=3, offset=2990, posOffset=2500),     # new rows not visible
    dict(S=3000, H=8, Hk=1, D=32, new_rows=2, offset=100, posOffset=2999, window=700),  # outside the window
    dict(S=2048, H=16, Hk=8, D=64, new_rows=1, offset=1000, causal=False, window=300),
    dict(S=1500, H=8, Hk=1, D=128, new_rows=1, offset=1499, softcap=30.0, alibi=True),
])
def test_decode_step_fused_cases(case):
    case = dict(case)
    _decode_step_case(case.pop("S"), case.pop("H"), case.pop("Hk"), case.pop("D"), case.pop("new_rows"),
                      case.pop("offset"), 500, kernel=DECODE, **case)


def test_decode_step_query_rows_fused():
    """A chunked step of T = 6 new rows runs as one decode launch."""
    _decode_step_case(700, 4, 2, 128, 6, 600, 501, T=6)
    _decode_step_case(3000, 32, 8, 128, 4, 2996, 503, T=4)


def test_decode_step_unfused_paths():
    """Shapes outside the decode kernel: a chunk of T = 12 rows (AUTO takes
    the prefill kernel past 8) and a head size the decode table does not
    cover run as three launches."""
    _decode_step_case(700, 4, 2, 128, 12, 600, 501, T=12)
    _decode_step_case(700, 4, 4, 96, 1, 650, 502)


@pytest.mark.parametrize("case", [
    dict(S=32768, H=32, Hk=8, D=128, T=1, new_rows=1, offset=32767, pinned=True),   # the decode workload
    dict(S=3000, H=8, Hk=4, D=64, T=1, new_rows=3, offset=2990, pinned=False, bias=True),
    dict(S=700, H=4, Hk=2, D=128, T=6, new_rows=6, offset=600, pinned=True),       # tensor-core decode (12 virtual heads)
    dict(S=32768, H=32, Hk=8, D=128, T=4, new_rows=4, offset=32764, pinned=True),  # the 4-row speculative workload
    dict(S=900, H=16, Hk=2, D=64, T=3, new_rows=3, offset=800, pinned=False),     # CUDA-core decode, 24 virtual heads
    dict(S=3000, H=32, Hk=8, D=128, T=1, new_rows=1, offset=2999, pinned="shifted"),  # pinned, off the 16-byte grid
])
def test_decode_step_host_buffers(case):
    """vtmu_decode_step_host: the step's inputs and output in host memory
    (pinned or pageable).  Caches bit-exact against the oracle's cache_write,
    the output bit-identical to the device-buffer step on the same data and
    within tolerance of the oracle."""
    S, H, Hk, D, T, n, off = (case[k] for k in ("S", "H", "Hk", "D", "T", "new_rows", "offset"))
    g = si.Stream(510)
    x = {"q": g.normal_f32(T * H * D).reshape(T, H * D), "kc": g.normal_f32(S * Hk * D).reshape(S, Hk * D),
         "vc": g.normal_f32(S * Hk * D).reshape(S, Hk * D), "kn": g.normal_f32(n * Hk * D).reshape(n, Hk * D),
         "vn": g.normal_f32(n * Hk * D).reshape(n, Hk * D)}
    bias = g.normal_f32(T * S).reshape(T, S) if case.get("bias") else None
    pos = off + n - T
    p = vtmu.make_params(T, S, heads=H, headDim=D, kvHeads=Hk, posOffset=pos,
                         bias_kind=vtmu.VTMU_BIAS_TS if bias is not None else vtmu.VTMU_BIAS_NONE)
    def host(a):
        if case["pinned"] == "shifted":  # staged: the kernels take 16-byte aligned rows only
            buf = torch.empty(a.size + 1, dtype=torch.float32).pin_memory()
            view = buf[1:].view(a.shape)
            view.copy_(torch.from_numpy(a))
            return view
        return torch.from_numpy(a).pin_memory() if case["pinned"] else a
    nb = vtmu.vtmu_decode_step_host_workspace_size(p, n)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    Kc, Vc = to_dev(x["kc"]), to_dev(x["vc"])
    out_h = host(np.zeros((T, H * D), np.float32))
    st = torch.cuda.current_stream().cuda_stream
    vtmu.vtmu_decode_step_host(Kc, Vc, S, host(x["kn"]), host(x["vn"]), n, off, host(x["q"]),
                               None if bias is None else host(bias), out_h, p, ws, nb, st)
    out_host = np.asarray(out_h).copy()
    Kd, Vd = to_dev(x["kc"]), to_dev(x["vc"])
    out_dev = vtmu.decode_step(Kd, Vd, to_dev(x["kn"]), to_dev(x["vn"]), off, to_dev(x["q"]),
                               None if bias is None else to_dev(bias), heads=H, headDim=D, kvHeads=Hk, posOffset=pos)
    torch.cuda.synchronize()
    assert out_host.tobytes() == out_dev.cpu().numpy().tobytes(), "host-buffer step differs from the device step"
    oracle.cache_write(x["kc"], x["kn"], off)
    oracle.cache_write(x["vc"], x["vn"], off)
    assert Kc.cpu().numpy().tobytes() == x["kc"].tobytes() and Vc.cpu().numpy().tobytes() == x["vc"].tobytes()
    ref = oracle.attention(x["q"], x["kc"], x["vc"], bias, heads=H, headDim=D, kvHeads=Hk, posOffset=pos)
    assert max_err(out_host, ref) <= TOL


def test_decode_step_refuses_rows_past_the_cache():
    Kc = torch.zeros((8, 4), device="cuda")
    Vc = torch.zeros((8, 4), device="cuda")
    with pytest.raises(vtmu.VtmuError) as e:
        vtmu.decode_step(Kc, Vc, torch.ones((2, 4), device="cuda"), torch.ones((2, 4), device="cuda"), 7,
                         torch.zeros((1, 8), device="cuda"), heads=2, headDim=4, kvHeads=1)
    assert e.value.status == vtmu.VTMU_ERR_RANGE
    torch.cuda.synchronize()
    assert torch.count_nonzero(Kc).item() == 0 and torch.count_nonzero(Vc).item() == 0


# ------------------------------------------------------ tcgen05 3xTF32 prefill
TC = vtmu.VTMU_KERNEL_PREFILL_TF32X3


def _tc_case(seed):
    g = np.random.default_rng(7000 + seed)
    H, Hk = [(1, 1), (4, 1), (4, 2), (6, 3), (8, 8), (8, 2)][seed % 6]
    D, Dv = [(32, 32), (64, 64), (96, 96), (128, 128), (192, 128), (256, 256)][int(g.integers(0, 6))]
    T = int(g.integers(1, 300))
    S = int(g.integers(1, 500))
    params = dict(heads=H, headDim=D, kvHeads=Hk, vHeadDim=Dv, causal=bool(g.integers(0, 4) > 0),
                  posOffset=int(g.choice([0, 5, max(S - T, 0), S + 7])))
    if g.random() < 0.4:
        params["window"] = int(g.integers(1, 120))
    if g.random() < 0.3:
        params["softcap"] = float(g.choice([5.0, 30.0, 50.0]))
    if g.random() < 0.3:
        params["scale"] = float(g.uniform(0.02, 0.5))
    r = g.random()
    if r < 0.2:
        params["alibi"] = True
    elif r < 0.3:
        params["alibiMax"] = 8.0
    bias = None if g.random() < 0.6 else str(g.choice(["ts", "hts"]))
    x = si.attention_inputs(T, S, H, Hk, D, Dv, 50 + seed, sigma=float(g.choice([1.0, 2.0])), bias=bias,
                            bias_mask_p=0.1 if bias else 0.0)
    if bias is not None:
        b = x["bias"]
        b[b == np.float32(-1e9)] = np.float32(-30.0)
    return x, params


@pytest.mark.parametrize("seed", range(40))
def test_tensor_core_prefill_random_sweep(seed):
    x, params = _tc_case(seed)
    check(x, dict(params, kernel=TC))


@pytest.mark.parametrize("T,S,pos", [(128, 128, 0), (129, 64, 0), (1, 40, 39), (300, 1, 0), (257, 1000, 743)])
def test_tensor_core_prefill_tile_edges(T, S, pos):
    x = si.attention_inputs(T, S, 4, 2, 128, 128, 61)
    check(x, dict(heads=4, headDim=128, kvHeads=2, posOffset=pos, kernel=TC))


@pytest.mark.parametrize("T,S,pos", [(128, 128, 0), (200, 333, 133), (1, 64, 63)])
def test_tensor_core_prefill_latent_shape(T, S, pos):
    """headDim 192 with vHeadDim 128 (one S buffer in TMEM)."""
    x = si.attention_inputs(T, S, 4, 4, 192, 128, 64, bias="ts")
    check(x, dict(heads=4, headDim=192, vHeadDim=128, posOffset=pos, causal=False, kernel=TC))


@pytest.mark.parametrize("T,S,pos,window", [(128, 128, 0, 0), (200, 333, 133, 0), (1, 64, 63, 0),
                                            (300, 300, 0, 100), (257, 1000, 743, 64)])
def test_tensor_core_prefill_head_dim_256(T, S, pos, window):
    """headDim = vHeadDim = 256: the V columns split over two CTAs per tile."""
    x = si.attention_inputs(T, S, 4, 2, 256, 256, 65, sigma=2.0)
    check(x, dict(heads=4, headDim=256, kvHeads=2, posOffset=pos, window=window, scale=1 / 16, softcap=50.0,
                  kernel=TC))


def test_tensor_core_prefill_masked_rows_give_zeros():
    x = si.attention_inputs(140, 50, 2, 1, 64, 64, 62, bias="ts")
    x["bias"][:, ::3] = -np.inf
    x["bias"][7, :] = -np.inf
    x["bias"][139, :] = -np.inf
    out, _ = check(x, dict(heads=2, headDim=64, kvHeads=1, causal=False, kernel=TC))
    assert np.array_equal(out[7], np.zeros_like(out[7])) and np.array_equal(out[139], np.zeros_like(out[139]))


def test_tensor_core_prefill_agrees_with_ffma():
    x = si.attention_inputs(512, 512, 8, 2, 128, 128, 63)
    params = dict(heads=8, headDim=128, kvHeads=2, window=200, softcap=30.0)
    a = gpu_attention(x["q"], x["k"], x["v"], kernel=TC, **params)
    b = gpu_attention(x["q"], x["k"], x["v"], kernel=FFMA, **params)
    assert max_err(a, b) <= 5e-5
    assert vtmu.vtmu_device_error() == 0
