"""Absorbed latent attention on the GPU against the oracle.

The IR schema page's mla_attention ($defs.op_mla_attention): the library
computes it in the absorbed order (queries through k_b, one shared latent
head, the output through v_b); the oracle expands every head's keys and
values (the definition).  Tolerance: max |err| <= 1e-4 absolute, outputs of
order 1 (keys and values have unit variance).  The decode step's cache
write is compared bit for bit."""
import numpy as np
import pytest

import seeded_inputs as si

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import f32_gqa_attention_gb300 as vtmu  # noqa: E402
import oracle  # noqa: E402

TOL = 1e-4
R, P = 512, 64


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check(out, ref, what):
    assert np.all(np.isfinite(out)), what
    err = float(np.max(np.abs(out.astype(np.float64) - ref))) if out.size else 0.0
    assert err <= TOL, f"{what}: max |err| {err:.3e}"
    return err


# (T, S, heads, qk_nope, v_head_dim, params)
CASES = [
    (1, 200, 16, 128, 128, dict(causal=True, posOffset=199)),
    (1, 1000, 4, 64, 32, dict(causal=True, posOffset=700)),
    (2, 333, 3, 16, 100, dict(causal=True, posOffset=331)),
    (4, 257, 33, 128, 128, dict(causal=True, posOffset=253)),
    (1, 96, 1, 0, 1, dict(causal=False)),
    (3, 500, 8, 32, 64, dict(causal=False, posOffset=250, window=40)),
    (1, 900, 16, 128, 128, dict(causal=True, posOffset=899, window=300, sinks=4)),
    (2, 64, 5, 48, 16, dict(causal=True, posOffset=62, window=8, sinks=20)),
    (17, 150, 2, 128, 128, dict(causal=True, posOffset=133)),
    (1, 40, 8, 128, 128, dict(causal=True, posOffset=39, scale=0.05)),
    (1, 31, 7, 24, 8, dict(causal=True, posOffset=30)),
    (2, 10, 9, 128, 128, dict(causal=True, posOffset=0, window=1)),
]


KERNELS = [vtmu.MLA_KERNEL_TENSOR_CORES, vtmu.MLA_KERNEL_CUDA_CORES]


@pytest.mark.parametrize("kernel", KERNELS, ids=["tensor_cores", "cuda_cores"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_mla_attention_cases(case, kernel):
    T, S, H, N, Dv, params = CASES[case]
    x = si.mla_inputs(S, T, H, R, N, P, Dv, 100 + case)
    kw = dict(heads=H, qk_nope=N, v_head_dim=Dv, **params)
    out = vtmu.mla_attention(_dev(x["q"]), _dev(x["state"]), _dev(x["k_b"]), _dev(x["v_b"]), kernel=kernel, **kw)
    torch.cuda.synchronize()
    ref = oracle.mla_attention(x["q"], x["state"], x["k_b"], x["v_b"], kv_rank=R, qk_rope=P, **kw)
    _check(out.cpu().numpy(), ref, f"case {case}")
    assert vtmu.vtmu_device_error() == 0


def test_mla_no_visible_key_gives_zeros():
    """A causal window that ends before the cache starts leaves a row with no
    key: its output is zero (as for op attention)."""
    T, S, H, N, Dv = 2, 50, 4, 32, 16
    x = si.mla_inputs(S, T, H, R, N, P, Dv, 3)
    kw = dict(heads=H, qk_nope=N, v_head_dim=Dv, causal=False, posOffset=200, window=20)
    out = vtmu.mla_attention(_dev(x["q"]), _dev(x["state"]), _dev(x["k_b"]), _dev(x["v_b"]), **kw)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), np.zeros((T, H * Dv), np.float32))


@pytest.mark.parametrize("kernel", KERNELS, ids=["tensor_cores", "cuda_cores"])
@pytest.mark.parametrize("name", ["mla_decode", "mla_decode_v3"])
def test_mla_decode_step_workload(name, kernel):
    """The full-size decode step (cache_write of the new latent row, then one
    query row over 32768 cache rows), as the benchmark runs it; the oracle
    recomputes every head (16) or 12 of them (128 heads), and the cache must
    hold the new row bit for bit."""
    w = si.WORKLOADS[name]
    x = si.workload_inputs(name)
    H, N, Dv, off = w["heads"], w["qk_nope"], w["v_head_dim"], w["offset"]
    state = _dev(x["state"])
    out = vtmu.mla_decode_step(state, _dev(x["state_new"]), off, _dev(x["q"]), _dev(x["k_b"]), _dev(x["v_b"]),
                               heads=H, qk_nope=N, v_head_dim=Dv, kernel=kernel, **w["params"])
    torch.cuda.synchronize()
    oracle.cache_write(x["state"], x["state_new"], off)
    st = state.cpu().numpy()
    assert np.array_equal(st[off:off + 1], x["state_new"]) and np.array_equal(st[:off], x["state"][:off])
    heads = list(range(H)) if H <= 16 else sorted({0, 1, 31, 32, 63, 64, 65, 96, 100, 126, 127, H // 2})
    rows = [(0, h) for h in heads]
    ref = oracle.mla_attention_rows(x["q"], x["state"], x["k_b"], x["v_b"], rows=rows, heads=H, kv_rank=R,
                                    qk_nope=N, qk_rope=P, v_head_dim=Dv, **w["params"])
    o = out.cpu().numpy()
    got = np.stack([o[0, h * Dv:(h + 1) * Dv] for _, h in rows])
    _check(got, ref, name)
    assert vtmu.vtmu_device_error() == 0


def test_mla_decode_steps_in_sequence():
    """Three decode steps in a row on one cache: each appends a latent row
    and attends over everything written so far."""
    S0, H, N, Dv = 300, 16, 128, 128
    x = si.mla_inputs(S0 + 3, 1, H, R, N, P, Dv, 21, new_rows=3)
    state_np = x["state"].copy()
    state = _dev(state_np)
    g = si.Stream(22)
    for i in range(3):
        q = g.normal_f32(H * (N + P)).reshape(1, -1)
        off = S0 + i
        out = vtmu.mla_decode_step(state, _dev(x["state_new"][i:i + 1]), off, _dev(q), _dev(x["k_b"]),
                                   _dev(x["v_b"]), heads=H, qk_nope=N, v_head_dim=Dv)
        torch.cuda.synchronize()
        oracle.cache_write(state_np, x["state_new"][i:i + 1], off)
        ref = oracle.mla_attention(q, state_np[:off + 1], x["k_b"], x["v_b"], heads=H, kv_rank=R, qk_nope=N,
                                   qk_rope=P, v_head_dim=Dv, posOffset=off)
        _check(out.cpu().numpy(), ref, f"step {i}")
    assert np.array_equal(state.cpu().numpy(), state_np)


def test_mla_refuses_widths_it_does_not_serve():
    p = vtmu.make_mla_params(1, 64, heads=2, kv_rank=256, qk_nope=64, v_head_dim=64)
    with pytest.raises(vtmu.VtmuError) as e:
        vtmu.vtmu_mla_workspace_size(p)
    assert e.value.status == vtmu.VTMU_ERR_UNSUPPORTED and "kv_rank" in str(e.value)


def _pinned_shifted(a):
    """A pinned copy of `a` that starts 4 bytes past a 16-byte boundary."""
    buf = torch.empty(a.size + 1, dtype=torch.float32).pin_memory()
    view = buf[1:].view(a.shape)
    view.copy_(torch.from_numpy(np.ascontiguousarray(a)))
    return view


@pytest.mark.parametrize("pinned", ["pinned", "pageable", "pinned_shifted"])
@pytest.mark.parametrize("T,kernel", [(1, vtmu.MLA_KERNEL_AUTO), (2, vtmu.MLA_KERNEL_TENSOR_CORES)])
def test_mla_decode_step_host_buffers(pinned, T, kernel):
    """vtmu_mla_decode_step_host: q, the new latent row and the output in host
    memory (pinned buffers are used in place, pageable ones and pinned ones
    off the 16-byte grid staged).  The output is bit-identical to the
    device-buffer step on the same data, the cache row bit-exact."""
    S0, H, N, Dv = 1500, 16, 128, 128
    x = si.mla_inputs(S0 + 1, T, H, R, N, P, Dv, 40 + T, new_rows=1)
    off = S0
    p = vtmu.make_mla_params(T, S0 + 1, heads=H, qk_nope=N, v_head_dim=Dv, posOffset=S0 + 1 - T, kernel=kernel)
    host = {"pinned": lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory(),
            "pageable": np.ascontiguousarray, "pinned_shifted": _pinned_shifted}[pinned]
    state = _dev(x["state"])
    out_h = host(np.zeros((T, H * Dv), np.float32))
    nb = vtmu.vtmu_mla_decode_step_host_workspace_size(p, 1)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    vtmu.vtmu_mla_decode_step_host(state, S0 + 1, host(x["state_new"][:1]), 1, off, host(x["q"]), _dev(x["k_b"]),
                                   _dev(x["v_b"]), out_h, p, ws, nb, torch.cuda.current_stream().cuda_stream)
    got = np.asarray(out_h).copy()
    state2 = _dev(x["state"])
    ref_dev = vtmu.mla_decode_step(state2, _dev(x["state_new"][:1]), off, _dev(x["q"]), _dev(x["k_b"]),
                                   _dev(x["v_b"]), heads=H, qk_nope=N, v_head_dim=Dv, posOffset=S0 + 1 - T,
                                   kernel=kernel)
    torch.cuda.synchronize()
    assert got.tobytes() == ref_dev.cpu().numpy().tobytes(), "host-buffer step differs from the device step"
    st = state.cpu().numpy()
    assert np.array_equal(st[off:off + 1], x["state_new"][:1]) and np.array_equal(st[:off], x["state"][:off])
    oracle.cache_write(x["state"], x["state_new"][:1], off)
    ref = oracle.mla_attention(x["q"], x["state"], x["k_b"], x["v_b"], heads=H, kv_rank=R, qk_nope=N, qk_rope=P,
                               v_head_dim=Dv, posOffset=S0 + 1 - T)
    _check(got, ref, "host buffers")
    assert vtmu.vtmu_device_error() == 0
