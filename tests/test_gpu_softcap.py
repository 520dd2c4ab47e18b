"""The softcap's two tanh approximations, pointwise, over a dense sweep.

Op "attention" caps a score as cap * tanh(x / cap) (param softcap; op
softcap gives the same formula).  The kernels evaluate tanh with their own
approximations: softcap_tanh (odd Taylor series below |y| = 1/4, the
identity tanh|y| = (1 - e) / (1 + e) with e = exp(-2|y|) above) and, for a
whole tile of scores, the odd series through y^13 when every |y| of a warp
is below 1/2.  End-to-end attention parity averages over many scores and
could hide a local error, so these tests compare the approximations point by
point with tanh in float64 and with the device's tanhf, on both sides of
both branch seams.  The probe kernels (tests/probes/softcap_probe.cu) call
the library's own device functions; they are compiled here, not shipped."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROBE_SRC = os.path.join(ROOT, "tests", "probes", "softcap_probe.cu")
CSRC = os.path.join(ROOT, "f32_gqa_attention_gb300", "csrc")
OUT_DIR = os.path.join(ROOT, "_build", "probes")
ABS_TOL = 1e-6


@pytest.fixture(scope="module")
def probe():
    from f32_gqa_attention_gb300 import _build
    os.makedirs(OUT_DIR, exist_ok=True)
    so = os.path.join(OUT_DIR, "softcap_probe.so")
    deps = [PROBE_SRC] + [os.path.join(CSRC, f) for f in ("attn_common.cuh", "softcap.cuh", "attn_desc.h")]
    if not os.path.exists(so) or any(os.path.getmtime(d) > os.path.getmtime(so) for d in deps):
        cmd = [_build.nvcc()] + _build.NVCC_FLAGS + ["-shared", PROBE_SRC, "-o", so]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
    lib = ctypes.CDLL(so)
    vp = ctypes.c_void_p
    lib.softcap_probe_scalar.argtypes = [vp, vp, vp, ctypes.c_int, vp]
    lib.softcap_probe_scalar.restype = ctypes.c_int
    lib.softcap_probe_tile.argtypes = [vp, vp, vp, ctypes.c_float, ctypes.c_float, ctypes.c_int, vp]
    lib.softcap_probe_tile.restype = ctypes.c_int
    lib.softcap_probe_values_per_warp.restype = ctypes.c_int
    return lib


def sweep():
    """y in [-30, 30] densely, plus dense bands around |y| = 1/4 and |y| = 1/2
    (the two branch seams) and tiny arguments, as float32."""
    parts = [np.linspace(-30.0, 30.0, 1 << 21)]
    for c in (0.25, 0.5):
        band = np.linspace(c - 1e-3, c + 1e-3, 1 << 16)
        parts += [band, -band]
    parts.append(np.linspace(-1e-3, 1e-3, 1 << 12))
    y = np.concatenate(parts).astype(np.float32)
    for c in (0.25, 0.5):  # the float32 neighbours of each seam
        s = np.float32(c)
        y = np.concatenate([y, [np.nextafter(s, np.float32(0)), s, np.nextafter(s, np.float32(1))]]).astype(
            np.float32)
        y = np.concatenate([y, -y[-3:]]).astype(np.float32)
    return y


def _worst(y, got, want):
    err = np.abs(got.astype(np.float64) - want)
    i = int(np.argmax(err))
    return float(err[i]), float(y[i])


def test_softcap_tanh_pointwise(probe):
    y = sweep()
    n = y.size
    yd = torch.from_numpy(y).cuda()
    out_lib = torch.empty_like(yd)
    out_ref = torch.empty_like(yd)
    st = torch.cuda.current_stream().cuda_stream
    assert probe.softcap_probe_scalar(yd.data_ptr(), out_lib.data_ptr(), out_ref.data_ptr(), n, st) == 0
    torch.cuda.synchronize()
    lib, ref = out_lib.cpu().numpy(), out_ref.cpu().numpy()
    exact = np.tanh(y.astype(np.float64))
    e_exact, y_exact = _worst(y, lib, exact)
    e_dev, y_dev = _worst(y, lib, ref.astype(np.float64))
    e_tanhf, _ = _worst(y, ref, exact)
    print(f"softcap_tanh: max |err| vs tanh (fp64) {e_exact:.3g} at y = {y_exact!r}; "
          f"vs device tanhf {e_dev:.3g} at y = {y_dev!r}; tanhf itself {e_tanhf:.3g}")
    assert e_exact <= ABS_TOL, (e_exact, y_exact)
    assert e_dev <= ABS_TOL, (e_dev, y_dev)
    assert np.all(np.abs(lib) <= 1.0)
    assert np.array_equal(np.sign(lib), np.sign(y))  # odd, and 0 stays 0
    big = np.abs(y) >= 20
    assert np.all(np.abs(lib[big]) == 1.0)  # both tails saturate exactly


def _tile(probe, y, qk_mul, cap):
    per = probe.softcap_probe_values_per_warp()
    n = (y.size + per - 1) // per * per
    yp = np.zeros(n, dtype=np.float32)
    yp[:y.size] = y
    yd = torch.from_numpy(yp).cuda()
    out = torch.empty_like(yd)
    flags = torch.zeros(n // per, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert probe.softcap_probe_tile(yd.data_ptr(), out.data_ptr(), flags.data_ptr(), qk_mul, cap, n, st) == 0
    torch.cuda.synchronize()
    return out.cpu().numpy()[:y.size], flags.cpu().numpy()


def test_tile_series_pointwise(probe):
    """|y| < 1/2 everywhere: every warp takes the odd series through y^13."""
    y = np.concatenate([np.linspace(-0.5, 0.5, 1 << 20, endpoint=False)[1:],
                        np.linspace(0.499, 0.4999999, 1 << 14), -np.linspace(0.499, 0.4999999, 1 << 14),
                        np.linspace(0.2499, 0.2501, 1 << 12)]).astype(np.float32)
    y = y[np.abs(y) < 0.5]
    got, flags = _tile(probe, y, 1.0, 1.0)
    assert np.all(flags == 1), "a warp left the series branch"
    e, at = _worst(y, got, np.tanh(y.astype(np.float64)))
    print(f"tile series: max |err| vs tanh (fp64) {e:.3g} at y = {at!r}")
    assert e <= ABS_TOL, (e, at)


def test_tile_form_over_the_whole_range(probe):
    """The full sweep through the tile form: warps holding any |y| >= 1/2 take
    softcap_tanh, the others the series; both within the bound."""
    y = sweep()
    got, flags = _tile(probe, y, 1.0, 1.0)
    assert flags.min() == 0 and flags.max() == 1  # both branches ran
    e, at = _worst(y, got, np.tanh(y.astype(np.float64)))
    print(f"tile form, full sweep: max |err| vs tanh (fp64) {e:.3g} at y = {at!r}")
    assert e <= ABS_TOL, (e, at)


def test_tile_form_with_the_workload_constants(probe):
    """The Gemma-2-style prefill's constants: scale 1/16, softcap 50, scores
    kept in base-2 units (cap * log2 e outside, scale / cap inside)."""
    log2e = 1.4426950408889634
    qk_mul, cap = np.float32((1.0 / 16) / 50.0), np.float32(50.0 * log2e)
    x = np.concatenate([np.linspace(-2000.0, 2000.0, 1 << 20), np.linspace(-399.0, 399.0, 1 << 18)]).astype(
        np.float32)
    got, _ = _tile(probe, x, float(qk_mul), float(cap))
    want = np.float64(cap) * np.tanh(x.astype(np.float64) * np.float64(qk_mul))
    e, at = _worst(x, got, want)
    print(f"tile form, workload constants: max |err| / cap {e / float(cap):.3g} at x = {at!r}")
    assert e / float(cap) <= 2 * ABS_TOL, (e, at)
