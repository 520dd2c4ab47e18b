"""The allocation-free decode entry point against the regular one.

vtmu_attention_decode_noalloc serves callers that cannot allocate device
memory (a plug-in inside a host process that owns all device memory, or a
decode loop that must not call cudaMalloc): it keeps the decode kernel's
scratch in a static device array instead of a caller's workspace.  This file
is collected last so that a run stopping at the first failure has already run
every other test; it passes alone in a fresh process as well."""
import numpy as np
import pytest

import seeded_inputs as si

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import f32_gqa_attention_gb300 as vtmu  # noqa: E402

def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _both(x, **params):
    """Output of the regular entry point (with a workspace) and of the
    allocation-free one, on the same inputs and stream."""
    vtmu.load_library()
    q, k, v = _dev(x["q"]), _dev(x["k"]), _dev(x["v"])
    b = _dev(x["bias"]) if "bias" in x else None
    bias_kind = vtmu.VTMU_BIAS_NONE if b is None else vtmu.VTMU_BIAS_HTS
    p = vtmu.make_params(1, k.shape[0], bias_kind=bias_kind, kernel=vtmu.VTMU_KERNEL_DECODE, **params)
    st = torch.cuda.current_stream().cuda_stream
    ws_bytes = vtmu.vtmu_attention_workspace_size(p)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.full((1, params["heads"] * params["headDim"]), float("nan"), device="cuda")
    vtmu.vtmu_attention(q, k, v, b, ref, p, ws, ws_bytes, st)
    out = torch.full_like(ref, float("nan"))
    vtmu.vtmu_attention_decode_noalloc(q, k, v, b, out, p, st)
    torch.cuda.synchronize()
    assert vtmu.vtmu_device_error() == 0, "a kernel wait gave up"
    return ref.cpu().numpy(), out.cpu().numpy()


def _same(ref, out):
    """Both calls run the same kernel with the same plan, so the outputs are
    bit-identical (a scratch-layout slip would show as a small difference)."""
    assert np.all(np.isfinite(out))
    assert np.array_equal(ref, out), float(np.max(np.abs(out - ref)))


def test_noalloc_decode_matches_regular_entry_point_on_two_calls():
    first = si.attention_inputs(1, 32768, 32, 8, 128, 128, 1)
    _same(*_both(first, heads=32, headDim=128, kvHeads=8, posOffset=32767))
    second = si.attention_inputs(1, 3000, 16, 2, 64, 64, 2, bias="hts")
    _same(*_both(second, heads=16, headDim=64, kvHeads=2, posOffset=2500, window=700, softcap=30.0))


def test_noalloc_after_a_larger_call_and_with_one_query_head_per_kv_head():
    """A call with many splits leaves partials all over the array; a later
    call with fewer splits and other heads must not read them.  Heads ==
    kvHeads (group size 1) pads every KV head to two virtual heads."""
    big = si.attention_inputs(1, 32768, 16, 16, 128, 128, 3)
    _same(*_both(big, heads=16, headDim=128, kvHeads=16, posOffset=32767, decode_splits=64))
    small = si.attention_inputs(1, 700, 8, 8, 32, 32, 4)
    _same(*_both(small, heads=8, headDim=32, kvHeads=8, posOffset=650))
    _same(*_both(big, heads=16, headDim=128, kvHeads=16, posOffset=20000, decode_splits=7))


def test_noalloc_refuses_a_shape_beyond_its_scratch():
    """64 query heads at vHeadDim 128 over 32768 keys need more decode scratch
    than the static array holds.  The buffers are real and sized for the
    shape, so nothing could go out of bounds even if the check were wrong."""
    H, Hk, D, S = 64, 8, 128, 32768
    p = vtmu.make_params(1, S, heads=H, headDim=D, kvHeads=Hk, posOffset=S - 1,
                         kernel=vtmu.VTMU_KERNEL_DECODE)
    assert vtmu.vtmu_attention_workspace_size(p) > vtmu.NOALLOC_SCRATCH_BYTES  # host-side, no launch
    q = torch.zeros((1, H * D), device="cuda")
    k = torch.zeros((S, Hk * D), device="cuda")
    v = torch.zeros((S, Hk * D), device="cuda")
    out = torch.zeros((1, H * D), device="cuda")
    with pytest.raises(vtmu.VtmuError) as e:
        vtmu.vtmu_attention_decode_noalloc(q, k, v, None, out, p, torch.cuda.current_stream().cuda_stream)
    assert e.value.status == vtmu.VTMU_ERR_WORKSPACE and "static scratch" in str(e.value)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
