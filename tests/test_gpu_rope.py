"""GPU parity of op "rope" (vtmu.mpakt.dev/api/ops) and of the decode step
with the rotary embedding fused in, through the C ABI, against the CPU
oracle on the same seeded inputs."""
import numpy as np
import pytest

import oracle
import seeded_inputs as si
from gpu_util import TOL, max_err, oracle_params, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import f32_gqa_attention_gb300 as vtmu  # noqa: E402

ROPE_TOL = 1e-5  # turned N(0,1) channels: hardware cos/sin (abs err < 2^-21) of an exactly reduced angle

ROPE_CASES = [
    dict(T=37, H=4, D=128, offset=0),
    dict(T=5, H=32, D=128, offset=32763, base=500000.0),                      # Llama 3 theta, late positions
    dict(T=64, H=3, D=64, offset=1000, interleaved=True),
    dict(T=9, H=2, D=96, offset=77, rotaryDim=32),                              # partial rotary
    dict(T=9, H=2, D=80, offset=10, rotaryDim=64, interleaved=True),
    dict(T=16, H=8, D=256, offset=4096, scaling={"rope_type": "linear", "factor": 4.0}),
    dict(T=4, H=2, D=32, offset=3, invFreq=[0.5 ** j for j in range(16)], attentionFactor=1.25),
    dict(T=1, H=1, D=2, offset=123456),
    dict(T=0, H=2, D=64, offset=5),
]


@pytest.mark.parametrize("case", ROPE_CASES, ids=[str(i) for i in range(len(ROPE_CASES))])
def test_rope_matches_oracle(case):
    case = dict(case)
    T, H, D, off = case.pop("T"), case.pop("H"), case.pop("D"), case.pop("offset")
    x = si.Stream(600 + T + D).normal_f32(T * H * D).reshape(T, H * D)
    ref = oracle.rope(x, headDim=D, offset=off, **case)
    xd = to_dev(x)
    out = vtmu.rope(xd, headDim=D, offset=off, **case)
    inplace = to_dev(x)
    vtmu.rope(inplace, headDim=D, offset=off, out=inplace, **case)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert max_err(got, ref) <= ROPE_TOL, max_err(got, ref)
    assert np.array_equal(inplace.cpu().numpy(), got), "in-place result differs"
    assert np.array_equal(xd.cpu().numpy(), x), "input changed"


def _rope_step_case(S, H, Hk, D, new_rows, offset, seed, rope, T=1, **params):
    g = si.Stream(seed)
    x = {
        "q": g.normal_f32(T * H * D).reshape(T, H * D),
        "kc": g.normal_f32(S * Hk * D).reshape(S, Hk * D),
        "vc": g.normal_f32(S * Hk * D).reshape(S, Hk * D),
        "kn": g.normal_f32(new_rows * Hk * D).reshape(new_rows, Hk * D),
        "vn": g.normal_f32(new_rows * Hk * D).reshape(new_rows, Hk * D),
    }
    pos = params.pop("posOffset", offset + new_rows - T)
    # fused
    Kc, Vc = to_dev(x["kc"]), to_dev(x["vc"])
    q = to_dev(x["q"])
    out = vtmu.decode_step_rope(Kc, Vc, to_dev(x["kn"]), to_dev(x["vn"]), offset, q, heads=H, headDim=D,
                                kvHeads=Hk, posOffset=pos, rope=rope, **params)
    # composed: op rope on q and on the new keys, then the plain decode step
    Kc2, Vc2 = to_dev(x["kc"]), to_dev(x["vc"])
    q2 = vtmu.rope(to_dev(x["q"]), headDim=D, offset=pos, **rope)
    kn2 = vtmu.rope(to_dev(x["kn"]), headDim=D, offset=offset, **rope)
    out2 = vtmu.decode_step(Kc2, Vc2, kn2, to_dev(x["vn"]), offset, q2, heads=H, headDim=D, kvHeads=Hk,
                            posOffset=pos, **params)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), x["q"]), "q changed"
    assert np.array_equal(Kc.cpu().numpy(), Kc2.cpu().numpy()), "fused K cache differs from rope + decode_step"
    assert np.array_equal(out.cpu().numpy(), out2.cpu().numpy()), "fused output differs from rope + decode_step"
    # oracle: rope, cache_write, attention
    qr = oracle.rope(x["q"], headDim=D, offset=pos, **rope)
    knr = oracle.rope(x["kn"], headDim=D, offset=offset, **rope)
    kc_ref = x["kc"].astype(np.float64).copy()
    kc_ref[offset:offset + new_rows] = knr
    assert max_err(Kc.cpu().numpy(), kc_ref) <= ROPE_TOL
    oracle.cache_write(x["vc"], x["vn"], offset)
    assert Vc.cpu().numpy().tobytes() == x["vc"].tobytes(), "V cache differs"
    ref = oracle.attention(qr.astype(np.float32), kc_ref.astype(np.float32), x["vc"], heads=H, headDim=D,
                           kvHeads=Hk, posOffset=pos, **oracle_params(params))
    err = max_err(out.cpu().numpy(), ref)
    assert err <= TOL, err


def test_decode_step_rope_workload():
    """The decode workload with Llama-3-style rotary embedding fused in: one
    new row at 32767 of the [32768, 1024] caches, theta 500000."""
    _rope_step_case(32768, 32, 8, 128, 1, 32767, 620, dict(base=500000.0))


@pytest.mark.parametrize("case", [
    dict(S=3000, H=16, Hk=4, D=128, new_rows=3, offset=2990, rope=dict(interleaved=True)),
    dict(S=3000, H=8, Hk=4, D=64, new_rows=1, offset=1200, rope=dict(rotaryDim=32), posOffset=2999),
    dict(S=2048, H=16, Hk=2, D=32, new_rows=2, offset=1000, rope=dict(scaling={"rope_type": "linear", "factor": 2.0}),
         window=300),
    dict(S=1500, H=8, Hk=1, D=128, new_rows=1, offset=1499, rope=dict(attentionFactor=0.75, base=1e6),
         softcap=30.0, alibi=True),
    dict(S=4000, H=16, Hk=4, D=128, new_rows=5, offset=1278, rope=dict(), decode_splits=7),
])
def test_decode_step_rope_cases(case):
    case = dict(case)
    _rope_step_case(case.pop("S"), case.pop("H"), case.pop("Hk"), case.pop("D"), case.pop("new_rows"),
                    case.pop("offset"), 621, case.pop("rope"), **case)


def test_spec_decode_step_rope_workload():
    """The 4-row speculative step (the tensor-core decode) with Llama-3-style
    rotary embedding fused in: four new rows at 32764 .. 32767 of the
    [32768, 1024] caches, theta 500000."""
    _rope_step_case(32768, 32, 8, 128, 4, 32764, 622, dict(base=500000.0), T=4)


@pytest.mark.parametrize("case", [
    dict(T=2, S=2500, H=16, Hk=2, new_rows=2, offset=2498, rope=dict(interleaved=True), window=500),
    dict(T=3, S=3000, H=12, Hk=3, new_rows=1, offset=2999, rope=dict(rotaryDim=64), posOffset=2997,
         window=700, sinks=40),
    dict(T=16, S=1800, H=4, Hk=4, new_rows=16, offset=1700, rope=dict(scaling={"rope_type": "linear", "factor": 4.0}),
         decode_splits=5),
    dict(T=4, S=900, H=8, Hk=2, new_rows=6, offset=600, rope=dict(attentionFactor=1.2, base=1e6), posOffset=896,
         scale=0.1),
    dict(T=8, S=4000, H=16, Hk=8, new_rows=0, offset=4000, rope=dict(rotaryDim=128, interleaved=True),
         posOffset=3992),
    dict(T=1, S=2100, H=16, Hk=1, new_rows=1, offset=2099, rope=dict(base=500000.0)),  # one row, group 16
])
def test_decode_step_rope_multi_row(case):
    """Query rows on the tensor-core decode (forced, so one row too): q row t
    turned at posOffset + t, the new keys at their cache rows (some of them
    outside the visible range, turned and written all the same)."""
    case = dict(case)
    _rope_step_case(case.pop("S"), case.pop("H"), case.pop("Hk"), 128, case.pop("new_rows"), case.pop("offset"),
                    623, case.pop("rope"), T=case.pop("T"), kernel=vtmu.VTMU_KERNEL_DECODE_TF32X3, **case)


def test_decode_step_rope_refuses_unaligned_rows_on_tensor_cores():
    """The tensor-core decode turns new keys only in its own fused write
    (float4 rows): 4- but not 16-byte aligned new rows are refused before any
    launch."""
    T, S, H, Hk, D = 2, 300, 8, 2, 128
    Kc = torch.zeros((S, Hk * D), device="cuda")
    Vc = torch.zeros((S, Hk * D), device="cuda")
    buf = torch.ones(T * Hk * D + 1, device="cuda")
    kn = buf[1:].view(T, Hk * D)
    with pytest.raises(vtmu.VtmuError) as e:
        vtmu.decode_step_rope(Kc, Vc, kn, kn.clone(), 100, torch.ones((T, H * D), device="cuda"), heads=H,
                              headDim=D, kvHeads=Hk, rope={})
    assert e.value.status == vtmu.VTMU_ERR_UNSUPPORTED and "compose" in str(e.value)
    torch.cuda.synchronize()
    assert torch.count_nonzero(Kc).item() == 0 and torch.count_nonzero(Vc).item() == 0


def test_decode_step_rope_refuses_unfused_shapes():
    """Only the fused form is offered: several rows outside the tensor-core
    decode's shapes, or a single row outside the decode kernel's, are refused
    before any launch (the caches stay as they were)."""
    Kc = torch.zeros((64, 2 * 96), device="cuda")
    Vc = torch.zeros((64, 2 * 96), device="cuda")
    kn = torch.ones((1, 2 * 96), device="cuda")
    with pytest.raises(vtmu.VtmuError) as e:  # headDim 96: not a decode-kernel shape
        vtmu.decode_step_rope(Kc, Vc, kn, kn.clone(), 10, torch.ones((1, 4 * 96), device="cuda"), heads=4,
                              headDim=96, kvHeads=2, rope={})
    assert e.value.status == vtmu.VTMU_ERR_UNSUPPORTED
    Kc = torch.zeros((64, 2 * 64), device="cuda")
    Vc = torch.zeros((64, 2 * 64), device="cuda")
    kn = torch.ones((3, 2 * 64), device="cuda")
    with pytest.raises(vtmu.VtmuError) as e:  # T = 3
        vtmu.decode_step_rope(Kc, Vc, kn, kn.clone(), 10, torch.ones((3, 4 * 64), device="cuda"), heads=4,
                              headDim=64, kvHeads=2, rope={})
    assert e.value.status == vtmu.VTMU_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.count_nonzero(Kc).item() == 0 and torch.count_nonzero(Vc).item() == 0
    assert vtmu.vtmu_device_error() == 0
