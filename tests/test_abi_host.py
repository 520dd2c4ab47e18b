"""The C-ABI library on the host (no GPU): it loads, exports every entry point
that include/*.h declares, and refuses bad requests before any launch."""
import glob
import os
import re

import pytest

import f32_gqa_attention_gb300 as vtmu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except ImportError:
        return False


# The tests below hand the library fake device addresses and rely on its host
# checks refusing each call before any launch.  They exist for the CPU-only
# machine; where a GPU is present they are skipped, so that a wrong check can
# never launch a kernel on those addresses.
host_only = pytest.mark.skipif(_has_gpu(), reason="host-only checks with fake device addresses")


@pytest.fixture(scope="module")
def lib():
    from f32_gqa_attention_gb300 import _build
    _build.build()
    return vtmu.load_library()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names.update(re.findall(r"VTMU_API\s+[\w\s\*]+?\b(vtmu_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("vtmu_attention", "vtmu_cache_write", "vtmu_attention_workspace_size",
              "vtmu_attention_params_init", "vtmu_features", "vtmu_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_symbols():
        assert hasattr(lib, n), f"libvtmu.so does not export {n}"


def test_exports_nothing_else(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", vtmu.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(declared_symbols()), exported ^ set(declared_symbols())


def test_features_name_the_catalog_features(lib):
    assert set(vtmu.vtmu_features().split()) == {
        "attention.alibi", "attention.bias", "attention.scale", "attention.softcap",
        "attention.window", "rope.interleaved", "rope.rotaryDim"}


def test_params_init_writes_defaults(lib):
    p = vtmu.vtmu_attention_params_init()
    assert p.causal == 1 and p.kv_heads == 0 and p.v_head_dim == 0 and p.has_scale == 0
    assert p.softcap == 0 and p.window == 0 and p.alibi == 0 and p.kernel == 0


def _err(fn):
    with pytest.raises(vtmu.VtmuError) as e:
        fn()
    return e.value


FAKE = 1 << 40  # never dereferenced: every case below fails before a launch


@host_only
@pytest.mark.parametrize("kw,status,word", [
    (dict(heads=3, headDim=8, kvHeads=2), vtmu.VTMU_ERR_INVALID, "multiple of kvHeads"),
    (dict(heads=0, headDim=8), vtmu.VTMU_ERR_INVALID, "heads"),
    (dict(heads=2, headDim=0), vtmu.VTMU_ERR_INVALID, "headDim"),
    (dict(heads=2, headDim=300), vtmu.VTMU_ERR_UNSUPPORTED, "headDim 300"),
    (dict(heads=2, headDim=8, vHeadDim=512), vtmu.VTMU_ERR_UNSUPPORTED, "vHeadDim 512"),
    (dict(heads=2, headDim=8, window=-1), vtmu.VTMU_ERR_INVALID, "window"),
    (dict(heads=2, headDim=8, softcap=-1.0), vtmu.VTMU_ERR_INVALID, "softcap"),
    (dict(heads=2, headDim=8, scale=float("inf")), vtmu.VTMU_ERR_INVALID, "scale"),
    (dict(heads=2, headDim=8, posOffset=-3), vtmu.VTMU_ERR_RANGE, "posOffset"),
    (dict(heads=2, headDim=8, alibiMax=-1.0), vtmu.VTMU_ERR_INVALID, "alibiMax"),
    (dict(heads=1024, headDim=8, alibi=True), vtmu.VTMU_ERR_UNSUPPORTED, "attention.alibi"),
])
def test_invalid_params_are_refused(lib, kw, status, word):
    p = vtmu.make_params(4, 4, **kw)
    e = _err(lambda: vtmu.vtmu_attention(FAKE, FAKE, FAKE, None, FAKE * 2, p, None, 0, 0))
    assert e.status == status and word in str(e), str(e)
    assert word in vtmu.vtmu_last_error()


@host_only
def test_decode_kernel_row_limit(lib):
    p = vtmu.make_params(17, 64, heads=4, headDim=64, kernel=vtmu.VTMU_KERNEL_DECODE)
    e = _err(lambda: vtmu.vtmu_attention(FAKE, FAKE, FAKE, None, FAKE * 2, p, None, 0, 0))
    assert e.status == vtmu.VTMU_ERR_INVALID and "1 <= T <= 16" in str(e)


@host_only
def test_decode_shape_outside_its_table_is_refused(lib):
    p = vtmu.make_params(1, 64, heads=4, headDim=96, kvHeads=2, kernel=vtmu.VTMU_KERNEL_DECODE)
    e = _err(lambda: vtmu.vtmu_attention(FAKE, FAKE, FAKE, None, FAKE * 2, p, None, 0, 0))
    assert e.status == vtmu.VTMU_ERR_UNSUPPORTED


@host_only
@pytest.mark.parametrize("kw", [
    dict(T=4, heads=32, kvHeads=4, headDim=128),             # group 8 x 4 rows: 32 virtual heads
    dict(T=2, heads=4, kvHeads=2, headDim=96),               # headDim other than 128
    dict(T=2, heads=4, kvHeads=2, headDim=64),
    dict(T=2, heads=4, kvHeads=2, headDim=128, softcap=30.0),
    dict(T=2, heads=4, kvHeads=2, headDim=128, alibi=True),
    dict(T=2, heads=4, kvHeads=2, headDim=128, vHeadDim=64),
    dict(T=2, heads=16385, kvHeads=16385, headDim=128),     # more KV heads than arrival counters
])
def test_tensor_core_decode_outside_its_shapes_is_refused(lib, kw):
    kw = dict(kw)
    p = vtmu.make_params(kw.pop("T"), 300, kernel=vtmu.VTMU_KERNEL_DECODE_TF32X3, **kw)
    e = _err(lambda: vtmu.vtmu_attention_workspace_size(p))
    assert e.status == vtmu.VTMU_ERR_UNSUPPORTED and "DECODE_TF32X3" in str(e)


@host_only
def test_unknown_kernel_is_refused(lib):
    p = vtmu.make_params(2, 300, heads=4, headDim=64, kernel=vtmu.VTMU_KERNEL_DECODE_TF32X3 + 1)
    e = _err(lambda: vtmu.vtmu_attention_workspace_size(p))
    assert e.status == vtmu.VTMU_ERR_INVALID and "vtmu_kernel" in str(e)


@host_only
def test_null_and_aliasing_pointers_are_refused(lib):
    p = vtmu.make_params(4, 4, heads=2, headDim=8)
    assert _err(lambda: vtmu.vtmu_attention(None, FAKE, FAKE, None, FAKE * 2, p, None, 0, 0)).status == \
        vtmu.VTMU_ERR_INVALID
    assert "overlaps" in str(_err(lambda: vtmu.vtmu_attention(FAKE, FAKE * 3, FAKE * 3, None, FAKE + 16, p,
                                                              None, 0, 0)))
    assert "4-byte" in str(_err(lambda: vtmu.vtmu_attention(FAKE + 2, FAKE * 3, FAKE * 3, None, FAKE * 2, p,
                                                            None, 0, 0)))
    pb = vtmu.make_params(4, 4, heads=2, headDim=8, bias_kind=vtmu.VTMU_BIAS_TS)
    assert "attention.bias" in str(_err(lambda: vtmu.vtmu_attention(FAKE, FAKE * 3, FAKE * 3, None, FAKE * 2,
                                                                    pb, None, 0, 0)))


@host_only
def test_decode_needs_its_workspace(lib):
    p = vtmu.make_params(1, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4095)
    need = vtmu.vtmu_attention_workspace_size(p)
    assert need > 0
    e = _err(lambda: vtmu.vtmu_attention(FAKE, FAKE * 3, FAKE * 5, None, FAKE * 2, p, FAKE * 7, need - 1, 0))
    assert e.status == vtmu.VTMU_ERR_WORKSPACE
    e = _err(lambda: vtmu.vtmu_attention(FAKE, FAKE * 3, FAKE * 5, None, FAKE * 2, p, FAKE * 7 + 16, need, 0))
    assert e.status == vtmu.VTMU_ERR_WORKSPACE and "256-byte" in str(e)


def test_ffma_prefill_needs_no_workspace(lib):
    p = vtmu.make_params(64, 64, heads=4, headDim=64, kernel=vtmu.VTMU_KERNEL_PREFILL_FFMA)
    assert vtmu.vtmu_attention_workspace_size(p) == 0
    assert vtmu.vtmu_attention_workspace_size(vtmu.make_params(16, 16, heads=4, headDim=32)) == 0


def test_tensor_core_prefill_workspace_holds_the_split_operands(lib):
    S, Hk, D = 1000, 2, 128
    p = vtmu.make_params(256, S, heads=4, headDim=D, kvHeads=Hk)  # AUTO picks the tcgen05 prefill
    assert vtmu.vtmu_attention_workspace_size(p) >= 4 * S * Hk * D * 4


@host_only
def test_tensor_core_prefill_shape_table(lib):
    p = vtmu.make_params(256, 256, heads=4, headDim=160, kernel=vtmu.VTMU_KERNEL_PREFILL_TF32X3)
    e = _err(lambda: vtmu.vtmu_attention(FAKE, FAKE, FAKE, None, FAKE * 2, p, None, 0, 0))
    assert e.status == vtmu.VTMU_ERR_UNSUPPORTED and "PREFILL_TF32X3" in str(e)


@host_only
def test_zero_query_rows_is_a_no_op(lib):
    vtmu.vtmu_attention(None, None, None, None, None, vtmu.make_params(0, 5, heads=2, headDim=8), None, 0, 0)


@host_only
@pytest.mark.parametrize("args,status", [
    ((FAKE, 10, 4, FAKE * 2, 2, 9), vtmu.VTMU_ERR_RANGE),
    ((FAKE, 10, 4, FAKE * 2, 2, -1), vtmu.VTMU_ERR_RANGE),
    ((FAKE, 10, 4, FAKE * 2, -1, 0), vtmu.VTMU_ERR_INVALID),
    ((None, 10, 4, FAKE * 2, 1, 0), vtmu.VTMU_ERR_INVALID),
    ((FAKE, 10, 4, FAKE + 16, 2, 0), vtmu.VTMU_ERR_INVALID),  # values overlap the rows written
])
def test_cache_write_refusals(lib, args, status):
    e = _err(lambda: vtmu.vtmu_cache_write(*args))
    assert e.status == status


@host_only
def test_cache_write_empty_is_a_no_op(lib):
    vtmu.vtmu_cache_write(None, 10, 4, None, 0, 10)


@host_only
def test_noalloc_refuses_a_shape_beyond_its_scratch(lib):
    p = vtmu.make_params(1, 32768, heads=64, headDim=128, kvHeads=8, posOffset=32767)
    e = _err(lambda: vtmu.vtmu_attention_decode_noalloc(FAKE, FAKE * 3, FAKE * 5, None, FAKE * 7, p, 0))
    assert e.status == vtmu.VTMU_ERR_WORKSPACE and "static scratch" in str(e)


@host_only
def test_noalloc_checks_parameters_first(lib):
    p = vtmu.make_params(1, 64, heads=3, headDim=128, kvHeads=2)
    e = _err(lambda: vtmu.vtmu_attention_decode_noalloc(FAKE, FAKE * 3, FAKE * 5, None, FAKE * 7, p, 0))
    assert e.status == vtmu.VTMU_ERR_INVALID


@host_only
def test_device_error_needs_an_output(lib):
    assert lib.vtmu_device_error(None) == vtmu.VTMU_ERR_INVALID


def test_host_decode_step_workspace_adds_the_staging_areas(lib):
    """vtmu_decode_step_host's workspace: the attention workspace, then q, the
    new rows, the bias and out, each on a 256-byte boundary."""
    p = vtmu.make_params(1, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4095)
    base = vtmu.vtmu_attention_workspace_size(p)
    up = lambda n: (n + 255) // 256 * 256
    want = up(base) + up(32 * 128 * 4) + 2 * up(3 * 8 * 128 * 4) + up(32 * 128 * 4)
    assert vtmu.vtmu_decode_step_host_workspace_size(p, 3) == want
    pb = vtmu.make_params(1, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4095, bias_kind=vtmu.VTMU_BIAS_HTS)
    assert vtmu.vtmu_decode_step_host_workspace_size(pb, 3) == want + up(32 * 4096 * 4)
    assert _err(lambda: vtmu.vtmu_decode_step_host_workspace_size(p, -1)).status == vtmu.VTMU_ERR_INVALID


@host_only
def test_host_decode_step_checks_before_any_copy(lib):
    import numpy as np

    p = vtmu.make_params(1, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4095)
    need = vtmu.vtmu_decode_step_host_workspace_size(p, 1)
    q = np.zeros((1, 32 * 128), np.float32)
    kn = np.zeros((1, 8 * 128), np.float32)
    out = np.zeros((1, 32 * 128), np.float32)
    call = lambda **o: _err(lambda: vtmu.vtmu_decode_step_host(
        o.get("kc", FAKE * 3), FAKE * 5, o.get("rows", 4096), kn, kn, 1, o.get("off", 4095), o.get("q", q),
        o.get("b"), out, o.get("p", p), o.get("ws", FAKE * 7), o.get("wsb", need), 0))
    assert call(wsb=need - 1).status == vtmu.VTMU_ERR_WORKSPACE
    assert "256-byte" in str(call(ws=FAKE * 7 + 16))
    assert call(q=None).status == vtmu.VTMU_ERR_INVALID
    assert call(off=4096).status == vtmu.VTMU_ERR_RANGE
    assert "attention.bias" in str(call(b=q))
    assert call(kc=None).status == vtmu.VTMU_ERR_INVALID
    assert call(rows=4000, off=3000).status == vtmu.VTMU_ERR_INVALID  # S > max_rows
    with pytest.raises(ValueError):
        vtmu.vtmu_decode_step_host(FAKE * 3, FAKE * 5, 4096, kn, kn, 1, 4095, q.astype(np.float64), None, out, p,
                                   FAKE * 7, need, 0)


@host_only
def test_rope_refusals(lib):
    ok = dict(headDim=64)
    call = lambda T=4, heads=2, off=0, x=FAKE, out=FAKE * 2, **kw: _err(
        lambda: vtmu.vtmu_rope(x, out, T, heads, off, vtmu.make_rope_params(**dict(ok, **kw)), 0))
    assert "rope.rotaryDim" in str(call(rotaryDim=33))
    assert "rope.rotaryDim" in str(call(rotaryDim=66))
    assert call(headDim=4096 + 2).status == vtmu.VTMU_ERR_INVALID
    assert call(headDim=512, rotaryDim=512).status == vtmu.VTMU_ERR_UNSUPPORTED
    e = call(scaling={"rope_type": "yarn", "factor": 4.0})
    assert e.status == vtmu.VTMU_ERR_UNSUPPORTED and "rope.scaling" in str(e)
    assert "rope.scaling" in str(call(scaling={"rope_type": "linear", "factor": 0.0}))
    assert call(base=-1.0).status == vtmu.VTMU_ERR_INVALID
    assert call(invFreq=[float("nan")] * 32).status == vtmu.VTMU_ERR_INVALID
    assert call(off=-1).status == vtmu.VTMU_ERR_RANGE
    assert call(x=None).status == vtmu.VTMU_ERR_INVALID
    assert call(heads=0).status == vtmu.VTMU_ERR_INVALID
    assert "overlaps" in str(call(out=FAKE + 4))
    vtmu.vtmu_rope(None, None, 0, 2, 0, vtmu.make_rope_params(headDim=64), 0)  # T == 0: nothing to do


@host_only
def test_decode_step_rope_refusals(lib):
    p = vtmu.make_params(1, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4095)
    need = vtmu.vtmu_attention_workspace_size(p)
    r = vtmu.make_rope_params(headDim=128)
    call = lambda p=p, r=r: _err(lambda: vtmu.vtmu_decode_step_rope(
        FAKE * 3, FAKE * 5, 4096, FAKE * 7, FAKE * 9, 1, 4095, FAKE, None, FAKE * 2, p, r, FAKE * 11, need, 0))
    assert "head_dim" in str(call(r=vtmu.make_rope_params(headDim=64)))
    e = call(p=vtmu.make_params(1, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4095,
                                kernel=vtmu.VTMU_KERNEL_PREFILL_FFMA))
    assert e.status == vtmu.VTMU_ERR_UNSUPPORTED and "compose" in str(e)
    # 5 rows x group 4 = 20 virtual heads: past the tensor-core decode, and
    # the CUDA-core decode turns one row only
    e = call(p=vtmu.make_params(5, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4091))
    assert e.status == vtmu.VTMU_ERR_UNSUPPORTED
    e = call(p=vtmu.make_params(2, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4094,
                                kernel=vtmu.VTMU_KERNEL_DECODE))
    assert e.status == vtmu.VTMU_ERR_UNSUPPORTED and "compose" in str(e)
    e = call(p=vtmu.make_params(0, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4095))
    assert e.status == vtmu.VTMU_ERR_UNSUPPORTED and "T = 0" in str(e)
    assert call(r=vtmu.make_rope_params(headDim=128, rotaryDim=130)).status == vtmu.VTMU_ERR_INVALID


@host_only
def test_negative_sinks_are_refused(lib):
    p = vtmu.make_params(4, 4, heads=2, headDim=8, window=2, sinks=-1)
    e = _err(lambda: vtmu.vtmu_attention(FAKE, FAKE, FAKE, None, FAKE * 2, p, None, 0, 0))
    assert e.status == vtmu.VTMU_ERR_INVALID and "sinks" in str(e)


def test_binding_lists_every_entry_point(lib):
    """The binding's EXPORTED names are exactly the entry points the header declares."""
    hdr = open(os.path.join(ROOT, "include", "vtmu_attention.h")).read()
    declared = set(re.findall(r"VTMU_API\s+[\w\s\*]+?\b(vtmu_\w+)\s*\(", hdr))
    assert set(vtmu.EXPORTED) == declared


@host_only
def test_noalloc_needs_one_query_row(lib):
    p = vtmu.make_params(2, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4094)
    e = _err(lambda: vtmu.vtmu_attention_decode_noalloc(FAKE, FAKE * 3, FAKE * 5, None, FAKE * 7, p, 0))
    assert e.status == vtmu.VTMU_ERR_INVALID and "T must be 1" in str(e)


@host_only
def test_noalloc_takes_only_the_decode_kernel(lib):
    p = vtmu.make_params(1, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4095,
                         kernel=vtmu.VTMU_KERNEL_PREFILL_FFMA)
    e = _err(lambda: vtmu.vtmu_attention_decode_noalloc(FAKE, FAKE * 3, FAKE * 5, None, FAKE * 7, p, 0))
    assert e.status == vtmu.VTMU_ERR_INVALID and "VTMU_KERNEL_DECODE" in str(e)


@host_only
def test_noalloc_checks_pointers_before_touching_its_scratch(lib):
    """Null, misaligned and overlapping pointers are refused before the call
    clears the shared array's counters (no CUDA call is made on this host)."""
    p = vtmu.make_params(1, 4096, heads=32, headDim=128, kvHeads=8, posOffset=4095)
    e = _err(lambda: vtmu.vtmu_attention_decode_noalloc(FAKE, FAKE * 3, FAKE * 5, None, None, p, 0))
    assert e.status == vtmu.VTMU_ERR_INVALID and "out is NULL" in str(e)
    e = _err(lambda: vtmu.vtmu_attention_decode_noalloc(FAKE + 4, FAKE * 3, FAKE * 5, None, FAKE * 7, p, 0))
    assert e.status == vtmu.VTMU_ERR_UNSUPPORTED and "16-byte" in str(e)
    e = _err(lambda: vtmu.vtmu_attention_decode_noalloc(FAKE, FAKE * 3, FAKE * 5, None, FAKE * 3, p, 0))
    assert e.status == vtmu.VTMU_ERR_INVALID and "overlaps" in str(e)
    e = _err(lambda: vtmu.vtmu_attention_decode_noalloc(FAKE, FAKE * 3, FAKE * 5, FAKE * 9, FAKE * 7, p, 0))
    assert e.status == vtmu.VTMU_ERR_INVALID and "bias" in str(e)


def test_noalloc_scratch_limit_in_virtual_heads(lib):
    """Over 32768 keys at vHeadDim 128 the static scratch holds 62 virtual
    heads: 62 query heads with groups of two or more, 31 when every query
    head has its own KV head (each KV head is padded to two virtual heads)."""
    def need(H, Hk):
        return vtmu.vtmu_attention_workspace_size(vtmu.make_params(
            1, 32768, heads=H, headDim=128, kvHeads=Hk, posOffset=32767, kernel=vtmu.VTMU_KERNEL_DECODE))
    cap = vtmu.NOALLOC_SCRATCH_BYTES
    assert need(62, 31) <= cap < need(64, 32)
    assert need(31, 31) <= cap < need(32, 32)


# ---- absorbed latent attention ------------------------------------------------
def test_mla_params_init_writes_defaults(lib):
    p = vtmu.vtmu_mla_params_init()
    assert p.causal == 1 and p.kv_rank == 512 and p.qk_rope == 64 and p.has_scale == 0 and p.window == 0


@pytest.mark.parametrize("kw,status,word", [
    (dict(kv_rank=256), vtmu.VTMU_ERR_UNSUPPORTED, "kv_rank"),
    (dict(qk_rope=32), vtmu.VTMU_ERR_UNSUPPORTED, "qk_rope"),
    (dict(qk_nope=600), vtmu.VTMU_ERR_UNSUPPORTED, "qk_nope"),
    (dict(v_head_dim=0), vtmu.VTMU_ERR_INVALID, "v_head_dim"),
    (dict(heads=0), vtmu.VTMU_ERR_INVALID, "heads"),
    (dict(posOffset=-1), vtmu.VTMU_ERR_RANGE, "posOffset"),
    (dict(window=-2), vtmu.VTMU_ERR_INVALID, "window"),
    (dict(scale=float("inf")), vtmu.VTMU_ERR_INVALID, "scale"),
    (dict(T=4097, heads=16), vtmu.VTMU_ERR_UNSUPPORTED, "T * heads"),
    (dict(kernel=3), vtmu.VTMU_ERR_INVALID, "kernel"),
    (dict(kernel=-1), vtmu.VTMU_ERR_INVALID, "kernel"),
])
def test_mla_invalid_params_are_refused(lib, kw, status, word):
    base = dict(T=1, S=128, heads=4, qk_nope=64, v_head_dim=64)
    base.update(kw)
    T, S = base.pop("T"), base.pop("S")
    e = _err(lambda: vtmu.vtmu_mla_workspace_size(vtmu.make_mla_params(T, S, **base)))
    assert e.status == status and word in str(e), str(e)


def test_mla_workspace_holds_queries_and_partials(lib):
    """The workspace holds the header, the absorbed queries (T * heads rows of
    576 floats) and at least one split's partials per virtual head."""
    p = vtmu.make_mla_params(1, 32768, heads=16, qk_nope=128, v_head_dim=128, posOffset=32767)
    n = vtmu.vtmu_mla_workspace_size(p)
    assert n >= 64 * 1024 + 16 * 576 * 4 + 16 * (512 + 2) * 4
    assert n < 64 * 1024 * 1024


@host_only
def test_mla_pointer_checks(lib):
    p = vtmu.make_mla_params(1, 128, heads=4, qk_nope=64, v_head_dim=64, posOffset=127)
    n = vtmu.vtmu_mla_workspace_size(p)
    e = _err(lambda: vtmu.vtmu_mla_attention(FAKE, None, FAKE * 5, FAKE * 7, FAKE * 9, p, FAKE * 11, n, 0))
    assert e.status == vtmu.VTMU_ERR_INVALID and "NULL" in str(e)
    e = _err(lambda: vtmu.vtmu_mla_attention(FAKE, FAKE * 3 + 4, FAKE * 5, FAKE * 7, FAKE * 9, p, FAKE * 11, n, 0))
    assert e.status == vtmu.VTMU_ERR_INVALID and "16-byte" in str(e)
    e = _err(lambda: vtmu.vtmu_mla_attention(FAKE, FAKE * 3, FAKE * 5, FAKE * 7, FAKE * 3, p, FAKE * 11, n, 0))
    assert e.status == vtmu.VTMU_ERR_INVALID and "overlaps" in str(e)
    e = _err(lambda: vtmu.vtmu_mla_attention(FAKE, FAKE * 3, FAKE * 5, FAKE * 7, FAKE * 9, p, FAKE * 11, n - 256, 0))
    assert e.status == vtmu.VTMU_ERR_WORKSPACE
    e = _err(lambda: vtmu.vtmu_mla_decode_step(FAKE * 3, 128, FAKE * 13, 1, 128, FAKE, FAKE * 5, FAKE * 7,
                                               FAKE * 9, p, FAKE * 11, n, 0))
    assert e.status == vtmu.VTMU_ERR_RANGE


def test_host_mla_decode_step_workspace_adds_the_staging_areas(lib):
    """vtmu_mla_decode_step_host's workspace: the latent attention's
    workspace, then q, the new latent rows and out, each on a 256-byte
    boundary."""
    p = vtmu.make_mla_params(2, 4096, heads=16, qk_nope=128, v_head_dim=128, posOffset=4094)
    base = vtmu.vtmu_mla_workspace_size(p)
    up = lambda n: (n + 255) // 256 * 256
    want = up(base) + up(2 * 16 * (128 + 64) * 4) + up(3 * 576 * 4) + up(2 * 16 * 128 * 4)
    assert vtmu.vtmu_mla_decode_step_host_workspace_size(p, 3) == want
    assert _err(lambda: vtmu.vtmu_mla_decode_step_host_workspace_size(p, -1)).status == vtmu.VTMU_ERR_INVALID


@host_only
def test_host_mla_decode_step_checks_before_any_copy(lib):
    import numpy as np

    p = vtmu.make_mla_params(1, 4096, heads=16, qk_nope=128, v_head_dim=128, posOffset=4095)
    need = vtmu.vtmu_mla_decode_step_host_workspace_size(p, 1)
    q = np.zeros((1, 16 * 192), np.float32)
    sn = np.zeros((1, 576), np.float32)
    out = np.zeros((1, 16 * 128), np.float32)
    call = lambda **o: _err(lambda: vtmu.vtmu_mla_decode_step_host(
        o.get("state", FAKE * 3), o.get("rows", 4096), o.get("sn", sn), 1, o.get("off", 4095), o.get("q", q),
        o.get("kb", FAKE * 5), FAKE * 7, out, p, o.get("ws", FAKE * 9), o.get("wsb", need), 0))
    assert call(wsb=need - 1).status == vtmu.VTMU_ERR_WORKSPACE
    assert "256-byte" in str(call(ws=FAKE * 9 + 16))
    assert call(q=None).status == vtmu.VTMU_ERR_INVALID
    assert call(sn=None).status == vtmu.VTMU_ERR_INVALID
    assert call(off=4096).status == vtmu.VTMU_ERR_RANGE
    assert call(rows=4000, off=3000).status == vtmu.VTMU_ERR_INVALID  # S > max_rows
    assert call(state=None).status == vtmu.VTMU_ERR_INVALID
    assert call(kb=None).status == vtmu.VTMU_ERR_INVALID
    assert "16-byte" in str(call(state=FAKE * 3 + 4))
