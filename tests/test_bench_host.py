"""The benchmark's work accounting on the host: visible-key counts (the
denominator of every TFLOP/s and GB/s figure) against a brute-force count
with the masking rule, and the algorithmic totals of the workloads."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import bench  # noqa: E402
import oracle_pins  # noqa: E402
import seeded_inputs as si  # noqa: E402


@pytest.mark.parametrize("seed", range(12))
def test_visible_counts_match_brute_force(seed):
    g = np.random.default_rng(seed)
    S = int(g.integers(1, 90))
    params = dict(causal=bool(g.integers(0, 2)), window=int(g.integers(0, 20)) if g.random() < 0.7 else 0,
                  sinks=int(g.integers(0, 12)) if g.random() < 0.6 else 0)
    pos = np.arange(int(g.integers(1, 40)), dtype=np.int64) + int(g.integers(0, 80))
    got = bench.visible_counts(pos, S, params)
    want = [sum(oracle_pins.visible(params["causal"], params["window"], int(p), s, params["sinks"]) for s in range(S))
            for p in pos]
    assert list(got) == want, (params, S)


def test_workload_totals():
    """Algorithmic work of the workloads (visible pairs x (2 headDim + 2 vHeadDim) FLOP for
    prefill; visible K/V rows, q/out rows and the new rows for decode)."""
    flops = {n: bench.prefill_flops(si.WORKLOADS[n]) for n in ("gqa_prefill", "swa_softcap_prefill",
                                                              "latent_bias_prefill", "alibi_prefill")}
    assert flops == {"gqa_prefill": 268500992 * 512, "swa_softcap_prefill": 402685952 * 1024,
                     "latent_bias_prefill": 536870912 * 640, "alibi_prefill": 67141632 * 512}
    assert bench.decode_bytes(si.WORKLOADS["gqa_decode"]) == (268435456, 268484608)
    # 4 query rows at 32764..32767 see all 32768 keys; 4 q/out rows and 4 new rows
    assert bench.decode_bytes(si.WORKLOADS["gqa_spec_decode"])[1] == 268435456 + 2 * 4 * 32 * 128 * 4 + 4 * 4 * 8 * 128 * 4
    # window 8188 + 4 sinks at 32767: 8192 key rows
    assert bench.decode_bytes(si.WORKLOADS["gqa_decode_sinks"])[0] == 2 * 8192 * 8 * 128 * 4
