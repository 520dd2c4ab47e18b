"""The CPU oracle against what the op catalog and mathematics fix (no GPU)."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import oracle  # noqa: E402
import oracle_pins  # noqa: E402


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=[p.__name__ for p in oracle_pins.ALL_PINS])
def test_oracle_pin(pin):
    pin(oracle.default())


def test_rows_match_full_output():
    import numpy as np
    g = np.random.default_rng(3)
    T, S, H, Hk, D, Dv = 9, 12, 4, 2, 8, 6
    q = g.standard_normal((T, H * D)).astype(np.float32)
    k = g.standard_normal((S, Hk * D)).astype(np.float32)
    v = g.standard_normal((S, Hk * Dv)).astype(np.float32)
    params = dict(heads=H, headDim=D, kvHeads=Hk, vHeadDim=Dv, posOffset=3, window=5,
                  softcap=3.0, alibi=True)
    full = oracle.attention(q, k, v, **params)
    rows = [(0, 0), (8, 3), (4, 1), (4, 2)]
    sel = oracle.attention_rows(q, k, v, rows=rows, **params)
    for i, (t, h) in enumerate(rows):
        assert np.array_equal(sel[i], full[t, h * Dv:(h + 1) * Dv])


def test_oracle_refuses_bad_shapes():
    import numpy as np
    q = np.zeros((2, 8), np.float32)
    with pytest.raises(ValueError):
        oracle.attention(q, np.zeros((3, 8), np.float32), np.zeros((3, 8), np.float32),
                         heads=3, headDim=8)
    with pytest.raises(ValueError):  # heads not a multiple of kvHeads
        oracle.attention(np.zeros((2, 12), np.float32), np.zeros((3, 8), np.float32),
                         np.zeros((3, 8), np.float32), heads=3, headDim=4, kvHeads=2)
