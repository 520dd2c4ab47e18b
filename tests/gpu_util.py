"""Helpers for the GPU parity tests: run the CUDA library through its C ABI
on seeded host inputs and compare with the CPU oracle on the same inputs."""
import numpy as np

TOL = 1e-4  # max |GPU - oracle|, absolute, outputs of order 1


def to_dev(x):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to("cuda")


def gpu_attention(q, k, v, bias=None, **params):
    """The library on host arrays; returns the f32 output as numpy."""
    import torch
    import f32_gqa_attention_gb300 as vtmu
    out = vtmu.attention(to_dev(q), to_dev(k), to_dev(v), to_dev(bias), **params)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def oracle_params(params):
    """Drop the library-only keywords before calling the oracle."""
    return {k: v for k, v in params.items() if k not in ("kernel", "decode_splits", "out",
                                                        "workspace", "stream")}


def max_err(a, b):
    if a.size == 0 and b.size == 0:
        return 0.0
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


def sample_rows(T, H, G, bm=(64, 128), extra=24, seed=0):
    """(t, h) rows that cover the first/last rows, tile edges, group edges and
    a few random ones."""
    g = np.random.default_rng(seed)
    ts = {0, 1, T - 1, T - 2, T // 2}
    for b in bm:
        ts.update({b - 1, b, 2 * b - 1, 2 * b})
    ts = sorted(t for t in ts if 0 <= t < T)
    hs = sorted({0, G - 1, G, H - 1, H // 2} & set(range(H)))
    rows = [(t, h) for t in ts for h in hs]
    rows += [(int(g.integers(0, T)), int(g.integers(0, H))) for _ in range(extra)]
    return rows


def sample_tile_rows(T, H, G, bm=128, seed=0):
    """One random row of every bm-row query tile for each of the heads 0,
    G - 1, H // 2 and H - 1 (the first and last group and the last head), so
    every (query tile, head group) work item of a full-size launch has a row
    checked."""
    g = np.random.default_rng(seed)
    hs = sorted({0, G - 1, H // 2, H - 1} & set(range(H)))
    rows = []
    for t0 in range(0, T, bm):
        t1 = min(T, t0 + bm)
        for h in hs:
            rows.append((int(g.integers(t0, t1)), h))
    return rows
