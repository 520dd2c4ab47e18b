"""Benchmark of the f32 attention library on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl vtmu|reference]
                    [--workload NAME] [--kernel auto|tc|ffma] [--no-cpu-baseline]
                    [--no-prefill] [--no-mla] [--no-rows] [--cpu-budget SEC]
                    [--prefill-cpu-budget SEC]

Workloads (seeded_inputs.WORKLOADS): gqa_decode (default), gqa_decode_rope
(the same step with the rotary embedding fused in), gqa_spec_decode (4 query
rows), gqa_decode_sinks (a window with attention sinks), gqa_prefill,
swa_softcap_prefill, swa_sinks_prefill, latent_bias_prefill, alibi_prefill,
tiny_prefill, mla_decode and mla_decode_v3 (absorbed latent attention, 16 and
128 heads).  `--kernel ffma` forces the FFMA prefill (for a decode workload:
the step as cache_writes + the FFMA prefill), `--kernel tc` the tensor cores.

Default workload: the GQA decode step (Llama-3-8B shape): cache_write of one
new K row and one new V row at position 32767 into [32768, 8*128] f32 caches,
then attention with T = 1 over S = 32768 keys, 32 query heads, 8 KV heads,
headDim 128.  A step is that whole decode step, run as one fused launch
(vtmu_decode_step); the line also reports the same step as three separate
launches (`unfused_ms_per_step`).  Two independent caches
(sessions) alternate between steps, so each step reads its 256 MiB of K/V
from HBM (working set 512 MiB > the 126 MiB L2).

One JSON line is printed by rank 0.  `value` is whole-job throughput in the
workload's unit (decode: algorithmic GB/s; prefill: algorithmic TFLOP/s).
After a decode workload the line also carries `prefill`: one entry per
prefill workload (gqa_prefill, swa_softcap_prefill, latent_bias_prefill,
alibi_prefill) with its step and kernel time, TFLOP/s, its tensor-pipe
roofline against two ceilings (the measured bf16 rate scaled to 3xTF32, and
the measured kind::tf32 rate per SM at the sampled SM clock), end-to-end
TFLOP/s from host buffers and a bounded oracle sample; `--no-prefill` leaves
them out.  It also carries `mla`: the latent-attention decode step (mla_decode,
DeepSeek-V2-Lite's shape) with its GB/s and both rooflines (`--no-mla`), and
(default workload only) `decode_rows`: the 4-row speculative step
(gqa_spec_decode, the tensor-core decode) with its GB/s and HBM roofline
(`--no-rows`).  `--impl reference` times the CPU oracle on the host cores
instead, on a bounded sample of the same workload.

N > 1 (torchrun): every rank runs an independent replica on its own GPU (the
op has no exchange step); ranks meet at a barrier around the timed region
and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

METRIC = "f32 attention: decode KV GB/s and prefill TFLOP/s on 1 GB300, % of roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
SMS = 152
FP32_LANES_PER_SM = 128


# ------------------------------------------------------------------ work model
def decode_bytes(w):
    """Algorithmic bytes of one decode step: every K and V row some query row
    sees once, the query and output rows once, and the two cache writes of
    the new rows (read + write)."""
    H, Hk, D, R = w["heads"], w["kvHeads"], w["headDim"], w.get("rows", 1)
    S = w["offset"] + R
    p = w["params"]
    seen = np.zeros(S, dtype=bool)
    for t in range(R):
        pos = p.get("posOffset", 0) + t
        s = np.arange(S)
        vis = np.ones(S, dtype=bool)
        if p.get("causal", True):
            vis &= s <= pos
        win = p.get("window") or 0
        if win:
            inw = (s > pos - win) if p.get("causal", True) else (np.abs(pos - s) <= win)
            vis &= inw | (s < (p.get("sinks") or 0))
        seen |= vis
    kv = 2 * int(seen.sum()) * Hk * D * 4
    qo = 2 * R * H * D * 4
    cw = 2 * 2 * R * Hk * D * 4
    return kv, kv + qo + cw


def visible_counts(pos, S, params):
    """Visible keys of query rows at positions `pos` (numpy int64), from the
    op's masking rule: the causal limit, the window, and attention sinks
    (keys before `sinks` escape the window)."""
    causal = params.get("causal", True)
    win = params.get("window") or 0
    sinks = params.get("sinks") or 0
    if causal:
        hi = np.minimum(pos, S - 1)
        lo = np.maximum(pos - win + 1, 0) if win else np.zeros_like(pos)
    else:
        lo = np.maximum(pos - win, 0) if win else np.zeros_like(pos)
        hi = np.minimum(pos + win, S - 1) if win else np.full_like(pos, S - 1)
    n = np.maximum(hi - lo + 1, 0)
    if win and sinks:
        cap = np.minimum(sinks, hi + 1) if causal else np.full_like(pos, min(sinks, S))
        n = n + np.maximum(np.minimum(cap, lo), 0) + np.maximum(cap - (hi + 1), 0)
    return n


def visible_pairs(w):
    """Visible (query, key) pairs per head, from the op's masking rule."""
    pos = np.arange(w["T"], dtype=np.int64) + w["params"].get("posOffset", 0)
    return int(visible_counts(pos, w["S"], w["params"]).sum())


def prefill_flops(w):
    D = w["headDim"]
    Dv = w.get("vHeadDim") or D
    return visible_pairs(w) * w["heads"] * (2 * D + 2 * Dv)


def mla_work(w):
    """Algorithmic bytes and FLOPs of one latent-attention decode step: the
    visible cache rows once (576 floats each), k_b and v_b once, q and out,
    the new cache rows read and written; FLOPs of the absorbed form (query
    absorption, 2 x 576 + 2 x 512 per visible (row, head, key), the output
    projection)."""
    H, R, N, P, Dv, off = w["heads"], w["kv_rank"], w["qk_nope"], w["qk_rope"], w["v_head_dim"], w["offset"]
    T = w.get("rows", 1)
    S = off + T
    pos = np.arange(T, dtype=np.int64) + w["params"].get("posOffset", 0)
    seen = np.zeros(S, dtype=bool)
    for p in pos:
        s = np.arange(S)
        vis = s <= p if w["params"].get("causal", True) else np.ones(S, dtype=bool)
        seen |= vis
    Wd = R + P
    nbytes = (int(seen.sum()) * Wd + H * N * R + H * Dv * R + T * H * (N + P) + T * H * Dv + 2 * T * Wd) * 4
    pairs = int(visible_counts(pos, S, w["params"]).sum())
    flops = 2 * T * H * N * R + pairs * H * (2 * Wd + 2 * R) + 2 * T * H * Dv * R
    return nbytes, flops


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
                "sm_max_mhz": 2070.0}, "fallback"


PREFILL_SET = ("gqa_prefill", "swa_softcap_prefill", "latent_bias_prefill", "alibi_prefill")
# kind::tf32 MMA throughput per SM measured on this GPU (one CTA, M = 128,
# N = 128, K = 8 every 64 cycles): the tensor pipe's clock-scaled ceiling.
TF32_FLOP_PER_CYCLE_SM = 4096


def kernel_source_hash(kernel_tag):
    """sha256 over a kernel's .cu file and every library header it includes
    (transitively), in a fixed order: a committed ncu summary is trusted only
    while this matches the hash it records."""
    csrc = os.path.join(ROOT, "f32_gqa_attention_gb300", "csrc")
    seen, order = set(), []

    def visit(fname):
        if fname in seen:
            return
        seen.add(fname)
        path = os.path.join(csrc, fname)
        data = open(path, "rb").read()
        order.append((fname, data))
        for inc in re.findall(rb'#include\s+"([^"]+)"', data):
            inc = inc.decode()
            if os.path.exists(os.path.join(csrc, inc)):
                visit(inc)

    try:
        visit(kernel_tag + ".cu")
    except OSError:
        return None
    h = hashlib.sha256()
    first, rest = order[0], sorted(order[1:])
    for fname, data in [first] + rest:
        h.update(fname.encode() + b"\0" + data + b"\0")
    return h.hexdigest()


def profile_info(profile_name):
    """Figures from a committed ncu summary `profiles/<kernel>__<workload>.md`
    (traffic per launch, tensor-pipe busy %), when the kernel source it was
    taken on is unchanged; {} otherwise."""
    path = os.path.join(ROOT, "profiles", f"{profile_name}.md")
    try:
        text = open(path).read()
    except OSError:
        return {}
    s = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    if not s or s.group(1) != kernel_source_hash(profile_name.split("__")[0]):
        return {}
    info = {}
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if m:
        info["traffic"] = int(m.group(1))
    m = re.search(r"tensor_pipe_active_pct:\s*([0-9.]+)", text)
    if m:
        info["tensor_pipe_active_pct"] = float(m.group(1))
    return info


def profile_traffic(profile_name):
    return profile_info(profile_name).get("traffic")


def tensor_ceilings(peaks, sm_mhz):
    """The 3xTF32 ceilings of the tensor pipe, in TFLOP/s: (measured bf16
    burst x 1.1/2.25 (tf32/bf16 nominal) / 3, measured kind::tf32 rate per SM
    x SMs x SM clock / 3).  Three tf32 products make one f32 product."""
    bf16_scaled = float(peaks["bf16_tflops"]) * (1.1 / 2.25) / 3.0
    clk = SMS * TF32_FLOP_PER_CYCLE_SM * float(sm_mhz) * 1e6 / 3.0 / 1e12
    return bf16_scaled, clk


# -------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running; summaries
    for any wall-clock window of the run."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.rows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        self.proc = None
        for ln in out.splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                self.rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue

    def summary(self, t0, t1):
        """Median SM clock, max clock and active throttle reasons of the
        samples inside [t0, t1] (timestamps have one-second resolution)."""
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sel = [r for r in self.rows if t0 - 1 <= r[0] <= t1 + 1] or self.rows[-3:]
        reasons = sorted({self.REASONS[i] for r in sel for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": reasons, "samples": len(sel)}


# ------------------------------------------------------------------ helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def workload_config(name, world):
    """The `config` object of a JSON line: the workload's shape and params,
    the replica count and how L2 is kept out of the timing (the same for both
    arms)."""
    w = si.WORKLOADS[name]
    l2 = {"decode": "inputs > L2: two 256 MiB K/V cache sets alternate between steps",
          "mla_decode": "inputs > L2: four 72 MiB latent caches alternate between steps"}.get(
        w["kind"], "L2 flushed between timed steps (256 MiB write, outside the timed events)")
    return {"workload": name, **{k: w[k] for k in w if k not in ("params", "kind")}, **w["params"],
            "parallelism": f"replicas x{world}", "l2": l2}


DATA = "synthetic (seeded SplitMix64 / Box-Muller, N(0,1) inputs of the workload's shapes)"


# ------------------------------------------------------------- oracle timing
def oracle_decode_step(x, w):
    import oracle
    H, Hk, D, off = w["heads"], w["kvHeads"], w["headDim"], w["offset"]
    q, kn = x["q"], x["k_new"]
    if w.get("rope"):  # op rope on q (at posOffset) and on the new key row (at its cache row)
        q = oracle.rope(q, headDim=D, offset=w["params"]["posOffset"], **w["rope"]).astype(np.float32)
        kn = oracle.rope(kn, headDim=D, offset=off, **w["rope"]).astype(np.float32)
    oracle.cache_write(x["kc"], kn, off)
    oracle.cache_write(x["vc"], x["v_new"], off)
    return oracle.attention(q, x["kc"], x["vc"], heads=H, headDim=D, kvHeads=Hk, **w["params"])


def oracle_mla_step(x, w):
    import oracle
    off = w["offset"]
    oracle.cache_write(x["state"], x["state_new"], off)
    return oracle.mla_attention(x["q"], x["state"][:off + w.get("rows", 1)], x["k_b"], x["v_b"], heads=w["heads"],
                                kv_rank=w["kv_rank"], qk_nope=w["qk_nope"], qk_rope=w["qk_rope"],
                                v_head_dim=w["v_head_dim"], **w["params"])


class OracleSampler:
    """Bounded samples of a workload computed by the oracle as it stands, on
    all host cores.  decode and latent-attention decode: one whole decode
    step per sample; prefill: 16 query rows x all heads per sample (rows
    drawn at random), counted by their visible pairs."""

    ROWS = 16

    def __init__(self, name, w, x=None):
        import oracle
        self.oracle = oracle
        self.name, self.w = name, w
        self.x = si.workload_inputs(name) if x is None else x
        self.cores = oracle.num_threads()
        self.order = np.random.default_rng(0).permutation(w.get("T", 1))
        self.next_row = 0

    def sample(self):
        """Runs one sample; returns (work in the unit's numerator, seconds)."""
        w, x = self.w, self.x
        t0 = time.perf_counter()
        if w["kind"] == "decode":
            oracle_decode_step(x, w)
            return decode_bytes(w)[1] / 1e9, time.perf_counter() - t0
        if w["kind"] == "mla_decode":
            oracle_mla_step(x, w)
            return mla_work(w)[0] / 1e9, time.perf_counter() - t0
        H = w["heads"]
        D = w["headDim"]
        Dv = w.get("vHeadDim") or D
        params = dict(heads=H, headDim=D, kvHeads=w["kvHeads"], vHeadDim=w.get("vHeadDim"), **w["params"])
        lo_i = self.next_row % w["T"]
        ts = self.order[lo_i:lo_i + self.ROWS]
        self.next_row += len(ts)
        rows = [(int(t), h) for t in ts for h in range(H)]
        self.oracle.attention_rows(x["q"], x["k"], x["v"], x.get("bias"), rows=rows, **params)
        dt = time.perf_counter() - t0
        pairs = int(visible_counts(np.asarray(ts, dtype=np.int64) + w["params"].get("posOffset", 0), w["S"],
                                   w["params"]).sum())
        return pairs * H * (2 * D + 2 * Dv) / 1e12, dt

    def describe(self, n):
        if self.w["kind"] == "decode":
            return f"{n} whole decode steps (cache_write x2 + attention over {self.w['offset'] + 1} keys)"
        if self.w["kind"] == "mla_decode":
            return (f"{n} whole latent decode steps (cache_write + {self.w['heads']} heads over "
                    f"{self.w['offset'] + 1} latent rows)")
        return f"{n} samples of {self.ROWS} random query rows x all {self.w['heads']} heads"


def time_oracle(name, w, budget_s=12.0, min_samples=2, x=None):
    """cpu_baseline: oracle samples for about `budget_s` seconds."""
    smp = OracleSampler(name, w, x)
    work = secs = 0.0
    n = 0
    while n < min_samples or secs < budget_s:
        a, b = smp.sample()
        work += a
        secs += b
        n += 1
    return work / secs, smp.describe(n), smp.cores


# ------------------------------------------------------------- the GPU arm
class Ctx:
    """What every measurement of one run shares: torch, the library, the
    device and stream, the peaks, the clock sampler, rank and world."""

    def __init__(self, torch, vtmu, dev, stream, peaks, peak_kind, sampler, rank, world, args):
        self.torch, self.vtmu, self.dev, self.stream = torch, vtmu, dev, stream
        self.st = stream.cuda_stream
        self.peaks, self.peak_kind, self.sampler = peaks, peak_kind, sampler
        self.rank, self.world, self.args = rank, world, args


def timed_loop(ctx, step, steps, warmup, flush=None):
    """W untimed steps, then K timed steps between a barrier and a device
    synchronisation on both sides.  Returns (ms per step, ms per step of the
    events `step` records around its dominant launch, wall-clock window).
    With `flush`, L2 is overwritten after every step outside the events and
    the step time is the sum of the steps; without, it is the span of the
    whole run, gaps between launches included."""
    torch, dev, stream = ctx.torch, ctx.dev, ctx.stream
    for i in range(warmup):
        step(i)
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.zero_()
    torch.cuda.synchronize(dev)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(ctx.world)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    for i in range(steps):
        if flush is not None or i == 0:
            sev[i][0].record(stream)
        step(i, kev[i])
        if flush is not None or i == steps - 1:
            sev[i][1].record(stream)
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.zero_()
    torch.cuda.synchronize(dev)
    barrier(ctx.world)
    t1 = time.time()
    if flush is None:
        step_ms = sev[0][0].elapsed_time(sev[-1][1]) / steps
    else:
        step_ms = sum(a.elapsed_time(b) for a, b in sev) / steps
    kern_ms = sum(a.elapsed_time(b) for a, b in kev) / steps
    return max_over_ranks(step_ms, ctx.world), max_over_ranks(kern_ms, ctx.world), (t0, t1)


def measure_prefill(ctx, name, steps, warmup, kernel_arg="auto", cpu_budget=0.0, e2e_steps=None):
    """One prefill workload: W + K steps of vtmu_attention with L2 flushed
    between steps, the same call end to end from pinned host buffers, and a
    bounded oracle sample on the host cores (rank 0, cpu_budget > 0).
    Returns the measurements; finish_prefill() adds clocks and rooflines."""
    torch, vtmu, dev, stream, st = ctx.torch, ctx.vtmu, ctx.dev, ctx.stream, ctx.st
    w = si.WORKLOADS[name]
    x = si.workload_inputs(name)
    H, Hk, D = w["heads"], w["kvHeads"], w["headDim"]
    Dv = w.get("vHeadDim") or D
    T, S = w["T"], w["S"]
    with torch.cuda.stream(stream):
        q = torch.from_numpy(x["q"]).to(dev)
        k = torch.from_numpy(x["k"]).to(dev)
        v = torch.from_numpy(x["v"]).to(dev)
        b = torch.from_numpy(x["bias"]).to(dev) if "bias" in x else None
        out = torch.empty((T, H * Dv), dtype=torch.float32, device=dev)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    bias_kind = vtmu.VTMU_BIAS_NONE if b is None else (vtmu.VTMU_BIAS_TS if b.dim() == 2 else vtmu.VTMU_BIAS_HTS)
    tc_ok = ((D == Dv and D in (32, 64, 96, 128, 256)) or (D, Dv) == (192, 128)) and T >= 64
    use_tc = tc_ok if kernel_arg == "auto" else kernel_arg == "tc"
    kernel = vtmu.VTMU_KERNEL_PREFILL_TF32X3 if use_tc else vtmu.VTMU_KERNEL_PREFILL_FFMA
    p = vtmu.make_params(T, S, heads=H, headDim=D, kvHeads=Hk, vHeadDim=w.get("vHeadDim"),
                         bias_kind=bias_kind, kernel=kernel, **w["params"])
    ws_bytes = vtmu.vtmu_attention_workspace_size(p)
    ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device=dev)

    def step(i, ev=None):
        if ev is not None:
            ev[0].record(stream)
        vtmu.vtmu_attention(q, k, v, b, out, p, ws, ws_bytes, st)
        if ev is not None:
            ev[1].record(stream)

    step_ms, kern_ms, window = timed_loop(ctx, step, steps, warmup, flush)

    # End to end through the public API: inputs copied in from pinned host
    # memory, the call, the output copied back, a host sync.
    qh = torch.from_numpy(x["q"]).pin_memory()
    kh = torch.from_numpy(x["k"]).pin_memory()
    vh = torch.from_numpy(x["v"]).pin_memory()
    bh = torch.from_numpy(x["bias"]).pin_memory() if "bias" in x else None
    outh = torch.empty(tuple(out.shape), dtype=torch.float32).pin_memory()

    def e2e_step():
        with torch.cuda.stream(stream):
            q.copy_(qh, non_blocking=True)
            k.copy_(kh, non_blocking=True)
            v.copy_(vh, non_blocking=True)
            if bh is not None:
                b.copy_(bh, non_blocking=True)
        vtmu.vtmu_attention(q, k, v, b, out, p, ws, ws_bytes, st)
        with torch.cuda.stream(stream):
            outh.copy_(out, non_blocking=True)
        stream.synchronize()

    flops = prefill_flops(w)
    e2e_step()
    n_e2e = e2e_steps or max(3, min(steps, 200))
    barrier(ctx.world)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, ctx.world)
    h2d = (qh.numel() + kh.numel() + vh.numel() + (bh.numel() if bh is not None else 0)) * 4
    e2e = {"value": round(flops / 1e12 * ctx.world / e2e_s, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": outh.numel() * 4, "steps": n_e2e,
           "transfer": "cudaMemcpyAsync from pinned buffers in, attention, copy out, host sync"}
    del q, k, v, b, out, flush, ws, qh, kh, vh, bh, outh
    torch.cuda.empty_cache()

    cpu = None
    if ctx.rank == 0 and cpu_budget > 0:
        val, sample, cores = time_oracle(name, w, budget_s=cpu_budget, min_samples=1, x=x)
        cpu = {"value": round(val, 5), "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}
    return {"workload": name, "kernel": "prefill_tc" if use_tc else "prefill_ffma", "flops": flops,
            "steps": steps, "warmup": warmup, "ms_per_step": step_ms, "kernel_ms": kern_ms,
            "gpu_launches": (3 if use_tc else 1) * steps, "e2e": e2e, "cpu_baseline": cpu, "_window": window}


def prefill_roofline(ctx, res, clocks):
    """The dominant kernel's roofline: algorithmic FLOPs / kernel time against
    the 3xTF32 tensor ceilings (both ways) or the FP32 FMA peak."""
    peaks = ctx.peaks
    name, kern_ms = res["workload"], res["kernel_ms"]
    achieved = res["flops"] / 1e12 / (kern_ms / 1e3)
    sm = clocks.get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    prof = profile_info(f"{res['kernel']}__{name}")
    if res["kernel"] == "prefill_tc":
        bf16_scaled, clk = tensor_ceilings(peaks, sm)
        return {"bound": "tensor", "kernel": "prefill_tc", "achieved": round(achieved, 3),
                "peak": round(bf16_scaled, 1), "unit": "TFLOP/s", "frac": round(achieved / bf16_scaled, 4),
                "peak_source": (f"{ctx.peak_kind} bf16 burst x 1.1/2.25 (tf32/bf16 nominal) / 3 (3xTF32 products)"),
                "peak_clock_scaled": round(clk, 1), "frac_clock_scaled": round(achieved / clk, 4),
                "peak_clock_scaled_source": (f"kind::tf32 {TF32_FLOP_PER_CYCLE_SM} FLOP/cycle/SM (measured) x "
                                             f"{SMS} SMs x {sm:.0f} MHz (sampled) / 3"),
                "tensor_pipe_active_pct": prof.get("tensor_pipe_active_pct"),
                "traffic": prof.get("traffic"), "kernel_ms": round(kern_ms, 5)}
    peak = SMS * FP32_LANES_PER_SM * 2 * sm * 1e6 / 1e12
    return {"bound": "alu", "kernel": "prefill_ffma", "achieved": round(achieved, 3), "peak": round(peak, 1),
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "peak_source": f"derived: {SMS} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {sm:.0f} MHz (sampled)",
            "traffic": prof.get("traffic"), "kernel_ms": round(kern_ms, 5)}


def finish_prefill(ctx, res):
    """A prefill entry of the JSON line, once the clock samples are in."""
    clocks = ctx.sampler.summary(*res.pop("_window"))
    flops = res["flops"]
    return {"workload": res["workload"], "config": workload_config(res["workload"], ctx.world),
            "value": round(flops * ctx.world / 1e12 / (res["ms_per_step"] / 1e3), 3), "unit": "TFLOP/s",
            "ms_per_step": round(res["ms_per_step"], 5), "kernel_ms": round(res["kernel_ms"], 5),
            "algorithmic_flop": flops, "steps": res["steps"], "warmup": res["warmup"],
            "roofline": prefill_roofline(ctx, res, clocks), "e2e": res["e2e"], "cpu_baseline": res["cpu_baseline"],
            "gpu_launches": res["gpu_launches"], "clocks": clocks}


def decode_launches(w, args):
    """(path, kernels launched per step) of a decode step: the CUDA-core
    decode kernel or the tensor-core decode of several query rows (each one
    launch with the cache write and the split merge inside), or, forced,
    cache writes plus the FFMA prefill (3)."""
    if args.kernel == "ffma":
        return ("prefill", 3)
    R, G = w.get("rows", 1), w["heads"] // w["kvHeads"]
    p = w["params"]
    tc = (R >= 2 and R * G <= 16 and w["headDim"] == 128 and not p.get("softcap") and not p.get("alibi")
          and not w.get("rope"))
    return ("tc", 1) if tc else ("ffma", 1)


def measure_decode(ctx, name):
    """The decode step of a decode workload: W + K fused steps alternating two
    cache sets (each step's K/V come from HBM), the same step as separate
    launches, and end to end from host buffers."""
    torch, vtmu, dev, stream, st, args = ctx.torch, ctx.vtmu, ctx.dev, ctx.stream, ctx.st, ctx.args
    w = si.WORKLOADS[name]
    x = si.workload_inputs(name)
    H, Hk, D, off = w["heads"], w["kvHeads"], w["headDim"], w["offset"]
    R = w.get("rows", 1)  # query rows = new cache rows of the step
    kv_bytes, step_bytes = decode_bytes(w)
    sessions = []
    with torch.cuda.stream(stream):
        for _ in range(2):
            sessions.append(dict(Kc=torch.from_numpy(x["kc"]).to(dev), Vc=torch.from_numpy(x["vc"]).to(dev)))
        q = torch.from_numpy(x["q"]).to(dev)
        kn = torch.from_numpy(x["k_new"]).to(dev)
        vn = torch.from_numpy(x["v_new"]).to(dev)
        out = torch.empty((R, H * D), dtype=torch.float32, device=dev)
    # --kernel ffma: the same step through the FFMA prefill (cache_writes
    # and attention as three launches), for comparison.
    forced = vtmu.VTMU_KERNEL_PREFILL_FFMA if args.kernel == "ffma" else vtmu.VTMU_KERNEL_AUTO
    p = vtmu.make_params(R, off + R, heads=H, headDim=D, kvHeads=Hk, kernel=forced, **w["params"])
    ws_bytes = vtmu.vtmu_attention_workspace_size(p)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    width = Hk * D
    rope = vtmu.make_rope_params(headDim=D, **w["rope"]) if w.get("rope") else None
    if rope is not None:
        with torch.cuda.stream(stream):
            q_rot, kn_rot = torch.empty_like(q), torch.empty_like(kn)

    def step(i, ev=None):
        # One fused launch: both cache_writes and the attention (and the
        # rotary embedding of q and the new key row).
        s = sessions[i % 2]
        if ev is not None:
            ev[0].record(stream)
        if rope is None:
            vtmu.vtmu_decode_step(s["Kc"], s["Vc"], off + R, kn, vn, R, off, q, None, out, p, ws, ws_bytes, st)
        else:
            vtmu.vtmu_decode_step_rope(s["Kc"], s["Vc"], off + R, kn, vn, R, off, q, None, out, p, rope, ws,
                                       ws_bytes, st)
        if ev is not None:
            ev[1].record(stream)

    def unfused_step(i):
        s = sessions[i % 2]
        qq, kk = q, kn
        if rope is not None:
            vtmu.vtmu_rope(q, q_rot, 1, H, w["params"]["posOffset"], rope, st)
            vtmu.vtmu_rope(kn, kn_rot, 1, Hk, off, rope, st)
            qq, kk = q_rot, kn_rot
        vtmu.vtmu_cache_write(s["Kc"], off + R, width, kk, R, off, st)
        vtmu.vtmu_cache_write(s["Vc"], off + R, width, vn, R, off, st)
        vtmu.vtmu_attention(qq, s["Kc"], s["Vc"], None, out, p, ws, ws_bytes, st)

    step_ms, kern_ms, window = timed_loop(ctx, step, args.steps, args.warmup)

    # The same decode step as separate launches, for comparison.
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(3):
        unfused_step(i)
    e0.record(stream)
    for i in range(args.steps):
        unfused_step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    unfused_ms = e0.elapsed_time(e1) / args.steps

    # ---- end to end through the public API with host buffers ----------------
    qh = torch.from_numpy(x["q"]).pin_memory()
    knh = torch.from_numpy(x["k_new"]).pin_memory()
    vnh = torch.from_numpy(x["v_new"]).pin_memory()
    outh = torch.empty((R, H * D), dtype=torch.float32).pin_memory()
    if rope is not None:
        # The rotary decode step has no host-buffer entry point: pinned copies
        # in, the fused step, the output back, a host sync.
        def e2e_step(i):
            with torch.cuda.stream(stream):
                q.copy_(qh, non_blocking=True)
                kn.copy_(knh, non_blocking=True)
                vn.copy_(vnh, non_blocking=True)
            step(i)
            with torch.cuda.stream(stream):
                outh.copy_(out, non_blocking=True)
            stream.synchronize()
    else:
        # The host-buffer decode step of the C ABI on pinned buffers: the
        # fused step's kernel reads q and the new rows from them and writes
        # the output row back over the host link (no staging copies), then
        # the call waits for it.
        hws_bytes = vtmu.vtmu_decode_step_host_workspace_size(p, R)
        hws = torch.zeros(hws_bytes, dtype=torch.uint8, device=dev)

        def e2e_step(i):
            s = sessions[i % 2]
            vtmu.vtmu_decode_step_host(s["Kc"], s["Vc"], off + R, knh, vnh, R, off, qh, None, outh, p, hws,
                                       hws_bytes, st)

    h2d = (qh.numel() + knh.numel() + vnh.numel()) * 4
    d2h = outh.numel() * 4
    e2e_step(0)
    n_e2e = max(3, min(args.steps, 200))
    barrier(ctx.world)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        e2e_step(i)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, ctx.world)
    e2e = {"value": round(step_bytes / 1e9 * ctx.world / e2e_s, 3), "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": n_e2e,
           "transfer": ("cudaMemcpyAsync from pinned buffers around the fused step, host sync" if rope is not None else
                        "vtmu_decode_step_host on pinned buffers, staged through the workspace (the prefill "
                        "kernels take device buffers), then the call waits" if args.kernel == "ffma" else
                        "vtmu_decode_step_host on pinned buffers: the kernel reads q and the new rows and writes "
                        "the output row over the host link, then the call waits")}
    del sessions, q, kn, vn, out, ws
    torch.cuda.empty_cache()
    kernel_tag = ("prefill_ffma" if args.kernel == "ffma" else
                  "decode_tc" if decode_launches(w, args)[0] == "tc" else "decode")
    return {"workload": name, "x": x, "w": w, "step_bytes": step_bytes, "step_ms": step_ms, "kernel_ms": kern_ms,
            "unfused_ms": unfused_ms, "e2e": e2e, "kernel_tag": kernel_tag,
            "launches_per_step": decode_launches(w, args)[1], "_window": window}


def measure_mla(ctx, name):
    """A latent-attention decode step (vtmu_mla_decode_step: the new latent
    row written, queries absorbed, split-KV attention over the latent cache,
    merge and output projection), W + K steps over four cache copies that
    alternate (302 MB > L2, so every step reads its cache from HBM), then the
    same step end to end from pinned host buffers."""
    torch, vtmu, dev, stream, st, args = ctx.torch, ctx.vtmu, ctx.dev, ctx.stream, ctx.st, ctx.args
    w = si.WORKLOADS[name]
    x = si.workload_inputs(name)
    H, N, Dv, off = w["heads"], w["qk_nope"], w["v_head_dim"], w["offset"]
    T = w.get("rows", 1)
    nbytes, flops = mla_work(w)
    with torch.cuda.stream(stream):
        states = [torch.from_numpy(x["state"]).to(dev) for _ in range(4)]
        q = torch.from_numpy(x["q"]).to(dev)
        k_b = torch.from_numpy(x["k_b"]).to(dev)
        v_b = torch.from_numpy(x["v_b"]).to(dev)
        sn = torch.from_numpy(x["state_new"]).to(dev)
        out = torch.empty((T, H * Dv), dtype=torch.float32, device=dev)
    p = vtmu.make_mla_params(T, off + T, heads=H, qk_nope=N, v_head_dim=Dv, kv_rank=w["kv_rank"],
                             qk_rope=w["qk_rope"], **w["params"])
    ws_bytes = vtmu.vtmu_mla_workspace_size(p)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    max_rows = w["max_rows"]

    def step(i, ev=None):
        if ev is not None:
            ev[0].record(stream)
        vtmu.vtmu_mla_decode_step(states[i % 4], max_rows, sn, T, off, q, k_b, v_b, out, p, ws, ws_bytes, st)
        if ev is not None:
            ev[1].record(stream)

    step_ms, kern_ms, window = timed_loop(ctx, step, args.steps, args.warmup)
    qh = torch.from_numpy(x["q"]).pin_memory()
    snh = torch.from_numpy(x["state_new"]).pin_memory()
    outh = torch.empty((T, H * Dv), dtype=torch.float32).pin_memory()

    # The host-buffer latent decode step of the C ABI on pinned buffers: the
    # absorb launch reads q and the new row from them, the projection writes
    # the output row back (no staging copies), and the call waits for it.
    hws_bytes = vtmu.vtmu_mla_decode_step_host_workspace_size(p, T)
    hws = torch.zeros(hws_bytes, dtype=torch.uint8, device=dev)

    def e2e_step(i):
        vtmu.vtmu_mla_decode_step_host(states[i % 4], max_rows, snh, T, off, qh, k_b, v_b, outh, p, hws, hws_bytes,
                                       st)

    e2e_step(0)
    n_e2e = max(3, min(args.steps, 200))
    barrier(ctx.world)
    t0 = time.perf_counter()
    for i in range(n_e2e):
        e2e_step(i)
    e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, ctx.world)
    e2e = {"value": round(nbytes / 1e9 * ctx.world / e2e_s, 3), "unit": "GB/s",
           "h2d_bytes_per_step": (qh.numel() + snh.numel()) * 4, "d2h_bytes_per_step": outh.numel() * 4,
           "steps": n_e2e,
           "transfer": "vtmu_mla_decode_step_host on pinned buffers: the absorb launch reads q and the new row, "
                       "the projection writes the output row over the host link, then the call waits"}
    del hws
    del states, q, k_b, v_b, sn, out, ws
    torch.cuda.empty_cache()
    return {"workload": name, "x": x, "w": w, "step_bytes": nbytes, "flops": flops, "step_ms": step_ms,
            "kernel_ms": kern_ms, "e2e": e2e, "_window": window}


def mla_roofline(ctx, d, clocks):
    """Both rooflines of the latent-attention step (its four launches timed
    together): algorithmic bytes against the HBM copy peak and algorithmic
    FLOPs against the FP32 FMA peak; `bound` is the one whose ideal time is
    longer."""
    peaks = ctx.peaks
    t = d["kernel_ms"] / 1e3
    sm = clocks.get("sm_mhz") or float(peaks.get("sm_max_mhz", 2070.0))
    hbm = float(peaks["hbm_gbs"])
    fp32 = SMS * FP32_LANES_PER_SM * 2 * sm * 1e6 / 1e12
    gbs = d["step_bytes"] / t / 1e9
    tfs = d["flops"] / t / 1e12
    t_hbm = d["step_bytes"] / (hbm * 1e9)
    t_alu = d["flops"] / (fp32 * 1e12)
    hbm_line = {"achieved": round(gbs, 3), "peak": round(hbm, 1), "unit": "GB/s", "frac": round(gbs / hbm, 4),
                "peak_source": ctx.peak_kind}
    alu_line = {"achieved": round(tfs, 3), "peak": round(fp32, 1), "unit": "TFLOP/s", "frac": round(tfs / fp32, 4),
                "peak_source": f"derived: {SMS} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {sm:.0f} MHz (sampled)"}
    main, other = (alu_line, hbm_line) if t_alu > t_hbm else (hbm_line, alu_line)
    return {"bound": "alu" if t_alu > t_hbm else "hbm", "kernel": "mla", **main,
            "traffic": profile_traffic("mla__" + d["workload"]), "kernel_ms": round(d["kernel_ms"], 5),
            "other_bound": other, "algorithmic_bytes": d["step_bytes"], "algorithmic_flop": d["flops"]}


def run_vtmu(args, rank, world, local):
    import torch
    import f32_gqa_attention_gb300 as vtmu
    vtmu.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_kind = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
        time.sleep(0.6)
    ctx = Ctx(torch, vtmu, dev, stream, peaks, peak_kind, sampler, rank, world, args)
    name = args.workload
    w = si.WORKLOADS[name]

    if w["kind"] == "mla_decode":
        d = measure_mla(ctx, name)
        sampler.stop()
        clocks = sampler.summary(*d["_window"])
        cpu = None
        if rank == 0 and not args.no_cpu_baseline:
            val, sample, cores = time_oracle(name, w, budget_s=args.cpu_budget, x=d["x"])
            cpu = {"value": round(val, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
        line = {
            "metric": METRIC, "value": round(d["step_bytes"] / 1e9 * world / (d["step_ms"] / 1e3), 3),
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(d["step_ms"], 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": DATA, "config": workload_config(name, world),
            "impl": "vtmu", "roofline": mla_roofline(ctx, d, clocks), "cpu_baseline": cpu, "e2e": d["e2e"],
            "gpu_launches": 4 * args.steps, "clocks": clocks,
        }
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if w["kind"] == "decode":
        d = measure_decode(ctx, name)
        block = []
        if not args.no_prefill:
            for pname in PREFILL_SET:
                block.append(measure_prefill(ctx, pname, args.steps, args.warmup,
                                             cpu_budget=0.0 if args.no_cpu_baseline else args.prefill_cpu_budget,
                                             e2e_steps=3))
        mla = None if args.no_mla else measure_mla(ctx, "mla_decode")
        # The few-query-row step (the scope table's second next row) beside
        # the one-row step it extends.
        rows = measure_decode(ctx, "gqa_spec_decode") if name == "gqa_decode" and not args.no_rows else None
        sampler.stop()
        clocks = sampler.summary(*d["_window"])
        achieved = d["step_bytes"] / (d["kernel_ms"] / 1e3) / 1e9
        peak = float(peaks["hbm_gbs"])
        roofline = {"bound": "hbm", "kernel": d["kernel_tag"], "achieved": round(achieved, 3), "peak": round(peak, 1),
                    "peak_source": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "traffic": profile_traffic(d["kernel_tag"] + "__" + name), "kernel_ms": round(d["kernel_ms"], 5)}
        cpu = None
        if rank == 0 and not args.no_cpu_baseline:
            val, sample, cores = time_oracle(name, w, budget_s=args.cpu_budget, x=d["x"])
            cpu = {"value": round(val, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
        line = {
            "metric": METRIC, "value": round(d["step_bytes"] / 1e9 * world / (d["step_ms"] / 1e3), 3),
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(d["step_ms"], 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": DATA, "config": workload_config(name, world),
            "impl": "vtmu", "roofline": roofline, "cpu_baseline": cpu, "e2e": d["e2e"],
            "gpu_launches": d["launches_per_step"] * args.steps, "clocks": clocks,
            "unfused_ms_per_step": round(d["unfused_ms"], 5),
        }
        if block:
            line["prefill"] = [finish_prefill(ctx, r) for r in block]
        if rows is not None:
            rclk = sampler.summary(*rows["_window"])
            rw = si.WORKLOADS["gqa_spec_decode"]
            r_ach = rows["step_bytes"] / (rows["kernel_ms"] / 1e3) / 1e9
            rcpu = None
            if rank == 0 and not args.no_cpu_baseline:
                val, sample, cores = time_oracle("gqa_spec_decode", rw, budget_s=args.prefill_cpu_budget, x=rows["x"])
                rcpu = {"value": round(val, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
            line["decode_rows"] = {
                "workload": "gqa_spec_decode", "config": workload_config("gqa_spec_decode", world),
                "value": round(rows["step_bytes"] / 1e9 * world / (rows["step_ms"] / 1e3), 3), "unit": "GB/s",
                "ms_per_step": round(rows["step_ms"], 5), "kernel_ms": round(rows["kernel_ms"], 5),
                "steps": args.steps, "warmup": args.warmup,
                "roofline": {"bound": "hbm", "kernel": rows["kernel_tag"], "achieved": round(r_ach, 3),
                             "peak": round(peak, 1), "peak_source": peak_kind, "unit": "GB/s",
                             "frac": round(r_ach / peak, 4),
                             "traffic": profile_traffic(rows["kernel_tag"] + "__gqa_spec_decode"),
                             "kernel_ms": round(rows["kernel_ms"], 5)},
                "e2e": rows["e2e"], "cpu_baseline": rcpu,
                "gpu_launches": rows["launches_per_step"] * args.steps, "clocks": rclk}
        if mla is not None:
            mclk = sampler.summary(*mla["_window"])
            mcpu = None
            if rank == 0 and not args.no_cpu_baseline:
                val, sample, cores = time_oracle("mla_decode", mla["w"], budget_s=args.prefill_cpu_budget,
                                                 min_samples=1, x=mla["x"])
                mcpu = {"value": round(val, 5), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
            line["mla"] = {"workload": "mla_decode", "config": workload_config("mla_decode", world),
                           "value": round(mla["step_bytes"] / 1e9 * world / (mla["step_ms"] / 1e3), 3),
                           "unit": "GB/s", "ms_per_step": round(mla["step_ms"], 5),
                           "kernel_ms": round(mla["kernel_ms"], 5), "steps": args.steps, "warmup": args.warmup,
                           "roofline": mla_roofline(ctx, mla, mclk), "e2e": mla["e2e"], "cpu_baseline": mcpu,
                           "gpu_launches": 4 * args.steps, "clocks": mclk}
    else:
        r = measure_prefill(ctx, name, args.steps, args.warmup, kernel_arg=args.kernel,
                            cpu_budget=0.0 if args.no_cpu_baseline else args.cpu_budget)
        sampler.stop()
        e = finish_prefill(ctx, r)
        line = {
            "metric": METRIC, "value": e["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": e["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": DATA, "config": workload_config(name, world),
            "impl": "vtmu", "roofline": e["roofline"], "cpu_baseline": e["cpu_baseline"], "e2e": e["e2e"],
            "gpu_launches": e["gpu_launches"], "clocks": e["clocks"], "kernel_ms": e["kernel_ms"],
        }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The oracle on the host cores: W untimed samples, then K timed ones."""
    if rank != 0:
        return
    name = args.workload
    w = si.WORKLOADS[name]
    unit = "GB/s" if w["kind"] in ("decode", "mla_decode") else "TFLOP/s"
    smp = OracleSampler(name, w)
    for _ in range(args.warmup):
        smp.sample()
    work = secs = 0.0
    for _ in range(args.steps):
        a, b = smp.sample()
        work += a
        secs += b
    value = work / secs
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
        "config": workload_config(name, world), "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": unit, "kind": "oracle", "cores": smp.cores,
                         "sample": smp.describe(args.steps)},
        "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["vtmu", "reference"], default="vtmu")
    ap.add_argument("--workload", choices=sorted(si.WORKLOADS), default="gqa_decode")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode workloads: leave out the four prefill workloads that follow the decode line")
    ap.add_argument("--no-rows", action="store_true",
                    help="default decode line: leave out the 4-row speculative step (decode_rows)")
    ap.add_argument("--no-mla", action="store_true",
                    help="decode workloads: leave out the latent-attention decode step that follows the decode line")
    ap.add_argument("--prefill-cpu-budget", type=float, default=3.0,
                    help="seconds of oracle timing per prefill workload after a decode line")
    ap.add_argument("--kernel", choices=["auto", "tc", "ffma"], default="auto",
                    help="prefill kernel: tcgen05 3xTF32 or FFMA (auto: tcgen05 where it covers the shape)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if world != args.gpus and "RANK" in os.environ:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    if world > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_vtmu(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
