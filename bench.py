"""Benchmark: exact tiled attention forward + backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole attention path over one batch of the workload:
fa_fwd (one kernel) then fa_bwd's three stages (preprocess, main, postprocess),
inputs resident in HBM.  The headline workload is the causal long-context one
(B1 H32 N65536 d128, 4.3 GB of inputs, far larger than L2); the other workloads
run as extra legs of the same line, each with its own stage times, roofline and
clock record.  Each timed step calls the API (--graphs instead captures each
stage's call once as a CUDA graph after the warm-up and replays the graphs).
Timed with CUDA events on the launching stream around each step; a second pass
puts an event between the stages for the per-kernel times.  L2 is flushed
between timed steps (512 MiB written, then 256 MiB read so that the flush's own
dirty lines are written back before the next step).  Max over ranks; rank 0
prints one JSON line.

FLOP convention: forward 4*B*H*N^2*d (halved when causal), backward 2.5x forward;
`value` is forward+backward TFLOP/s.  Beside it: "algorithmic" FLOPs count the
128x128 tile pairs the kernels visit (4*128*128*d per pair forward, 10*128*128*d
backward), "useful" FLOPs the visible query/key pairs only (4*d per pair forward,
14*d forward+backward).  The roofline object reports the dominant kernel against
the measured dense bf16 peak.

nvidia-smi is polled every 200 ms for the whole run; each leg reports the median
SM clock and the throttle reasons seen during its own timed region.

--impl reference times the fp64 CPU oracle on the host cores instead, as the
reference arm: each step is the oracle's row pass over a seeded sample of query
rows of the workload's first head, and the whole-workload time is extrapolated
from it by visible pair count.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from io_aware_exact_attention_gb300 import inputs  # noqa: E402

METRIC = "attention TFLOP/s fwd & fwd+bwd bf16 on 1 GB300; % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
FLUSH_BYTES = 512 << 20       # written between timed steps (L2 is 129 MB)
FLUSH_READ_BYTES = 256 << 20  # then read, so L2 holds clean lines only when a step starts


class L2Flush:
    """Evicts the workload from L2 between timed steps: writes FLUSH_BYTES, then reads
    FLUSH_READ_BYTES of another buffer.  The read pass makes L2 write back the dirty
    lines of the write pass, so the next step starts on a cold, clean L2 instead of
    paying for the flush's write-back in its first kernel."""

    def __init__(self, torch):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(FLUSH_READ_BYTES // 4, dtype=torch.float32, device="cuda")
        self.acc = torch.empty((), dtype=torch.float32, device="cuda")
        self.torch = torch

    def __call__(self):
        self.w.zero_()
        self.torch.sum(self.r, dim=0, out=self.acc)
TILE = 128
HEADLINE_WORKLOAD = "long_causal_64k"
EXTRA_WORKLOADS = ("long_causal_16k", "gpt2_causal", "block_sparse_8k", "bert_large_padded")
FP8_WORKLOAD = "long_causal_16k"
EXTRA_MIN_SECONDS = 1.0   # an extra leg's timed region lasts at least this long (clock samples)


# ------------------------------------------------------------------ host logic

def formula_fwd_flops(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def visited_tile_pairs(N, causal, kv_len, block_mask, B, H):
    """Number of (query tile, key tile) pairs the kernels visit, summed over heads."""
    T = (N + TILE - 1) // TILE
    qt = np.arange(T)[:, None]
    kt = np.arange(T)[None, :]
    total = 0
    for b in range(B):
        vis = np.ones((T, T), bool)
        kl = N if kv_len is None else int(min(max(kv_len[b], 0), N))
        vis &= kt * TILE < kl
        if causal:
            vis &= kt <= qt
        if block_mask is not None:
            vis &= np.asarray(block_mask).astype(bool)
        total += int(vis.sum()) * H
    return total


def algorithmic_flops(pairs, d):
    return {"fwd": pairs * 4.0 * TILE * TILE * d, "bwd": pairs * 10.0 * TILE * TILE * d}


def row_visible_counts(N, rows, causal, kv_len, block_mask, tile=TILE):
    """Number of keys each query row in `rows` sees (one sequence: kv_len an int or None)."""
    rows = np.asarray(rows, np.int64)
    lim = np.full(rows.shape, N if kv_len is None else min(max(int(kv_len), 0), N), np.int64)
    if causal:
        lim = np.minimum(lim, rows + 1)
    if block_mask is None:
        return lim
    bm = np.asarray(block_mask).astype(bool)
    counts = np.zeros(rows.shape, np.int64)
    for tj in range((N + tile - 1) // tile):
        width = np.clip(np.minimum(lim, min(N, (tj + 1) * tile)) - tj * tile, 0, None)
        counts += np.where(bm[rows // tile, tj], width, 0)
    return counts


def useful_score_pairs(N, causal, kv_len, block_mask, B, H):
    """Visible (query, key) pairs summed over heads: the scores the method must compute."""
    rows = np.arange(N)
    total = 0
    for b in range(B):
        kl = None if kv_len is None else int(kv_len[b])
        total += int(row_visible_counts(N, rows, causal, kl, block_mask).sum()) * H
    return total


def splitkv_work(B, H, Nq, Nk, d):
    """Forward FLOPs (4 * Nq * Nk * d per head, no mask) and algorithmic bytes of a
    split-KV call: K and V read once, Q read, O (bf16) and LSE (fp32) written."""
    flops = 4.0 * B * H * Nq * Nk * d
    nbytes = 2.0 * (2 * B * H * Nk * d + 2 * B * H * Nq * d) + 4.0 * B * H * Nq
    return flops, nbytes


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        p = json.load(open(path))
        return {"bf16_tflops": float(p["bf16_tflops"]), "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def _code_only(text):
    """Source text without comments, trailing blanks and blank lines, so that editing a
    comment does not count as changing a kernel."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_digest(kernel):
    import hashlib
    src = {"bwd_main": "fa_bwd_bf16.cu", "fwd": "fa_fwd.cu", "fwd_fp8": "fa_fwd.cu", "fwd_splitkv": "fa_fwd.cu"}.get(kernel)
    if src is None:
        return None
    h = hashlib.sha256()
    for name in (src, "sm103_ptx.cuh", "fa_tiles.cuh"):
        with open(os.path.join(ROOT, "io_aware_exact_attention_gb300", "csrc", name)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source; None otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    pat = re.compile(r"^\|\s*" + re.escape(kernel) + r"\s*\|\s*" + re.escape(workload) +
                     r"\s*\|\s*([0-9.eE+]+)\s*\|\s*([0-9a-f]+)\s*\|")
    digest = kernel_source_digest(kernel)
    for line in open(path):
        m = pat.match(line)
        if m and m.group(2) == digest:
            return float(m.group(1))
    return None


def reduce_max_over_ranks(x, dist=None):
    """Max of a float over ranks (identity without a process group)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_line(per_rank_flops, world, max_ms_step, steps):
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    total_flops = per_rank_flops * world
    return total_flops / (max_ms_step * 1e-3) / 1e12


class ClockSampler:
    """Polls nvidia-smi (SM clock, max clock, power, throttle reasons) every `period`
    seconds on a background thread for the whole run; `window(t0, t1)` summarises the
    samples taken between two time.monotonic() stamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period=0.2):
        import threading
        self.gpu_index = gpu_index
        self.period = period
        self.samples = []  # (monotonic time of the query's midpoint, csv line)
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, daemon=True)
        self.available = True

    def _run(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-i", str(self.gpu_index)]
        while not self._stop.is_set():
            t0 = time.monotonic()
            try:
                out = subprocess.run(cmd, capture_output=True, text=True, timeout=5).stdout
            except (OSError, subprocess.SubprocessError):
                self.available = False
                return
            t1 = time.monotonic()
            for ln in out.splitlines():
                if ln.strip():
                    self.samples.append((0.5 * (t0 + t1), ln))
            self._stop.wait(max(0.0, self.period - (t1 - t0)))

    def start(self):
        self._thread.start()
        return self

    def stop(self):
        self._stop.set()
        self._thread.join(timeout=10)

    def window(self, t0, t1):
        return parse_clock_lines([ln for t, ln in list(self.samples) if t0 <= t <= t1])


def parse_clock_lines(lines):
    sm, mx, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for ln in lines:
        f = [x.strip() for x in ln.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            mx = float(f[2])
        except ValueError:
            continue
        for name, val in zip(names, f[5:9]):
            if val.lower().startswith("active"):
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
            "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm

def device_inputs(inp, torch):
    def dev(name):
        a = inp.device_array(name)
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    t = {n: dev(n) for n in ("q", "k", "v", "dout")}
    t["block_mask"] = torch.from_numpy(inp.block_mask).cuda() if inp.block_mask is not None else None
    t["kv_len"] = torch.from_numpy(inp.kv_len).cuda() if inp.kv_len is not None else None
    return t


def time_workload(name, steps, warmup, torch, fa, flush, dist=None, override=None, graphs=False, min_seconds=0.0):
    """Run timed fwd+bwd steps on one workload; per-stage CUDA-event times.

    Exactly `steps` timed steps, or more if `min_seconds` asks for a longer timed
    region (the extra legs, so that the clock sampler sees them).  With `graphs`,
    each stage's API call is captured once as a CUDA graph after the warm-up and the
    timed steps replay the graphs (same kernels, same arguments)."""
    spec = inputs.WORKLOADS[name]
    inp = inputs.workload_inputs(name, **(override or {}))
    B, H, N, d = inp.q.shape
    t = device_inputs(inp, torch)
    q, k, v, do, bm, kl = t["q"], t["k"], t["v"], t["dout"], t["block_mask"], t["kv_len"]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = fa.new_workspace(q)
    stream = torch.cuda.current_stream()
    scale, causal = inp.scale, spec["causal"]

    stages = [
        lambda s: fa.fa_fwd(q, k, v, o, lse, scale, causal, bm, kl, s),
        lambda s: fa.fa_bwd_preprocess(o, do, ws, s),
        lambda s: fa.fa_bwd_main(q, k, v, lse, do, dk, dv, ws, scale, causal, bm, kl, s),
        lambda s: fa.fa_bwd_postprocess(dq, ws, s),
    ]
    launch = [lambda fn=fn: fn(stream) for fn in stages]

    def step(ev=None):
        for j, run in enumerate(launch):
            if ev is not None:
                ev[j].record(stream)
            run()
        if ev is not None:
            ev[len(launch)].record(stream)

    torch.cuda.synchronize()
    tw = time.perf_counter()
    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    warm_step_s = (time.perf_counter() - tw) / max(1, warmup)
    launch_mode = "api calls"
    if graphs:
        try:
            captured = []
            for fn in stages:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    fn(torch.cuda.current_stream())
                captured.append(g)
            torch.cuda.synchronize()
            launch = [g.replay for g in captured]
            launch_mode = "CUDA graph per stage, replayed"
        except Exception as exc:  # keep measuring through the API if capture is refused
            torch.cuda.synchronize()
            launch_mode = f"api calls (graph capture failed: {type(exc).__name__})"
        for _ in range(2):
            flush()
            step()
    if min_seconds > 0:
        steps = max(steps, min(5000, math.ceil(min_seconds / max(warm_step_s, 1e-6))))
    # Timed steps: one event pair around each step.  The four launches of a step run
    # back to back, so each kernel's launch overlaps the tail of the one before it.
    step_events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    if dist is not None and dist.is_initialized():
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    m0 = time.monotonic()
    for i in range(steps):
        flush()
        step_events[i][0].record(stream)
        step()
        step_events[i][1].record(stream)
    torch.cuda.synchronize()
    m1 = time.monotonic()
    wall = time.perf_counter() - t0
    # Stage breakdown: a second pass with an event between the stages (which
    # serialises them), for the per-kernel times and the roofline.
    n_stage = max(3, min(steps, 100))
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_stage)]
    for i in range(n_stage):
        flush()
        step(events[i])
    torch.cuda.synchronize()
    if dist is not None and dist.is_initialized():
        dist.barrier()
    if fa.fa_get_device_status() != 0:
        raise RuntimeError("device status reports a timed-out wait")
    stage = {"fwd": 0.0, "bwd_preprocess": 0.0, "bwd_main": 0.0, "bwd_postprocess": 0.0}
    keys = list(stage)
    for ev in events:
        for j, key in enumerate(keys):
            stage[key] += ev[j].elapsed_time(ev[j + 1])
    ms = {k2: v2 / n_stage for k2, v2 in stage.items()}
    ms["stages_sum"] = sum(ms.values())
    ms["step"] = sum(ev[0].elapsed_time(ev[1]) for ev in step_events) / steps
    ms["wall_s"] = wall
    ms["launch"] = launch_mode
    ms["steps"] = steps
    ms["window"] = (m0, m1)
    pairs = visited_tile_pairs(N, causal, inp.kv_len, inp.block_mask, B, H)
    return inp, ms, pairs


# ---------------------------------------------------- standard attention (comparison)

STANDARD_SWEEP_N = (1024, 2048, 4096, 8192, 16384)


def standard_attention(torch, q, k, v, scale, causal):
    """Standard (materialising) attention, the comparison the method is measured
    against: the whole score matrix S = scale * Q K^T is written to HBM, then
    P = softmax(S) (a second N x N tensor), then O = P V -- the three steps of the
    "Standard Attention" procedure in khetwal.com's worked example and of its section
    "The Quadratic Memory Bottleneck", written as a framework user writes them
    (cuBLAS GEMMs and PyTorch's softmax; with autograd, the backward keeps P and
    forms dP, dS as further N x N tensors).  It shares nothing with the tiled kernels.
    Inputs [B, H, N, d]; S and P are held in the inputs' dtype."""
    s = torch.matmul(q, k.transpose(-1, -2))
    s.mul_(scale)
    if causal:
        n = q.shape[-2]
        above = torch.ones(n, n, dtype=torch.bool, device=q.device).triu_(1)
        s.masked_fill_(above, float("-inf"))
    p = torch.softmax(s, dim=-1)
    return torch.matmul(p, v)


def time_standard_vs_tiled(torch, fa, flush, N, B=1, H=32, d=128, causal=True, steps=3, warmup=2, seed=1008):
    """Device time and peak extra device memory of standard attention and of the tiled
    path on one causal shape, forward and forward+backward.  Inputs are seeded N(0,1)
    drawn on the device; the peak is measured above the inputs' own allocation."""
    gen = torch.Generator(device="cuda").manual_seed(seed + N)
    shape = (B, H, N, d)
    q, k, v, do = (torch.randn(shape, generator=gen, device="cuda", dtype=torch.float32).to(torch.bfloat16)
                   for _ in range(4))
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(warmup):
            flush()
            fn()
        torch.cuda.synchronize()
        ms = 0.0
        for _ in range(steps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ms += e0.elapsed_time(e1)
        return ms / steps

    def peak_extra(fn):
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        fn()
        torch.cuda.synchronize()
        return torch.cuda.max_memory_allocated() - base

    def std_fwd():
        with torch.no_grad():
            standard_attention(torch, q, k, v, scale, causal)

    def std_fwd_bwd():
        qg, kg, vg = (t.detach().requires_grad_(True) for t in (q, k, v))
        o = standard_attention(torch, qg, kg, vg, scale, causal)
        o.backward(do)

    def ours_fwd():
        fa.attention_forward(q, k, v, scale, causal)

    def ours_fwd_bwd():
        o, lse = fa.attention_forward(q, k, v, scale, causal)
        fa.attention_backward(q, k, v, o, lse, do, scale, causal)

    row = {"N": N}
    for name, fn in (("standard_fwd", std_fwd), ("standard_fwd_bwd", std_fwd_bwd), ("tiled_fwd", ours_fwd),
                     ("tiled_fwd_bwd", ours_fwd_bwd)):
        row[name + "_ms"] = round(timed(fn), 4)
        row[name + "_peak_bytes"] = int(peak_extra(fn))
    if fa.fa_get_device_status() != 0:
        raise RuntimeError("device status reports a timed-out wait")
    row["speedup_fwd"] = round(row["standard_fwd_ms"] / row["tiled_fwd_ms"], 2)
    row["speedup_fwd_bwd"] = round(row["standard_fwd_bwd_ms"] / row["tiled_fwd_bwd_ms"], 2)
    row["score_matrix_fp32_bytes"] = 4 * B * H * N * N  # the N x N fp32 matrix of the pages' arithmetic
    del q, k, v, do
    torch.cuda.empty_cache()
    return row


def leg_report(inp, ms, pairs, peaks, clocks):
    """Throughput, fractions of peak and the roofline of one timed workload."""
    B, H, N, d = inp.q.shape
    causal = inp.causal
    f = formula = formula_fwd_flops(B, H, N, d, causal)
    alg = algorithmic_flops(pairs, d)
    useful = useful_score_pairs(N, causal, inp.kv_len, inp.block_mask, B, H) * 4.0 * d
    bwd_ms = ms["bwd_preprocess"] + ms["bwd_main"] + ms["bwd_postprocess"]
    burst = peaks["bf16_tflops"]

    def tf(flops, t_ms):
        return flops / (t_ms * 1e-3) / 1e12

    kern = {"fwd": (ms["fwd"], alg["fwd"]), "bwd_main": (ms["bwd_main"], alg["bwd"])}
    dom = max(kern, key=lambda k2: kern[k2][0])
    achieved = tf(kern[dom][1], kern[dom][0])
    long_step = ms["step"] >= 5.0
    dense_equivalent = None
    if inp.block_mask is not None:
        # a tile mask skips most of the N x N pairs: rates and fractions count the visited
        # tiles (4*128*128*d per pair forward, 2.5x that backward); the dense formula's
        # rate is reported beside them as the dense-equivalent figure
        dense_equivalent = {"fwd_tflops": round(tf(f, ms["fwd"]), 2), "bwd_tflops": round(tf(2.5 * f, bwd_ms), 2),
                            "fwd_bwd_tflops": round(tf(3.5 * f, ms["step"]), 2)}
        f = alg["fwd"]
    rep = {
        "config": {"B": B, "H": H, "N": N, "d": d, "causal": causal, "key_padding": inp.kv_len is not None,
                   "block_mask": inp.block_mask is not None, "seed": inp.seed},
        "fwd_tflops": round(tf(f, ms["fwd"]), 2),
        "bwd_tflops": round(tf(2.5 * f, bwd_ms), 2),
        "fwd_bwd_tflops": round(tf(3.5 * f, ms["step"]), 2),
        "fwd_frac_of_peak": round(tf(f, ms["fwd"]) / burst, 4),
        "bwd_frac_of_peak": round(tf(2.5 * f, bwd_ms) / burst, 4),
        "bwd_main_frac_of_peak": round(tf(alg["bwd"], ms["bwd_main"]) / burst, 4),
        "fwd_bwd_frac_of_peak": round(tf(3.5 * f, ms["step"]) / burst, 4),
        "algorithmic_tflops": {"fwd": round(tf(alg["fwd"], ms["fwd"]), 2),
                               "bwd_main": round(tf(alg["bwd"], ms["bwd_main"]), 2)},
        "useful_tflops": {"fwd": round(tf(useful, ms["fwd"]), 2),
                          "fwd_bwd": round(tf(3.5 * useful, ms["step"]), 2)},
        "stage_ms": {k2: round(v2, 5) for k2, v2 in ms.items() if k2 not in ("wall_s", "launch", "steps", "window")},
        "timed_steps": ms["steps"],
        "flops_per_step": {"formula_fwd": formula, "formula_fwd_bwd": 3.5 * formula, "visited_tile_pairs": pairs,
                           "algorithmic_fwd": alg["fwd"], "algorithmic_bwd": alg["bwd"],
                           "useful_fwd": useful, "useful_fwd_bwd": 3.5 * useful},
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 2), "peak": burst,
                     "unit": "TFLOP/s", "frac": round(achieved / burst, 4), "traffic": None,
                     "peak_source": f"bf16_tflops burst, {peaks['source']}"},
        "clocks": clocks,
    }
    if dense_equivalent is not None:
        rep["flops_basis"] = "visited 128x128 tile pairs (block mask)"
        rep["dense_equivalent"] = dense_equivalent
    if long_step:
        sus = peaks["bf16_tflops_sustained"]
        rep["roofline"]["frac_of_sustained"] = round(achieved / sus, 4)
        rep["roofline"]["peak_sustained"] = sus
    return rep


def _timed_loop(run, steps, warmup, torch, fa, flush, stream, min_seconds=0.0):
    """Warm up, then time `run` once per step (L2 flushed between steps, one event pair
    per step on the launching stream), for `steps` steps or at least `min_seconds`.
    Returns (mean ms per call, monotonic window of the timed region)."""
    torch.cuda.synchronize()
    tw = time.perf_counter()
    for _ in range(warmup):
        flush()
        run()
    torch.cuda.synchronize()
    if min_seconds > 0:
        per = (time.perf_counter() - tw) / max(1, warmup)
        steps = max(steps, min(20000, math.ceil(min_seconds / max(per, 1e-6))))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    torch.cuda.synchronize()
    m0 = time.monotonic()
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        run()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    m1 = time.monotonic()
    if fa.fa_get_device_status() != 0:
        raise RuntimeError("device status reports a timed-out wait")
    return sum(e[0].elapsed_time(e[1]) for e in ev) / steps, (m0, m1)


def time_fp8_forward(name, steps, warmup, torch, fa, flush, min_seconds=0.0):
    """fa_fwd_fp8 on the E4M3 version of a workload (one launch per step, L2 flushed
    between steps, one event pair per step on the launching stream).  Returns
    (inputs, mean ms per launch, timed window)."""
    inp = inputs.workload_fp8_inputs(name)
    B, H, N, d = inp.q8.shape
    dev = {n: torch.from_numpy(np.ascontiguousarray(getattr(inp, n))).cuda() for n in ("q8", "k8", "vt8")}
    bm = torch.from_numpy(inp.block_mask).cuda() if inp.block_mask is not None else None
    kl = torch.from_numpy(inp.kv_len).cuda() if inp.kv_len is not None else None
    o = torch.empty((B, H, N, d), device="cuda", dtype=torch.bfloat16)
    lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()

    def run():
        fa.fa_fwd_fp8(dev["q8"], dev["k8"], dev["vt8"], o, lse, inp.scale, inp.descale_q, inp.descale_k,
                      inp.descale_v, inp.causal, bm, kl, stream)

    ms, window = _timed_loop(run, steps, warmup, torch, fa, flush, stream, min_seconds)
    return inp, ms, window


def time_splitkv(name, steps, warmup, torch, fa, flush, min_seconds=0.0):
    """fa_fwd_splitkv on a query block / key cache workload (automatic split count; both
    launches of the call inside each event pair; L2 flushed between steps).  Returns
    (inputs, n_splits, mean ms per call, timed window)."""
    inp = inputs.qk_workload_inputs(name)
    B, H, Nq, d = inp.q.shape
    Nk = inp.k.shape[2]

    def dev(n):
        return torch.from_numpy(inp.device_array(n).view(np.int16)).view(torch.bfloat16).cuda()

    q, k, v = dev("q"), dev("k"), dev("v")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), device="cuda", dtype=torch.float32)
    n_splits = fa.fa_fwd_splitkv_pick_splits(B, H, Nq, Nk)
    ws = torch.empty(fa.fa_fwd_splitkv_workspace_size(B, H, Nq, d, n_splits), device="cuda", dtype=torch.uint8)
    stream = torch.cuda.current_stream()

    def run():
        fa.fa_fwd_splitkv(q, k, v, o, lse, inp.scale, None, n_splits, ws, stream)

    ms, window = _timed_loop(run, steps, warmup, torch, fa, flush, stream, min_seconds)
    return inp, n_splits, ms, window


def e2e_throughput(inp, steps, torch, fa, depth=2):
    """The same fwd+bwd through the API (fa_fwd, fa_bwd) from pinned host buffers,
    with every step's host->device copy of Q, K, V, dO (and the masks) and its
    device->host copy of O, LSE, dQ, dK, dV inside the timed region.

    The steps form a pipeline over `depth` sets of device buffers: step i+1's inputs
    upload while step i computes and step i-1's results download, on three streams.
    A set is reused only after the step before it has finished computing on it and
    its results are on the host."""
    B, H, N, d = inp.q.shape
    causal = inp.causal
    host = {n: torch.from_numpy(np.ascontiguousarray(inp.device_array(n)).view(np.int16)).view(torch.bfloat16)
            .pin_memory() for n in ("q", "k", "v", "dout")}
    host_kl = torch.from_numpy(inp.kv_len).pin_memory() if inp.kv_len is not None else None
    host_bm = torch.from_numpy(inp.block_mask).pin_memory() if inp.block_mask is not None else None
    sets = []
    for _ in range(depth):
        dev = {n: torch.empty(host[n].shape, dtype=torch.bfloat16, device="cuda") for n in host}
        sets.append({
            "in": dev,
            "kl": torch.empty_like(host_kl, device="cuda") if host_kl is not None else None,
            "bm": torch.empty_like(host_bm, device="cuda") if host_bm is not None else None,
            "out": {n: torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda") for n in ("o", "dq", "dk", "dv")},
            "lse": torch.empty((B, H, N), dtype=torch.float32, device="cuda"),
            "ws": fa.new_workspace(dev["q"]),
            "host_out": {n: torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory()
                         for n in ("o", "dq", "dk", "dv")},
            "host_lse": torch.empty((B, H, N), dtype=torch.float32).pin_memory(),
            "ev": [torch.cuda.Event() for _ in range(3)],  # inputs on device, computed, results on host
            "used": False,
        })
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    h2d += (host_kl.numel() * 4 if host_kl is not None else 0) + (host_bm.numel() if host_bm is not None else 0)
    d2h = 4 * B * H * N * d * 2 + B * H * N * 4

    def one(i):
        st = sets[i % depth]
        ev_in, ev_comp, ev_out = st["ev"]
        if st["used"]:
            s_in.wait_event(ev_comp)  # the step before on this set has read its inputs
        with torch.cuda.stream(s_in):
            for n in host:
                st["in"][n].copy_(host[n], non_blocking=True)
            if st["kl"] is not None:
                st["kl"].copy_(host_kl, non_blocking=True)
            if st["bm"] is not None:
                st["bm"].copy_(host_bm, non_blocking=True)
            ev_in.record(s_in)
        s_comp.wait_event(ev_in)
        if st["used"]:
            s_comp.wait_event(ev_out)  # its previous results are on the host
        q, k, v, do = (st["in"][n] for n in ("q", "k", "v", "dout"))
        out = st["out"]
        fa.fa_fwd(q, k, v, out["o"], st["lse"], inp.scale, causal, st["bm"], st["kl"], s_comp)
        fa.fa_bwd(q, k, v, out["o"], st["lse"], do, out["dq"], out["dk"], out["dv"], st["ws"], inp.scale, causal,
                  st["bm"], st["kl"], s_comp)
        ev_comp.record(s_comp)
        s_out.wait_event(ev_comp)
        with torch.cuda.stream(s_out):
            for n in ("o", "dq", "dk", "dv"):
                st["host_out"][n].copy_(out[n], non_blocking=True)
            st["host_lse"].copy_(st["lse"], non_blocking=True)
            ev_out.record(s_out)
        st["used"] = True

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for s in (s_comp, s_out):
        s.wait_event(e0)
    for i in range(3, 3 + steps):
        one(i)
    for s in (s_comp, s_out):
        s_in.wait_stream(s)
    e1.record(s_in)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    if fa.fa_get_device_status() != 0:
        raise RuntimeError("device status reports a timed-out wait")
    return ms, h2d, d2h


def oracle_row_sample(inp, n_rows, seed, nthreads=0):
    """The fp64 oracle's row pass (O, LSE, D and dQ) over `n_rows` seeded query rows of
    head (0, 0).  Returns (seconds, visible pairs processed)."""
    import oracle
    N = inp.q.shape[2]
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(N, size=min(n_rows, N), replace=False)).astype(np.int32)
    kl = None if inp.kv_len is None else int(inp.kv_len[0])
    t0 = time.perf_counter()
    oracle.head_rows(inp.q[0, 0], inp.k[0, 0], inp.v[0, 0], inp.dout[0, 0], inp.scale, causal=inp.causal,
                     kv_len=kl, block_mask=inp.block_mask, rows=rows, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, int(row_visible_counts(N, rows, inp.causal, kl, inp.block_mask).sum())


def extrapolated_oracle_seconds(sample_s, sample_pairs, total_pairs):
    """Whole-workload fp64 oracle time from a row-pass sample.  The oracle's column
    pass (dK, dV) does the same vector work per visible pair as its row pass (two dot
    products and two axpys of length d), so the whole forward+backward takes about
    twice the row pass, and the row pass scales with the visible pairs."""
    return 2.0 * sample_s * total_pairs / max(sample_pairs, 1)


def cpu_baseline_sample(name, n_rows=2048):
    """The fp64 oracle, as it stands, on the host cores: a seeded row sample of the
    workload's first head, extrapolated to the whole workload; plus one-thread times
    of the small workloads."""
    import oracle
    full = inputs.WORKLOADS[name]
    B, H, N, d = full["B"], full["H"], full["N"], full["d"]
    # the generator fills [B, H, N, d] in C order, so with H = 1 head (0, 0) is the full
    # workload's first head, and the key lengths (one per sequence) are the same
    inp = inputs.workload_inputs(name, H=1)
    dt, pairs = oracle_row_sample(inp, n_rows, seed=0)
    total_pairs = useful_score_pairs(N, inp.causal, inp.kv_len, inp.block_mask, B, H)
    t_all = extrapolated_oracle_seconds(dt, pairs, total_pairs)
    flops = 3.5 * formula_fwd_flops(B, H, N, d, inp.causal)
    threads = oracle.default_threads()
    res = {"value": flops / t_all / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
           "sample": (f"fp64 oracle row pass (O, LSE, dQ) on {min(n_rows, N)} seeded query rows of head (0,0) of "
                      f"{name}: {dt:.2f} s measured for {pairs:.3g} visible pairs; whole workload "
                      f"({total_pairs:.3g} pairs, forward+backward with the column pass counted at the row pass's "
                      f"per-pair cost) extrapolated to {t_all:.0f} s on {threads} threads"),
           "measured_s": round(dt, 3), "extrapolated_s": round(t_all, 1)}
    one = {}
    for small in ("tiny_fp32", "bert_large_padded", "gpt2_causal"):
        s_inp = inputs.workload_inputs(small, H=1) if small != "tiny_fp32" else inputs.workload_inputs(small)
        sB, _, sN, sd = s_inp.q.shape
        t0 = time.perf_counter()
        if small == "tiny_fp32":
            oracle.attention_forward(s_inp.q, s_inp.k, s_inp.v, s_inp.scale, nthreads=1)
            fl, what = formula_fwd_flops(1, 1, sN, sd, False), "forward, the whole workload"
        else:
            kl = None if s_inp.kv_len is None else s_inp.kv_len[:1]
            oracle.attention_backward(s_inp.q[:1, :1], s_inp.k[:1, :1], s_inp.v[:1, :1], s_inp.dout[:1, :1],
                                      s_inp.scale, causal=s_inp.causal, kv_len=kl, nthreads=1)
            fl, what = 3.5 * formula_fwd_flops(1, 1, sN, sd, s_inp.causal), "forward+backward, head (0,0)"
        dt1 = time.perf_counter() - t0
        one[small] = {"tflops": fl / dt1 / 1e12, "seconds": round(dt1, 4), "what": what}
    res["one_thread"] = one
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist
    import io_aware_exact_attention_gb300 as fa

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    fa.load()
    flush = L2Flush(torch)
    sampler = ClockSampler(local).start()
    peaks = load_peaks()
    extra = rank == 0 and world == 1 and not args.no_extra
    try:
        inp, ms, pairs = time_workload(args.workload, args.steps, args.warmup, torch, fa, flush,
                                       dist if world > 1 else None, graphs=args.graphs)
        B, H, N, d = inp.q.shape
        causal = inp.causal
        fwd_formula = formula_fwd_flops(B, H, N, d, causal)
        step_ms = reduce_max_over_ranks(ms["step"], dist if world > 1 else None)
        fwd_ms = reduce_max_over_ranks(ms["fwd"], dist if world > 1 else None)
        value = aggregate_line(3.5 * fwd_formula, world, step_ms, args.steps)
        rep = leg_report(inp, ms, pairs, peaks, sampler.window(*ms["window"]))
        rep["roofline"]["traffic"] = recorded_traffic(rep["roofline"]["kernel"], args.workload)
        bwd_ms = ms["bwd_preprocess"] + ms["bwd_main"] + ms["bwd_postprocess"]
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, **rep["config"],
                       "l2": "flushed between timed steps (512 MiB written, 256 MiB read)",
                       "launch": ms["launch"],
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "fwd_tflops": round(aggregate_line(fwd_formula, world, fwd_ms, args.steps), 3),
            "bwd_tflops": rep["bwd_tflops"],
            "fwd_frac_of_peak": rep["fwd_frac_of_peak"],
            "bwd_frac_of_peak": rep["bwd_frac_of_peak"],
            "bwd_main_frac_of_peak": rep["bwd_main_frac_of_peak"],
            "fwd_bwd_frac_of_peak": round(value / world / peaks["bf16_tflops"], 4),
            "peak_tflops": {"burst": peaks["bf16_tflops"], "sustained": peaks["bf16_tflops_sustained"],
                            "source": peaks["source"]},
            "stage_ms": rep["stage_ms"],
            "bwd_ms": round(bwd_ms, 5),
            "wall_ms_per_step": round(ms["wall_s"] / args.steps * 1e3, 5),
            "flops_per_step": rep["flops_per_step"],
            "algorithmic_tflops": rep["algorithmic_tflops"],
            "useful_tflops": rep["useful_tflops"],
            "roofline": rep["roofline"],
            "gpu_launches": 4 * args.steps,
            "clocks": rep["clocks"],
        }
        if rank == 0 and world == 1 and not args.no_e2e:
            e2e_ms, h2d, d2h = e2e_throughput(inp, max(10, min(args.steps, 200)), torch, fa)
            line["e2e"] = {"value": round(3.5 * fwd_formula / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5)}
        del inp
        legs = set(args.legs.split(","))
        if extra and "extras" in legs:
            line["extras"] = {}
            for name in EXTRA_WORKLOADS:
                if name == args.workload:
                    continue
                xin, xms, xpairs = time_workload(name, 10, 3, torch, fa, flush, graphs=args.graphs,
                                                 min_seconds=EXTRA_MIN_SECONDS)
                xrep = leg_report(xin, xms, xpairs, peaks, sampler.window(*xms["window"]))
                xrep["roofline"]["traffic"] = recorded_traffic(xrep["roofline"]["kernel"], name)
                line["extras"][name] = xrep
        if extra and "fp8" in legs:
            finp, fms, fwin = time_fp8_forward(FP8_WORKLOAD, 10, 3, torch, fa, flush, min_seconds=EXTRA_MIN_SECONDS)
            fB, fH, fN, fd = finp.q8.shape
            ff = formula_fwd_flops(fB, fH, fN, fd, finp.causal)
            fpairs = visited_tile_pairs(fN, finp.causal, finp.kv_len, finp.block_mask, fB, fH)
            fach = algorithmic_flops(fpairs, fd)["fwd"] / (fms * 1e-3) / 1e12
            fp8_peak = 2.0 * peaks["bf16_tflops"]
            line["fp8_forward"] = {
                "workload": FP8_WORKLOAD, "dtype": "e4m3 in, fp32 accumulate, bf16 out",
                "tflops": round(ff / (fms * 1e-3) / 1e12, 2), "ms": round(fms, 4),
                "roofline": {"kernel": "fwd_fp8", "bound": "tensor", "achieved": round(fach, 2),
                             "peak": round(fp8_peak, 1), "unit": "TFLOP/s", "frac": round(fach / fp8_peak, 4),
                             "traffic": recorded_traffic("fwd_fp8", FP8_WORKLOAD),
                             "peak_source": f"ASSUMED, not measured: bf16_tflops burst ({peaks['source']}) x 2, "
                                            "the nominal dense fp8:bf16 ratio (4.5 : 2.25 PFLOP/s)"},
                "clocks": sampler.window(*fwin),
            }
            del finp
        if extra and "splitkv" in legs:
            line["split_kv"] = {}
            for qk_name in sorted(args.splitkv_workloads.split(",")):
                sin, n_splits, sms, swin = time_splitkv(qk_name, 20, 3, torch, fa, flush,
                                                        min_seconds=EXTRA_MIN_SECONDS)
                sB, sH, sNq, sd = sin.q.shape
                sNk = sin.k.shape[2]
                flops, nbytes = splitkv_work(sB, sH, sNq, sNk, sd)
                gbs = nbytes / (sms * 1e-3) / 1e9
                line["split_kv"][qk_name] = {
                    "config": {"B": sB, "H": sH, "Nq": sNq, "Nk": sNk, "d": sd, "n_splits": n_splits},
                    "ms": round(sms, 4), "tflops": round(flops / (sms * 1e-3) / 1e12, 2),
                    "roofline": {"kernel": "fwd_splitkv + combine (one call)", "bound": "hbm",
                                 "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                 "frac": round(gbs / peaks["hbm_gbs"], 4),
                                 "traffic": recorded_traffic("fwd_splitkv", qk_name),
                                 "algorithmic_bytes": "Q, K, V read once, O (bf16) and LSE written"},
                    "clocks": sampler.window(*swin),
                }
                del sin
        if extra and "standard" in legs and not args.no_standard:
            std = {"config": {"B": 1, "H": 32, "d": 128, "causal": True, "dtype": "bf16",
                              "standard": "cuBLAS GEMMs + PyTorch softmax, S and P materialised in HBM "
                                          "(bf16); backward by autograd",
                              "tiled": "fa_fwd + fa_bwd (this library)",
                              "peak": "peak device bytes allocated above the inputs during one call"},
                   "sweep": []}
            t0 = time.monotonic()
            for n in STANDARD_SWEEP_N:
                std["sweep"].append(time_standard_vs_tiled(torch, fa, flush, n))
            std["clocks"] = sampler.window(t0, time.monotonic())
            line["standard_attention"] = std
    finally:
        sampler.stop()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(args.workload, args.cpu_rows)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The oracle as the reference arm, on the host cores: each step is the row pass
    over a seeded sample of query rows of the workload's first head; the rate is the
    whole workload's convention FLOPs over its extrapolated oracle time."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return
    import oracle
    full = inputs.WORKLOADS[args.workload]
    B, H, N, d = full["B"], full["H"], full["N"], full["d"]
    inp = inputs.workload_inputs(args.workload, H=1)
    kv_len = inp.kv_len
    total_pairs = useful_score_pairs(N, inp.causal, kv_len, inp.block_mask, B, H)
    for i in range(args.warmup):
        oracle_row_sample(inp, args.ref_rows, seed=i)
    t_sum, pairs_sum = 0.0, 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        dt, pairs = oracle_row_sample(inp, args.ref_rows, seed=args.warmup + i)
        t_sum += dt
        pairs_sum += pairs
    wall = time.perf_counter() - t0
    t_all = extrapolated_oracle_seconds(t_sum, pairs_sum, total_pairs)
    value = 3.5 * formula_fwd_flops(B, H, N, d, inp.causal) / t_all / 1e12
    sample = (f"fp64 oracle row pass (O, LSE, dQ) on {min(args.ref_rows, N)} seeded query rows of head (0,0) of "
              f"{args.workload} per step ({args.steps} steps, {wall:.1f} s, {pairs_sum:.3g} visible pairs); whole "
              f"workload ({total_pairs:.3g} pairs, forward+backward with the column pass counted at the row pass's "
              f"per-pair cost) extrapolated to {t_all:.0f} s")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "H": H, "N": N, "d": d, "causal": inp.causal,
                       "sample": f"{min(args.ref_rows, N)} seeded query rows of head (0,0) per step"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.default_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graphs", action="store_true", help="replay one CUDA graph per stage instead of calling the API")
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-standard", action="store_true", help="skip the standard-attention comparison sweep")
    ap.add_argument("--legs", default="extras,fp8,splitkv,standard",
                    help="comma list of the extra legs to run: extras, fp8, splitkv, standard")
    ap.add_argument("--splitkv-workloads", default=",".join(sorted(inputs.QK_WORKLOADS)),
                    help="comma list of the split-KV workloads the splitkv leg times")
    ap.add_argument("--cpu-rows", type=int, default=2048, help="query rows the cpu_baseline oracle sample covers")
    ap.add_argument("--ref-rows", type=int, default=1024, help="query rows per reference-arm step")
    args = ap.parse_args(argv)
    for qk in args.splitkv_workloads.split(","):
        if qk not in inputs.QK_WORKLOADS:
            ap.error(f"unknown split-KV workload {qk}")
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.workload == "tiny_fp32":
        ap.error("tiny_fp32 is a parity case (fp32, forward only), not a bench workload")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
