#!/usr/bin/env python3
"""Benchmark of the truncated-Taylor fixed-state attention hot path on B300.

One JSON line on rank 0. The headline `value` is prefill tokens/s on the
8,192-token workload (B=1, H=8, N=8192, d_k=16, d_v=64, n=3, fp32): one step is
one tsa_prefill call over that batch (feature map, chunk-state contraction,
span scan, inter-chunk readout, intra-chunk attention, normalise and store).
The same line carries the decode workload (B=64, H=16, d_k=16, d_v=64, n=3,
bf16 inputs, fp32 states prefilled with 65,536 tokens): microseconds per
decode step and state GB/s, and the state merge.

Timing: CUDA events on the launching stream; between timed prefill steps the
L2 is flushed by writing a buffer larger than L2 (outside the events). The
headline prefill step is one tsa_prefill call captured in a CUDA graph and
replayed, so that it measures the device and not the host's issue rate (the
per-call timing is reported beside it as ms_per_step_eager). Host-side timings
(eager steps, host time per call, the end-to-end steps) start after a short
busy wait of the host thread, so that they measure the library's host work
and not an idle core's wake-up. Decode
steps rotate over 8 independent state sets (8 x 41.5 MB > L2), captured in a
CUDA graph, so every step streams its state from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
import warnings

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "prefill tokens/s at N=8192 (n=3); decode µs/token and state GB/s on 1 B300"
PREFILL = dict(workload="prefill_B1_H8_N8192", B=1, H=8, N=8192, d_k=16, d_v=64, n_terms=3, dtype="f32", seed=2)
DECODE = dict(workload="decode_B64_H16_N65536", B=64, H=16, N=65536, d_k=16, d_v=64, n_terms=3, dtype="bf16", seed=3)
ORDER4 = dict(workload="order4_B4_H16_N32768", B=4, H=16, N=32768, d_k=16, d_v=64, n_terms=4, dtype="bf16", seed=4)
WIDE = dict(workload="wide_B2_H32_N65536", B=2, H=32, N=65536, d_k=32, d_v=128, n_terms=3, dtype="bf16", seed=5)
L2_FLUSH_BYTES = 256 << 20
DECODE_ROTATE = 8
APPEND_LENGTHS = (16, 32, 64, 256)
# tsa_plan.path values (include/tsa.h)
PATH_NAMES = ("simt", "tc", "tc_f32", "short")
ORDER_SWEEP = (1, 2, 3, 4, 5)
# chunk lengths the library builds for the fp32 prefill (64: CUDA cores; 128:
# tensor cores, the default)
CHUNK_SWEEP = (64, 128)
APPEND_REPS = 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], "measured"
    except Exception:
        return 6400.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_seed(seed: int, rank: int) -> int:
    """Weak scaling: every rank runs its own batch of the workload, drawn from
    its own seed."""
    return seed + 1000 * rank


def warm_host(seconds: float = 0.2) -> None:
    """Keep this thread busy for a moment before a host-side timing. A host
    core that has idled (sleeps, blocking synchronizations) first runs the
    library's host code (argument checks, plan, tensor maps, launches)
    several times slower: measured 65-95 us per prefill call instead of
    15 us, and eager steps that wait for their launches."""
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        pass


def max_over_ranks(x: float, ws: int, device) -> float:
    """The slowest rank's time (all_reduce MAX over the process group; the
    tensor lives on `device`: the GPU under NCCL, the CPU under gloo)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(ws: int, tokens_per_rank: int, ms_max: float) -> float:
    """Whole-job tokens/s: all ranks' tokens over the slowest rank's time."""
    return ws * tokens_per_rank / (ms_max / 1e3)


def _algorithmic_prefill_bytes(w) -> int:
    """q, k, v read + out written (element size of the dtype) + final states
    written (fp32, D*(d_v+1) per head)."""
    es = 4 if w["dtype"] == "f32" else 2
    heads = w["B"] * w["H"]
    D = sum(__import__("math").comb(w["d_k"] + m - 1, m) for m in range(w["n_terms"]))
    io = heads * w["N"] * (2 * w["d_k"] + 2 * w["d_v"]) * es
    return io + heads * D * (w["d_v"] + 1) * 4


def _algorithmic_prefill_flops(w) -> float:
    """Per token-head: state update 2*D*(d_v+1), readout 2*D*(d_v+1), intra-chunk
    2*C*(d_k+d_v+1) at the reference chunk C = 64 (dense; padding and the
    implementation's own chunk length are not counted)."""
    import math
    D = sum(math.comb(w["d_k"] + m - 1, m) for m in range(w["n_terms"]))
    per = 4 * D * (w["d_v"] + 1) + 2 * 64 * (w["d_k"] + w["d_v"] + 1)
    return float(per) * w["B"] * w["H"] * w["N"]


def _bf16_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["bf16_tflops"], p["bf16_tflops_sustained"], "measured"
    except Exception:
        return 1800.0, 1400.0, "fallback"


def _algorithmic_decode_bytes(w) -> int:
    """State read + written once per step (D*(d_v+1) fp32 per head; padding not
    counted) plus the step's q, k, v in and out."""
    es = 4 if w["dtype"] == "f32" else 2
    heads = w["B"] * w["H"]
    D = sum(__import__("math").comb(w["d_k"] + m - 1, m) for m in range(w["n_terms"]))
    return heads * (2 * D * (w["d_v"] + 1) * 4 + (2 * w["d_k"] + 2 * w["d_v"]) * es)


def _algorithmic_append_bytes(w, L: int) -> int:
    """A short append of L tokens to every head: the state read + written once
    (D*(d_v+1) fp32 per head; padding not counted) plus the segment's q, k, v in
    and out."""
    es = 4 if w["dtype"] == "f32" else 2
    heads = w["B"] * w["H"]
    D = sum(__import__("math").comb(w["d_k"] + m - 1, m) for m in range(w["n_terms"]))
    return heads * (2 * D * (w["d_v"] + 1) * 4 + L * (2 * w["d_k"] + 2 * w["d_v"]) * es)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms; the summary
    keeps the samples taken between __enter__ and __exit__ (the timed work).

    The sampler process must be started before this process initialises CUDA:
    a child process started after that slowed every later host-side CUDA call
    of the parent about twofold (kernel launches, event records), whatever it
    queried, while one started before had no effect."""
    Q = ("timestamp,index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int):
        vis = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
        self.gpu = vis[local_rank] if local_rank < len(vis) else str(local_rank)
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL,
                                      preexec_fn=lambda: os.nice(19))
        except Exception:
            self.p = None
        return self

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()
            self.p = None

    def __enter__(self):
        time.sleep(0.25)
        self.t0 = time.time()
        return self

    def __exit__(self, *a):
        self.t1 = time.time()
        time.sleep(0.15)

    def _mine(self, rows):
        """Rows of the GPU this rank uses: by uuid, by index, or the only one."""
        if self.gpu.startswith("GPU-"):
            return [r for r in rows if r[2].strip() == self.gpu]
        idx = {r[1].strip() for r in rows}
        if len(idx) == 1:
            return rows
        return [r for r in rows if r[1].strip() == self.gpu]

    def summary(self):
        from datetime import datetime
        self.stop()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        rows = [r for r in rows if len(r) >= 11]
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self._mine(rows):
            try:
                ts = datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if self.t0 is None or not (self.t0 <= ts <= self.t1):
                    continue
                sm.append(float(r[3])); mx = max(mx, float(r[4]))
                for nm, val in zip(names, r[7:11]):
                    if "Active" in val and "Not" not in val:
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "every_ms": 100}


def _oracle_head_prefill(args):
    """One head's recurrent float64 prefill (a worker of the multi-core leg);
    returns its wall time in seconds."""
    w, h = args
    from fixed_state_recurrence_phi_b300.inputs import np_qkv
    from oracle import tsa_oracle as O
    q, k, v = np_qkv(w["N"], w["d_k"], w["d_v"], seed=[w["seed"], h])
    t0 = time.perf_counter()
    O.prefill_recurrent(q, k, v, w["n_terms"])
    return time.perf_counter() - t0


def cpu_baseline_prefill(w, inputs=None, max_heads=None):
    """The float64 oracle (recurrent form, as it stands) on one host core.
    With `inputs` (host float64 q, k, v of the GPU run, [heads, N, d]) it runs
    on those and also returns its outputs and states per head, for the parity
    figures; otherwise on freshly drawn inputs of the same recipe."""
    from fixed_state_recurrence_phi_b300.inputs import np_qkv
    from oracle import tsa_oracle as O
    heads = w["B"] * w["H"] if max_heads is None else max_heads
    t, refs = 0.0, []
    for h in range(heads):
        if inputs is None:
            q, k, v = np_qkv(w["N"], w["d_k"], w["d_v"], seed=[w["seed"], h])
        else:
            q, k, v = inputs[0][h], inputs[1][h], inputs[2][h]
        t0 = time.perf_counter()
        refs.append(O.prefill_recurrent(q, k, v, w["n_terms"]))
        t += time.perf_counter() - t0
    per_head = t / heads
    all_heads = w["B"] * w["H"]
    src = "the GPU run's own inputs" if inputs is not None else "inputs of the same recipe"
    return {"value": w["B"] * w["N"] / (per_head * all_heads), "unit": "tokens/s", "cores": 1,
            "kind": "oracle",
            "sample": f"recurrent float64 prefill, {heads} of {all_heads} heads x {w['N']} tokens on 1 "
                      f"core ({src}); tokens/s = B*N / (mean head time x {all_heads} heads)"}, refs


def parity_vs_oracle(out_g, S_g, refs, dv, tol):
    """The timed call's results against the oracle's, per head, for the
    outputs, the state's value part and its normaliser column (worst head of
    each): normwise max|g - r| / max|r| (the parity measure, tolerance `tol`);
    elementwise |g - r| / |r| over the elements with |r| >= 1% of max|r|; and
    elementwise |g - r| / (|r| + 1e-6 max|r|) over all elements."""
    def three(g, r):
        a = float(np.abs(r).max())
        d = np.abs(g - r)
        big = np.abs(r) >= 0.01 * a
        return (float(d.max() / a), float((d[big] / np.abs(r[big])).max()),
                float((d / (np.abs(r) + 1e-6 * a)).max()))
    worst = {"out": [0.0, 0.0, 0.0], "state": [0.0, 0.0, 0.0], "normaliser": [0.0, 0.0, 0.0]}
    for h, (o_r, S_r) in enumerate(refs):
        for key, g, r in (("out", out_g[h], o_r), ("state", S_g[h][:, :dv], S_r[:, :dv]),
                          ("normaliser", S_g[h][:, dv], S_r[:, dv])):
            worst[key] = [max(x, y) for x, y in zip(worst[key], three(g, r))]
    r3 = lambda x: float(f"{x:.3g}")
    return {"heads": len(refs), "tol_normwise": tol,
            "normwise": {k: r3(v[0]) for k, v in worst.items()},
            "elementwise_ge_1pct": {k: r3(v[1]) for k, v in worst.items()},
            "elementwise_floor_1e-6": {k: r3(v[2]) for k, v in worst.items()},
            "ok": all(v[0] <= tol for v in worst.values())}


def cpu_baseline_prefill_cores(w):
    """The same oracle with the heads spread over the host cores (one process
    per head, started with spawn: this process has initialised CUDA)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    heads = w["B"] * w["H"]
    cores = max(1, min(heads, len(os.sched_getaffinity(0))))
    with cf.ProcessPoolExecutor(max_workers=cores, mp_context=mp.get_context("spawn")) as ex:
        list(ex.map(_oracle_head_prefill, [(w, 0)] * cores))   # warm the workers (imports)
        t0 = time.perf_counter()
        list(ex.map(_oracle_head_prefill, [(w, h) for h in range(heads)]))
        t = time.perf_counter() - t0
    return {"value": w["B"] * w["N"] / t, "unit": "tokens/s", "cores": cores,
            "sample": f"recurrent float64 prefill of all {heads} heads x {w['N']} tokens, "
                      f"one process per head on {cores} cores (wall time of the batch)"}


def cpu_baseline_prefill_extrapolated(w, n_sample=4096):
    """The oracle's recurrent float64 prefill of one head of workload `w` on
    its first n_sample tokens (1 core), extrapolated to w's N and all its heads:
    the recurrent form does the same work for every token, so the time is
    linear in N and in the number of heads. Labelled as extrapolated."""
    from fixed_state_recurrence_phi_b300.inputs import np_qkv
    from oracle import tsa_oracle as O
    q, k, v = np_qkv(n_sample, w["d_k"], w["d_v"], seed=[w["seed"], 0])
    t0 = time.perf_counter()
    O.prefill_recurrent(q, k, v, w["n_terms"])
    t = time.perf_counter() - t0
    heads = w["B"] * w["H"]
    t_full = t * (w["N"] / n_sample) * heads
    return {"tokens_per_s": w["B"] * w["N"] / t_full, "s_per_call": t_full, "cores": 1, "extrapolated": True,
            "sample": f"recurrent float64 prefill of 1 head x {n_sample} tokens on 1 core ({t:.3f} s), "
                      f"extrapolated linearly to {w['N']} tokens x {heads} heads",
            "what": f"prefill, {w['workload']} (extrapolated)"}


def cpu_baseline_decode(w, steps=2):
    """The oracle's float64 decode step (as it stands: one call per head) over
    every head of the decode workload, on one core, for a few steps."""
    from oracle import tsa_oracle as O
    heads = w["B"] * w["H"]
    D = sum(__import__("math").comb(w["d_k"] + m - 1, m) for m in range(w["n_terms"]))
    rng = np.random.default_rng(w["seed"])
    S = [np.zeros((D, w["d_v"] + 1)) for _ in range(heads)]
    x = rng.standard_normal((steps, heads, 2, w["d_k"]))
    x /= np.linalg.norm(x, axis=-1, keepdims=True)
    vv = rng.standard_normal((steps, heads, w["d_v"]))
    t0 = time.perf_counter()
    for s in range(steps):
        for h in range(heads):
            _, S[h] = O.decode_step(x[s, h, 0], x[s, h, 1], vv[s, h], S[h], w["n_terms"])
    t = (time.perf_counter() - t0) / steps
    return {"us_per_step": t * 1e6, "state_GBps": heads * D * (w["d_v"] + 1) * 8 * 2 / t / 1e9,
            "cores": 1, "sample": f"{steps} steps over all {heads} heads, float64, one decode_step call per "
                                  f"head (state bytes counted in float64)"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    w = PREFILL
    heads = w["B"] * w["H"]
    times = []
    for i in range(args.warmup + args.steps):
        t_step = sum(_oracle_head_prefill((w, h)) for h in range(heads))
        if i >= args.warmup:
            times.append(t_step)
    t = statistics.mean(times)
    value = w["B"] * w["N"] / t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w["workload"], "B": w["B"], "H": w["H"], "N": w["N"], "d_k": w["d_k"],
                   "d_v": w["d_v"], "n_terms": w["n_terms"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: recurrent float64 prefill of all {heads} heads x {w['N']} "
                                   "tokens on 1 host core (inputs drawn outside the timing)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    ws, rank, local = _dist()
    # the extension build (a compiler subprocess when sources changed) and the
    # clock sampler both start before CUDA is initialised (ClockSampler)
    from fixed_state_recurrence_phi_b300 import build as tsa_build
    tsa_build.build()
    clk = ClockSampler(local).start()
    try:
        _run_ours(args, clk)
    finally:
        clk.stop()


def _run_ours(args, clk):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    from fixed_state_recurrence_phi_b300 import tsa as T
    from fixed_state_recurrence_phi_b300.inputs import torch_qkv

    hbm_peak, peak_src = _peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    def slowest(x: float) -> float:
        return max_over_ranks(x, ws, dev)

    # ---------------- prefill workload (weak scaling: one batch per rank) ----
    w = PREFILL
    cfg = T.Config(w["B"], w["H"], w["d_k"], w["d_v"], w["n_terms"], w["dtype"])
    q, k, v = torch_qkv(w["B"], w["H"], w["N"], w["d_k"], w["d_v"], w["dtype"], rank_seed(w["seed"], rank),
                        0, dev)
    out = torch.empty((w["B"], w["H"], w["N"], w["d_v"]), dtype=q.dtype, device=dev)
    st = T.new_states(cfg, dev)
    plan = T.prefill_plan(cfg, w["N"])

    def prefill_step():
        T.prefill(cfg, w["N"], q, k, v, out, st, stream=stream)

    do_pre = args.only in ("all", "prefill")
    do_dec = args.only in ("all", "decode")
    ms = ms_eager = e2e_ms = host_us = float("nan"); h2d = d2h = 0
    timing = "n/a"
    dec_us = eager_us = long_prefill_ms = merge_ms = float("nan")
    append_lines = []
    pre_result = None
    steps, reps = 1024, 3
    dw = DECODE
    dcfg = T.Config(dw["B"], dw["H"], dw["d_k"], dw["d_v"], dw["n_terms"], dw["dtype"])
    with clk:
      if do_pre:
          for _ in range(max(3, args.warmup)):
              flush.fill_(1.0)
              prefill_step()
          barrier()
          evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)]
          warm_host()
          for i in range(args.steps):
              flush.fill_(float(i))
              evs[i][0].record(stream)
              prefill_step()
              evs[i][1].record(stream)
          barrier()
          step_ms = [a.elapsed_time(b) for a, b in evs]
          ms = slowest(statistics.mean(step_ms))
          # host time of one call (argument checks, plan, tensor maps, launches)
          hs = []
          warm_host()
          for _ in range(9):
              torch.cuda.synchronize()
              h0 = time.perf_counter()
              prefill_step()
              hs.append((time.perf_counter() - h0) * 1e6)
          torch.cuda.synchronize()
          host_us = statistics.median(hs)
          ms_eager = ms
          if ws == 1 and not args.no_cpu_baseline:
              # the timed call's results, checked against the oracle below
              pre_result = (out[0].double().cpu().numpy(), T.canonical_states(cfg, st)[0].double().cpu().numpy(),
                            [x[0].double().cpu().numpy() for x in (q, k, v)])

          # the same call captured once in a CUDA graph and replayed: device
          # time of the step, independent of how fast the host issues it
          try:
              g = torch.cuda.CUDAGraph()
              gs = torch.cuda.Stream()
              gs.wait_stream(stream)
              with torch.cuda.stream(gs):
                  with torch.cuda.graph(g, stream=gs):
                      T.prefill(cfg, w["N"], q, k, v, out, st, stream=gs)
              stream.wait_stream(gs)
              for _ in range(max(3, args.warmup)):
                  flush.fill_(1.0)
                  g.replay()
              barrier()
              gevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(args.steps)]
              for i in range(args.steps):
                  flush.fill_(float(i))
                  gevs[i][0].record(stream)
                  g.replay()
                  gevs[i][1].record(stream)
              barrier()
              T.sync_status(stream)
              ms = slowest(statistics.mean([a.elapsed_time(b) for a, b in gevs]))
              timing = "CUDA graph of one tsa_prefill call, replayed per step"
              del g
          except Exception as e:  # capture unsupported here: keep the per-call timing
              timing = f"one tsa_prefill call per step (graph capture failed: {type(e).__name__})"

          # -------- e2e: pinned host buffers in, host result out, through the ABI.
          # Each step copies its inputs in, runs the call and copies its outputs
          # and states out, on one of two streams with their own device buffers,
          # so that one step's copies overlap the other's (the two directions
          # use separate copy engines); whole-job time over the steps.
          qh = q.cpu().pin_memory(); kh = k.cpu().pin_memory(); vh = v.cpu().pin_memory()
          e2e_streams = [torch.cuda.Stream(), torch.cuda.Stream()]
          bufs = []
          for _ in range(2):
              bufs.append(dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v),
                               out=torch.empty_like(out), st=torch.empty_like(st),
                               oh=torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                               sh=torch.empty(st.shape, dtype=st.dtype).pin_memory(),
                               flush=torch.empty(L2_FLUSH_BYTES // 8, dtype=torch.float32, device=dev)))

          def e2e_step(i):
              bb, es = bufs[i % 2], e2e_streams[i % 2]
              with torch.cuda.stream(es):
                  bb["q"].copy_(qh, non_blocking=True); bb["k"].copy_(kh, non_blocking=True)
                  bb["v"].copy_(vh, non_blocking=True)
                  bb["flush"].fill_(float(i))   # evict the previous step's data from L2
                  T.prefill(cfg, w["N"], bb["q"], bb["k"], bb["v"], bb["out"], bb["st"], stream=es)
                  bb["oh"].copy_(bb["out"], non_blocking=True); bb["sh"].copy_(bb["st"], non_blocking=True)

          for i in range(4):
              e2e_step(i)
          barrier()
          a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
          warm_host()
          a.record(stream)
          for es in e2e_streams:
              es.wait_stream(stream)
          for i in range(args.steps):
              e2e_step(i)
          for es in e2e_streams:
              stream.wait_stream(es)
          b.record(stream)
          barrier()
          T.sync_status(stream)
          e2e_ms = slowest(a.elapsed_time(b) / args.steps)
          oh, sh = bufs[0]["oh"], bufs[0]["sh"]
          h2d = sum(x.numel() * x.element_size() for x in (qh, kh, vh))
          d2h = oh.numel() * oh.element_size() + sh.numel() * sh.element_size()
          qd = kd = vd = None
          del bufs
          del qh, kh, vh, oh, sh, qd, kd, vd

      tc_lines = []
      for tw in (ORDER4, WIDE):
          if args.only not in ("all", tw["workload"].split("_")[0]):
              continue
          tw = dict(tw)
          if args.tc_n:
              tw["N"] = args.tc_n
          tcfg = T.Config(tw["B"], tw["H"], tw["d_k"], tw["d_v"], tw["n_terms"], tw["dtype"])
          tq, tk, tv = torch_qkv(tw["B"], tw["H"], tw["N"], tw["d_k"], tw["d_v"], tw["dtype"],
                                 rank_seed(tw["seed"], rank), 0, dev)
          tout = torch.empty((tw["B"], tw["H"], tw["N"], tw["d_v"]), dtype=tq.dtype, device=dev)
          tst = T.new_states(tcfg, dev)
          tplan = T.prefill_plan(tcfg, tw["N"])
          for _ in range(3):
              flush.fill_(1.0)
              T.prefill(tcfg, tw["N"], tq, tk, tv, tout, tst, stream=stream)
          barrier()
          tev = []
          for i in range(max(3, args.steps // 2)):
              flush.fill_(float(i))
              a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
              a.record(stream)
              T.prefill(tcfg, tw["N"], tq, tk, tv, tout, tst, stream=stream)
              b.record(stream)
              tev.append((a, b))
          barrier()
          tms = slowest(statistics.mean([a.elapsed_time(b) for a, b in tev]))
          T.sync_status(stream)
          fl = _algorithmic_prefill_flops(tw)
          pk_burst, pk_sust, pk_src = _bf16_peaks()
          ach = fl / (tms / 1e3) / 1e12
          tc_lines.append({
              "workload": tw["workload"], "N": tw["N"], "ms": tms,
              "tokens_per_s": ws * tw["B"] * tw["N"] / (tms / 1e3),
              "path": ("tensor cores (tcgen05, bf16 in, fp32 TMEM accumulators"
                       + (", CTA pairs" if tplan["cluster"] == 2 else "") + ")") if tplan["path"] == 1 else "simt",
              "plan": {k2: tplan[k2] for k2 in ("chunk", "n_slices", "slice_width", "n_spans", "launches", "cluster")},
              "roofline": {"bound": "tensor", "achieved": ach, "peak": pk_burst, "unit": "TFLOP/s",
                           "frac": ach / pk_burst, "frac_of_sustained": ach / pk_sust,
                           "peak_source": f"{pk_src} cuBLAS bf16 (burst; sustained {pk_sust})",
                           "algorithmic_flops": fl},
          })
          del tq, tk, tv, tout, tst
          torch.cuda.empty_cache()

      order_lines = []
      if args.only in ("all", "orders"):
          # ---------------- order sweep on the prefill workload's shape -------
          # state size and throughput per number of Taylor terms (the accuracy
          # side of the sweep is a parity test against exact softmax)
          for n in ORDER_SWEEP:
              ocfg = T.Config(w["B"], w["H"], w["d_k"], w["d_v"], n, w["dtype"])
              oplan = T.prefill_plan(ocfg, w["N"])
              ost = T.new_states(ocfg, dev)
              T.prefill(ocfg, w["N"], q, k, v, out, ost, stream=stream)
              barrier()
              og = torch.cuda.CUDAGraph()
              ogs = torch.cuda.Stream()
              ogs.wait_stream(stream)
              with torch.cuda.stream(ogs):
                  with torch.cuda.graph(og, stream=ogs):
                      T.prefill(ocfg, w["N"], q, k, v, out, ost, stream=ogs)
              stream.wait_stream(ogs)
              for _ in range(3):
                  flush.fill_(1.0)
                  og.replay()
              barrier()
              oev = []
              for i in range(max(3, args.steps // 2)):
                  flush.fill_(float(i))
                  a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                  a.record(stream)
                  og.replay()
                  b.record(stream)
                  oev.append((a, b))
              barrier()
              T.sync_status(stream)
              oms = slowest(statistics.mean([a.elapsed_time(b) for a, b in oev]))
              del og
              order_lines.append({
                  "workload": w["workload"], "n_terms": n, "ms": oms,
                  "tokens_per_s": ws * w["B"] * w["N"] / (oms / 1e3),
                  "state_bytes_per_head": T.state_elems(ocfg) * 4,
                  "path": PATH_NAMES[oplan["path"]],
                  "timing": "CUDA graph of one tsa_prefill call, replayed per step, L2 flushed between steps",
              })
              del ost

      chunk_lines = []
      if args.only in ("all", "orders"):
          # ---------------- chunk lengths on the prefill workload -----------
          for ch in CHUNK_SWEEP:
              ccfg = T.Config(w["B"], w["H"], w["d_k"], w["d_v"], w["n_terms"], w["dtype"], ch)
              cplan = T.prefill_plan(ccfg, w["N"])
              cst = T.new_states(ccfg, dev)
              T.prefill(ccfg, w["N"], q, k, v, out, cst, stream=stream)
              barrier()
              cg = torch.cuda.CUDAGraph()
              cgs = torch.cuda.Stream()
              cgs.wait_stream(stream)
              with torch.cuda.stream(cgs):
                  with torch.cuda.graph(cg, stream=cgs):
                      T.prefill(ccfg, w["N"], q, k, v, out, cst, stream=cgs)
              stream.wait_stream(cgs)
              for _ in range(3):
                  flush.fill_(1.0)
                  cg.replay()
              barrier()
              cev = []
              for i in range(max(3, args.steps // 2)):
                  flush.fill_(float(i))
                  a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                  a.record(stream)
                  cg.replay()
                  b.record(stream)
                  cev.append((a, b))
              barrier()
              T.sync_status(stream)
              cms = slowest(statistics.mean([a.elapsed_time(b) for a, b in cev]))
              del cg, cst
              chunk_lines.append({"chunk": ch, "ms": cms, "path": PATH_NAMES[cplan["path"]],
                                  "n_spans": cplan["n_spans"]})

      if do_dec:
          # ---------------- decode workload ----------------------------------
          dstates = []
          dq, dk, dv = torch_qkv(dw["B"], dw["H"], args.decode_prefill_n, dw["d_k"], dw["d_v"], dw["dtype"],
                                 rank_seed(dw["seed"], rank), 0, dev)
          dout = torch.empty((dw["B"], dw["H"], args.decode_prefill_n, dw["d_v"]), dtype=dq.dtype, device=dev)
          s0 = T.new_states(dcfg, dev)
          pa, pb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
          pa.record(stream)
          T.prefill(dcfg, args.decode_prefill_n, dq, dk, dv, dout, s0, stream=stream)
          pb.record(stream)
          torch.cuda.synchronize()
          long_prefill_ms = pa.elapsed_time(pb)
          del dq, dk, dv, dout
          torch.cuda.empty_cache()
          for _ in range(DECODE_ROTATE):
              dstates.append(s0.clone())
          tq, tk, tv = torch_qkv(dw["B"], dw["H"], steps, dw["d_k"], dw["d_v"], dw["dtype"],
                                 rank_seed(dw["seed"], rank), 1, dev)
          tq = tq.permute(2, 0, 1, 3).contiguous(); tk = tk.permute(2, 0, 1, 3).contiguous()
          tv = tv.permute(2, 0, 1, 3).contiguous()
          touts = torch.empty((steps, dw["B"], dw["H"], dw["d_v"]), dtype=tq.dtype, device=dev)

          def decode_all(s):
              for t in range(steps):
                  T.decode_step(dcfg, tq[t], tk[t], tv[t], touts[t], dstates[t % DECODE_ROTATE], stream=s)

          # eager, per-step events (first 64 steps, L2 rotation as in the graph)
          decode_all(stream)
          barrier()
          eager = []
          warm_host()
          for t in range(64):
              a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
              a.record(stream)
              T.decode_step(dcfg, tq[t], tk[t], tv[t], touts[t], dstates[t % DECODE_ROTATE], stream=stream)
              b.record(stream)
              eager.append((a, b))
          barrier()
          eager_us = statistics.median([a.elapsed_time(b) * 1e3 for a, b in eager])
          # graph of 1024 steps
          gs = torch.cuda.Stream()
          gs.wait_stream(stream)
          g = torch.cuda.CUDAGraph()
          with torch.cuda.stream(gs):
              with torch.cuda.graph(g, stream=gs):
                  decode_all(gs)
          stream.wait_stream(gs)
          g.replay(); barrier()
          a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
          a.record(stream)
          for _ in range(reps):
              g.replay()
          b.record(stream)
          barrier()
          dec_us = slowest(a.elapsed_time(b) * 1e3 / (reps * steps))

          # ---------------- short appends (prefill with ACCUMULATE) ---------
          # L new tokens per head folded into the decode states: one
          # tsa_prefill call continuing every head; a CUDA graph of one call
          # per state set (rotated, > L2), replayed.
          for L in APPEND_LENGTHS:
              aq, ak, av = torch_qkv(dw["B"], dw["H"], L, dw["d_k"], dw["d_v"], dw["dtype"],
                                     rank_seed(dw["seed"], rank), 2, dev)
              ao = torch.empty((dw["B"], dw["H"], L, dw["d_v"]), dtype=aq.dtype, device=dev)
              aplan = T.prefill_plan(dcfg, L)

              def append_all(s):
                  for st_i in dstates:
                      T.prefill(dcfg, L, aq, ak, av, ao, st_i, accumulate=True, stream=s)

              append_all(stream)
              barrier()
              gs = torch.cuda.Stream()
              gs.wait_stream(stream)
              g = torch.cuda.CUDAGraph()
              with torch.cuda.stream(gs):
                  with torch.cuda.graph(g, stream=gs):
                      append_all(gs)
              stream.wait_stream(gs)
              g.replay(); barrier()
              a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
              a.record(stream)
              for _ in range(APPEND_REPS):
                  g.replay()
              b.record(stream)
              barrier()
              T.sync_status(stream)
              a_us = slowest(a.elapsed_time(b) * 1e3 / (APPEND_REPS * len(dstates)))
              abytes = _algorithmic_append_bytes(dw, L)
              append_lines.append({
                  "workload": f"append_B{dw['B']}_H{dw['H']}_L{L}", "L": L, "us_per_call": a_us,
                  "tokens_per_s": ws * dw["B"] * L / (a_us / 1e6),
                  "path": PATH_NAMES[aplan["path"]],
                  "roofline": {"bound": "hbm", "achieved": abytes / (a_us / 1e6) / 1e9, "peak": hbm_peak,
                               "unit": "GB/s", "frac": abytes / (a_us / 1e6) / 1e9 / hbm_peak,
                               "algorithmic_bytes": abytes},
                  "timing": f"CUDA graph of {len(dstates)} calls (one per state set) x {APPEND_REPS}",
              })
              del g, aq, ak, av, ao

          # ---------------- merge -------------------------------------------
          m_ms = []
          for i in range(10):
              flush.fill_(float(i))
              a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
              a.record(stream); T.state_merge(dcfg, dstates[0], dstates[1], stream=stream); b.record(stream)
              m_ms.append((a, b))
          barrier()
          merge_ms = statistics.median([a.elapsed_time(b) for a, b in m_ms])

      # ---------------- the exact-softmax comparison (one GPU) ---------------
      softmax = None
      if args.only in ("all", "softmax") and ws == 1:
          softmax = softmax_comparison(T, dev, stream, flush, ws, rank)
    clocks = clk.summary()

    # ---------------- report -------------------------------------------------
    tokens = w["B"] * w["N"]
    value = weak_scaling_value(ws, tokens, ms) if do_pre else None
    pre_bytes = _algorithmic_prefill_bytes(w)
    dec_bytes = _algorithmic_decode_bytes(dw)
    state_bytes_step = dw["B"] * dw["H"] * T.state_elems(dcfg) * 4 * 2
    ach = pre_bytes / (ms / 1e3) / 1e9 if do_pre else float("nan")
    if rank != 0:
        return
    cpu = parity = None
    if ws == 1 and do_pre and not args.no_cpu_baseline:
        cpu, refs = cpu_baseline_prefill(w, inputs=pre_result[2] if pre_result else None)
        if pre_result:
            parity = parity_vs_oracle(pre_result[0], pre_result[1], refs, w["d_v"], 1e-4)
        cpu["legs"] = [dict(cpu_baseline_prefill_cores(w), what="prefill, heads over cores")]
        if do_dec:
            cpu["legs"].append(dict(cpu_baseline_decode(dw), what=f"decode step, {dw['workload']}"))
        for tw in (ORDER4, WIDE):
            cpu["legs"].append(cpu_baseline_prefill_extrapolated(tw))
    traffic = _profile_traffic()
    r3 = lambda x: None if x is None else float(f"{x:.4g}")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w["workload"], "B": w["B"], "H": w["H"], "N": w["N"], "d_k": w["d_k"],
                   "d_v": w["d_v"], "n_terms": w["n_terms"], "chunk": plan["chunk"],
                   "n_spans": plan["n_spans"], "path": PATH_NAMES[plan["path"]],
                   "l2": "flushed between timed steps (256 MB write)", "timing": timing},
        "roofline": {"bound": "hbm", "kernel": "tsa_prefill (all launches of the call)",
                     "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak,
                     "peak_source": f"{peak_src} (copy bandwidth)",
                     "algorithmic_bytes": pre_bytes,
                     "traffic": traffic.get("prefill")},
        "e2e": {"value": weak_scaling_value(ws, tokens, e2e_ms) if do_pre else None, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "timing": "pinned host q, k, v in and out + states out every step; steps alternate over two "
                          "streams (copies of one overlap the other's call); whole-job time / steps"},
        "gpu_launches": args.steps * plan["launches"] if do_pre else 0,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "ms_per_step_eager": ms_eager,
        "host_us_per_call": host_us,
        # compact sections; the tensor-core prefill and the decode come last
        "append": [{"L": a["L"], "us": r3(a["us_per_call"]), "frac_hbm": r3(a["roofline"]["frac"]),
                    "path": a["path"]} for a in append_lines],
        "orders": [{"n": o["n_terms"], "ms": r3(o["ms"]), "state_B_per_head": o["state_bytes_per_head"],
                    "path": o["path"]} for o in order_lines],
        "merge": {"ms": r3(merge_ms), "GBps": r3(3 * T.state_bytes(dcfg) / (merge_ms / 1e3) / 1e9)},
        # the timed 8192-token call against the float64 oracle, every head
        "parity": parity,
        "chunks": [{"chunk": c_["chunk"], "ms": r3(c_["ms"]), "path": c_["path"], "n_spans": c_["n_spans"]}
                   for c_ in chunk_lines],
        # the pages' speed comparison re-measured here: states path against
        # exact softmax on the library's fastest attention backend
        "softmax": softmax,
        "prefill_tensor_core": [
            {"workload": t["workload"], "ms": r3(t["ms"]), "tokens_per_s": r3(t["tokens_per_s"]),
             "plan": t["plan"],
             "roofline": {"bound": "tensor", "achieved": r3(t["roofline"]["achieved"]),
                          "peak": t["roofline"]["peak"], "unit": "TFLOP/s", "frac": r3(t["roofline"]["frac"]),
                          "frac_of_sustained": r3(t["roofline"]["frac_of_sustained"]),
                          "traffic": traffic.get(t["workload"])}} for t in tc_lines],
        "decode": {"workload": dw["workload"], "us_per_step": r3(dec_us), "us_per_step_eager": r3(eager_us),
                   "state_GBps": r3(state_bytes_step / (dec_us / 1e6) / 1e9),
                   "roofline": {"bound": "hbm", "kernel": "decode_kernel",
                                "achieved": r3(dec_bytes / (dec_us / 1e6) / 1e9), "peak": hbm_peak,
                                "unit": "GB/s", "frac": r3(dec_bytes / (dec_us / 1e6) / 1e9 / hbm_peak),
                                "algorithmic_bytes": dec_bytes, "traffic": traffic.get("decode")},
                   "timing": f"graph of {steps} steps x {reps}, {DECODE_ROTATE} state sets (> L2)",
                   "gpu_launches": reps * steps, "states_prefill_ms": r3(long_prefill_ms)},
    }
    print(json.dumps(line), flush=True)


SOFTMAX_PREFILL_N = (256, 512, 1024, 2048, 4096, 8192, 16384, 32768, 65536)
SOFTMAX_DECODE_N = (1024, 4096, 16384, 65536)
SOFTMAX_FIT_MIN_N = 2048


def loglog_slope(ns, ts) -> float:
    """Least-squares exponent p of t ~ N^p."""
    return float(np.polyfit(np.log(np.asarray(ns, float)), np.log(np.asarray(ts, float)), 1)[0])


def crossover_n(ns, ours, soft):
    """The sequence length above which the states path stays faster than
    softmax: log-log interpolation across the last sweep interval where the
    sign of log(soft / ours) changes. ns[0] if ours is faster everywhere,
    None if never."""
    r = [float(np.log(s / o)) for s, o in zip(soft, ours)]
    if r[-1] <= 0:
        return None
    i = max([j for j, x in enumerate(r) if x <= 0], default=-1)
    if i < 0:
        return ns[0]
    x0, x1 = np.log(ns[i]), np.log(ns[i + 1])
    return float(np.exp(x0 + (0.0 - r[i]) / (r[i + 1] - r[i]) * (x1 - x0)))


def softmax_comparison(T, dev, stream, flush, ws, rank):
    """The pages' speed comparison re-measured on this GPU: the states path
    (tsa_prefill, tsa_decode_step) against exact causal softmax attention on
    the library's fastest backend (fixed_state_recurrence_phi_b300.softmax_
    baseline), prefill over a sweep of N on the 8-head d_k=16, d_v=64, n=3
    shape in fp32 and bf16, and one KV-cache decode step on the B=64, H=16
    decode shape (bf16) over a sweep of context lengths. Both sides are timed
    the same way: eager calls on the same stream, CUDA events around each
    call, median; the L2 is flushed before each prefill call; the decode
    steps stream caches and rotated state sets larger than L2."""
    import torch
    from fixed_state_recurrence_phi_b300 import softmax_baseline as SB
    from fixed_state_recurrence_phi_b300.inputs import torch_qkv

    def median_ms(fn, reps, do_flush):
        fn()
        torch.cuda.synchronize()
        evs = []
        warm_host()
        for i in range(reps):
            if do_flush:
                flush.fill_(float(i))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn(i)
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        return statistics.median([a.elapsed_time(b) for a, b in evs])

    def fastest(make_call, reps, do_flush):
        """(name, ms): every backend and form that takes the inputs, timed by
        median_ms like the states path; the fastest is the comparator."""
        best = None
        for c in SB.candidates(dev):
            try:
                fn = make_call(c)
                with warnings.catch_warnings():   # refusals are expected here
                    warnings.simplefilter("ignore", UserWarning)
                    fn(0)
                torch.cuda.synchronize()
            except RuntimeError:
                continue
            ms = median_ms(fn, reps, do_flush)
            del fn
            if best is None or ms < best[1]:
                best = (c.name, ms)
        if best is None:
            raise RuntimeError("no softmax attention backend takes the comparison's inputs")
        return best

    r4 = lambda x: None if x is None else float(f"{x:.4g}")
    B, H, d, dv, n = 1, 8, 16, 64, 3
    prefill = []
    for dtype in ("f32", "bf16"):
        cfg = T.Config(B, H, d, dv, n, dtype)
        ours, soft, names = [], [], []
        for N in SOFTMAX_PREFILL_N:
            q, k, v = torch_qkv(B, H, N, d, dv, dtype, rank_seed(21, rank), 0, dev)
            out = torch.empty((B, H, N, dv), dtype=q.dtype, device=dev)
            st = T.new_states(cfg, dev)
            reps = 10 if N <= 16384 else 5
            ours.append(median_ms(lambda i=0: T.prefill(cfg, N, q, k, v, out, st, stream=stream), reps, True))

            def prefill_call(c, q=q, k=k, v=v):
                qq, kk = c.keys(q, dv), c.keys(k, dv)
                return lambda i=0: c.prefill(qq, kk, v)

            name, ms_soft = fastest(prefill_call, reps, True)   # the fastest exact softmax at this N
            names.append(name)
            soft.append(ms_soft)
            del q, k, v, out, st
        T.sync_status(stream)
        fit = [j for j, N in enumerate(SOFTMAX_PREFILL_N) if N >= SOFTMAX_FIT_MIN_N]
        sel = lambda xs: [xs[j] for j in fit]
        ns_fit = sel(SOFTMAX_PREFILL_N)
        prefill.append({
            "dtype": dtype, "backend": names,
            "N": list(SOFTMAX_PREFILL_N), "ours_ms": [r4(x) for x in ours], "softmax_ms": [r4(x) for x in soft],
            "exponent": {"ours": r4(loglog_slope(ns_fit, sel(ours))),
                         "softmax": r4(loglog_slope(ns_fit, sel(soft))), "fit": f"N >= {SOFTMAX_FIT_MIN_N}"},
            "crossover_N": r4(crossover_n(SOFTMAX_PREFILL_N, ours, soft)),
            "speedup": {str(N): r4(s_ / o_) for N, o_, s_ in zip(SOFTMAX_PREFILL_N, ours, soft)
                        if N in (8192, 65536)},
        })
        torch.cuda.empty_cache()

    def decode_sweep(Bd, Hd, rotate):
        """One decode step of B x H heads (bf16) at each context length: the
        states path (rotating over `rotate` state sets) against softmax with
        a KV cache of N tokens."""
        dcfg = T.Config(Bd, Hd, d, dv, n, "bf16")
        tq, tk, tv = (x.permute(2, 0, 1, 3).contiguous()
                      for x in torch_qkv(Bd, Hd, 64, d, dv, "bf16", rank_seed(23, rank), 1, dev))
        tout = torch.empty((Bd, Hd, dv), dtype=tq.dtype, device=dev)
        sts = [T.new_states(dcfg, dev) for _ in range(rotate)]
        ours_us = 1e3 * median_ms(
            lambda i=0: T.decode_step(dcfg, tq[i % 64], tk[i % 64], tv[i % 64], tout, sts[i % rotate],
                                      stream=stream),
            64, False)
        T.sync_status(stream)
        del sts
        soft_us, dnames = [], []
        for N in SOFTMAX_DECODE_N:
            q, k, v = torch_qkv(Bd, Hd, N, d, dv, "bf16", rank_seed(24, rank), 0, dev)
            k1, v1 = k[:, :, -1].contiguous(), v[:, :, -1].contiguous()

            def decode_call(c, q=q, k=k, v=v, N=N, k1=k1, v1=v1):
                kc, vc = c.cache(k, v)
                # the new token's q in the comparator's form, made before the timed calls
                q1 = c.keys(q[:, :, -1], dv).contiguous()
                return lambda i=0: c.decode_step(q1, k1, v1, kc, vc, N - 1)

            name, ms_soft = fastest(decode_call, 20, False)
            dnames.append(name)
            soft_us.append(1e3 * ms_soft)
            del q, k, v, k1, v1
            torch.cuda.empty_cache()
        return {
            "dtype": "bf16", "workload": f"B{Bd}_H{Hd}_d{d}_dv{dv}", "backend": dnames,
            "N": list(SOFTMAX_DECODE_N),
            "ours_us": r4(ours_us), "softmax_us": [r4(x) for x in soft_us],
            "exponent_softmax": r4(loglog_slope(SOFTMAX_DECODE_N, soft_us)),
            "speedup": {str(N): r4(s_ / ours_us) for N, s_ in zip(SOFTMAX_DECODE_N, soft_us)},
            "ours_timing": f"eager decode steps, {rotate} rotated state sets",
        }

    # the decode workload's batch (B=64, H=16; states and caches exceed L2) and
    # one sequence of the prefill shape (B=1, H=8: the per-token latency the
    # pages quote; its caches up to 84 MB may stay in L2 between steps, as
    # its states do)
    decode = decode_sweep(64, 16, DECODE_ROTATE)
    decode_one = decode_sweep(1, 8, DECODE_ROTATE)
    return {"what": "exact causal softmax (weights exp(q.k), scale 1) on the library's fastest attention "
                    "backend at each N (cuDNN, flash or memory-efficient, q and k unpadded or zero-padded to "
                    "d_v) against the states path; eager calls, CUDA events, median per call",
            "prefill": prefill, "decode": decode, "decode_one_sequence": decode_one}


def _profile_traffic():
    """DRAM traffic per launch from the committed ncu summary, if present and
    current (profiles/traffic.json, written from a capture of this build)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            return json.load(f)
    except Exception:
        return {}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "prefill", "decode", "order4", "wide", "orders", "softmax"],
                    default="all",
                    help="run one part (profiling captures on small cases)")
    ap.add_argument("--tc-n", type=int, default=0,
                    help="sequence length of the order4/wide workloads (default: theirs)")
    ap.add_argument("--decode-prefill-n", type=int, default=DECODE["N"],
                    help="tokens prefilled before the decode steps (default 65536)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
