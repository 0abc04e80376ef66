"""Benchmark of the KDA forward on GB300 (one JSON line on rank 0).

Step = one chunked KDA forward (gate + cumsum, causal scores, triangular solve,
WY terms, state scan, output) over the dense bf16 workload B=4, T=4096, H=64,
K=V=128, C=64 (safe gate, lower_bound -5), inputs resident in HBM.  The
workload's inputs (1.34 GB) are larger than L2, so consecutive steps re-read
them from HBM.  A decode measurement (512 one-token sequences, H=32,
K=V=128, FP32 states updated in place) is reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own copy of the workload on its own
GPU (independent batches, no collective on the data path: weak scaling); the
timed region is bracketed by barriers, the time is the max over ranks and the
value counts the head-tokens of all ranks.  ``--impl reference`` times the
float64 CPU oracle (the reference arm of this build) on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA fwd tokens/s (B*T*H) and TFLOP/s, % of GB300 roofline; decode steps/s"
WORKLOAD = "dense_bf16_b4_t4096_h64_d128"
UNIT = "head-tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def algorithmic_flops_per_head_token(K, V, C):
    """6KV + 2K(C+16) + CK + CV + (C+1)V + C^2/3: state read-outs and updates, causal
    scores on 16-row sub-blocks, WY terms, output (lower-triangular counts)."""
    return 6 * K * V + 2 * K * (C + 16) + C * K + C * V + (C + 1) * V + C * C / 3.0


# DRAM bytes (read + write) per chunk_fused_kernel launch on the default workload, from one ncu
# capture (--set full) of that launch on that workload, of the kernel whose code digest
# (kernel_code_digest) starts with `source_sha256`.  Reported only while the source is
# unchanged; a changed kernel reports null until it is captured again.
FUSED_TRAFFIC = {"source_sha256": "97754695245fcd55", "workload": "dense_bf16_b4_t4096_h64_d128",
                 "bytes": 1078.205e6 + 252.189e6}


def kernel_code_digest(path):
    """sha256 of a CUDA source with // comments, surrounding blanks and empty lines removed,
    so only code changes alter it."""
    import hashlib
    import re

    with open(path) as f:
        lines = [re.sub(r"//.*$", "", ln).strip() for ln in f]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def fused_traffic_bytes(workload):
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "chunked_kda_gb300", "csrc",
                       "chunk_fused.cu")
    try:
        digest = kernel_code_digest(src)
    except OSError:
        return None
    if workload != FUSED_TRAFFIC["workload"] or not digest.startswith(FUSED_TRAFFIC["source_sha256"]):
        return None
    return FUSED_TRAFFIC["bytes"]


def algorithmic_bytes_per_head_token(K, V, in_bytes=2, g_bytes=2):
    """q, k, g (K each), v (V), beta in; o (V) out."""
    return in_bytes * (2 * K + V) + g_bytes * K + in_bytes + in_bytes * V


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples in a background process."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        rows = self.samples
        if self.window:
            inside = [r for r in rows if self.window[0] - 0.05 <= r[0] <= self.window[1] + 0.05]
            if inside:
                rows = inside
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for _, f in rows:
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_seconds, local_units, world, device=None):
    """Max time and summed work over ranks (identity at world size 1)."""
    if world == 1:
        return local_seconds, local_units
    import torch
    import torch.distributed as dist

    t = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def oracle_sample(w, n_units, nthreads, seed=0):
    """Time the float64 oracle on n_units (sequence, head) units of workload w.
    Returns (head-tokens, wall seconds)."""
    import numpy as np

    import oracle

    r = np.random.default_rng(seed)
    units = [(int(r.integers(w.B)), int(r.integers(w.H))) for _ in range(n_units)]
    # slice the sampled units out first so the conversion to float64 stays small
    heads = sorted({h for _, h in units})
    rows = sorted({b for b, _ in units})
    pick = {name: getattr(w, name)[rows][:, :, heads].cpu() for name in ("q", "k", "v", "g", "beta")}
    local = [(rows.index(b), heads.index(h)) for b, h in units]
    al = w.A_log[heads].cpu() if w.A_log is not None else None
    db = w.dt_bias[heads].cpu() if w.dt_bias is not None else None
    t0 = time.perf_counter()
    oracle.forward(pick["q"], pick["k"], pick["v"], pick["g"], pick["beta"], al, db, w.mode,
                   w.lower_bound, None, None, units=local, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return n_units * w.T, dt


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, world, rank):
    """The reference arm: the float64 CPU oracle, timed on the host cores."""
    if rank != 0:
        return
    import torch

    import oracle
    from chunked_kda_gb300 import workloads

    oracle.build()
    w = workloads.make(WORKLOAD, device="cuda" if torch.cuda.is_available() else "cpu")
    cores = host_cores()
    n_units = cores  # one (sequence, head) unit per core per step
    for _ in range(args.warmup):
        oracle_sample(w, max(1, cores // 4), cores, seed=99)
    tot_tokens, tot_s = 0, 0.0
    for s in range(args.steps):
        tok, dt = oracle_sample(w, n_units, cores, seed=s)
        tot_tokens += tok  # head-tokens: each unit is one head of one sequence
        tot_s += dt
    value = tot_tokens / tot_s
    sample = f"{n_units} random (sequence, head) units of {WORKLOAD} per step ({w.T} tokens each)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "B": 4, "T": 4096, "H": 64, "K": 128,
                                        "V": 128, "chunk_size": 64, "sampled": True},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import torch

    import chunked_kda_gb300 as kda
    from chunked_kda_gb300 import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    barrier = (lambda: torch.distributed.barrier()) if world > 1 else (lambda: None)
    kda.load_library()
    peaks, peak_src = load_peaks()

    w = workloads.make(args.workload, device=dev)
    B, T, H, K, V, C = w.B, w.T, w.H, w.K, w.V, w.chunk_size
    stream = torch.cuda.current_stream()
    o = torch.empty((B, T, H, V), device=dev, dtype=w.q.dtype)  # o in the dtype of q, k, v
    n_ws = 0 if w.cu_seqlens is None else w.n_seqs
    ws_bytes = kda.kda_chunk_workspace_bytes(w.q.dtype, B, T, H, K, V, C, n_ws, w.mode)
    ws = torch.empty(max(ws_bytes, 1), device=dev, dtype=torch.uint8)
    # the workload's own initial state and packing; a final state is written when an initial
    # state is given (the dense B4 T4096 H64 case is the output-only forward)
    S_fin = None if w.initial_state is None else torch.empty_like(w.initial_state)
    # kernels one call launches (the library's own count: 1 fused, 2 with its split schedule
    # for dense batches of a little more than one wave of units, 6 stage-by-stage)
    n_launch = kda.kda_chunk_fwd_launches(w.q.dtype, B, T, H, K, V, C, n_ws, w.mode, o.dtype)

    def step():
        kda.kda_chunk_fwd(w.q, w.k, w.v, w.g, w.beta, w.A_log, w.dt_bias, w.mode, w.lower_bound,
                          w.initial_state, False, w.cu_seqlens, C, o=o, workspace=ws,
                          final_state=S_fin)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier()
    sampler.mark(wall0, wall1)
    local_s = ev0.elapsed_time(ev1) / 1e3
    head_tokens = w.head_tokens()  # valid tokens x heads (packed: the sum of the lengths)
    t_max, units_all = aggregate(local_s, head_tokens * args.steps, world, dev)
    ms_per_step = 1e3 * t_max / args.steps

    if args.chunk_only:
        sampler.stop()
        if rank == 0:
            state_bytes = 0 if w.initial_state is None else 2 * w.initial_state.numel() * 4
            nb = (algorithmic_bytes_per_head_token(K, V, w.q.element_size(), w.g.element_size())
                  * head_tokens + state_bytes)
            print(json.dumps({"workload": args.workload, "ms_per_step": ms_per_step,
                              "head_tokens_per_s": units_all / t_max,
                              "path": path_of(w),
                              "launches_per_call": n_launch,
                              "algorithmic_gbs": nb / (ms_per_step / 1e3) / 1e9,
                              "frac_of_hbm": nb / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"]}),
                  flush=True)
        return

    # end to end through the public API: pinned host inputs -> device, forward, o -> host, every
    # step.  Two device input / output sets and three streams let the copies of one step
    # overlap the forward of another: step i copies into set i % 2 once the forward of step
    # i - 2 has read it, and the forward writes o into set i % 2 once that o has been copied out.
    names = ("q", "k", "v", "g", "beta")
    host = {n: getattr(w, n).cpu().pin_memory() for n in names}
    dbufs = [{n: torch.empty_like(getattr(w, n)) for n in names} for _ in range(2)]
    obufs = [torch.empty_like(o) for _ in range(2)]
    o_host = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o_host.numel() * o_host.element_size()
    s_in, s_fw, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_fw = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps_run(n_steps):
        for i in range(n_steps):
            b = i % 2
            if i >= 2:
                s_in.wait_event(ev_fw[b])
            with torch.cuda.stream(s_in):
                for n in names:
                    dbufs[b][n].copy_(host[n], non_blocking=True)
            ev_in[b].record(s_in)
            s_fw.wait_event(ev_in[b])
            if i >= 2:
                s_fw.wait_event(ev_out[b])
            d = dbufs[b]
            kda.kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.A_log, w.dt_bias,
                              w.mode, w.lower_bound, w.initial_state, False, w.cu_seqlens, C,
                              o=obufs[b], workspace=ws, final_state=S_fin, stream=s_fw)
            ev_fw[b].record(s_fw)
            s_out.wait_event(ev_fw[b])
            with torch.cuda.stream(s_out):
                o_host.copy_(obufs[b], non_blocking=True)
            ev_out[b].record(s_out)

    e2e_steps_run(2)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 10))
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    e2e_steps_run(e2e_steps)
    s_out.wait_event(ev_fw[(e2e_steps - 1) % 2])
    e1.record(s_out)  # after the last copy out, which follows every forward and copy in
    torch.cuda.synchronize()
    e2e_s, _ = aggregate(e0.elapsed_time(e1) / 1e3, 0, world, dev)
    e2e_value = world * head_tokens * e2e_steps / e2e_s
    del host, dbufs, obufs

    dec_s, dec_bytes = time_decode(kda, workloads, dev, stream, 512, 64)
    sampler.stop()
    # the per-configuration lines at one GPU only (a multi-rank run times the headline step)
    per_config = (None if args.no_per_config or world > 1
                  else per_config_lines(kda, workloads, dev, peaks, 10))
    gate = None if args.no_per_config or world > 1 else time_gate(kda, workloads, dev, peaks, 10)

    if rank != 0:
        return
    flops = algorithmic_flops_per_head_token(K, V, C) * head_tokens
    nbytes = algorithmic_bytes_per_head_token(K, V) * head_tokens
    t_step = ms_per_step / 1e3
    achieved_gbs = nbytes / t_step / 1e9
    value = units_all / t_max
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": B, "T": T, "H": H, "K": K, "V": V, "chunk_size": C,
                   "gate": "safe, lower_bound -5", "initial_state": None,
                   "output_final_state": False, "l2": "inputs (1.34 GB) larger than L2",
                   "parallelism": f"replicas x{world}"},
        "tflops": flops / t_step / 1e12,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"],
                     "traffic": fused_traffic_bytes(args.workload),
                     "peak_source": peak_src,
                     "kernel": "chunk_fused_kernel (one launch per kda_chunk_fwd call)" if n_launch == 1
                               else f"chunk_fused_kernel ({n_launch} launches per kda_chunk_fwd call, "
                                    f"timed together)"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "pipelined": "two device buffer sets, copy-in / forward / copy-out streams"},
        "gpu_launches": args.steps * n_launch,
        "decode": {"steps_per_s": 1.0 / dec_s, "ms_per_step": 1e3 * dec_s,
                   "achieved_gbs": dec_bytes / dec_s / 1e9,
                   "frac": dec_bytes / dec_s / 1e9 / peaks["hbm_gbs"],
                   "workload": "512 one-token sequences, H=32, K=V=128, bf16, states in place"},
        "clocks": sampler.summary(),
    }
    if per_config is not None:
        line["per_config"] = per_config
    if gate is not None:
        line["gate"] = gate
    if not args.no_cpu_baseline:
        cores = host_cores()
        tok, dt = oracle_sample(w, 2 * cores, cores, seed=1234)
        tok1, dt1 = oracle_sample(w, 1, 1, seed=1235)
        line["cpu_baseline"] = {"value": tok / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{2 * cores} random (sequence, head) units of {args.workload} "
                                          f"({w.T} tokens each), float64, one OpenMP thread "
                                          f"per unit",
                                "single_core": {"value": tok1 / dt1, "unit": UNIT,
                                                "sample": "one (sequence, head) unit, one thread"}}
    print(json.dumps(line), flush=True)


# every configured chunked workload, timed beside the headline one (the headline workload is
# the line's own value); decode is reported under "decode"
PER_CONFIG = (
    ("config 0", "tiny_fp32_b1_t128_h2_d64"),
    ("config 1", "dense_bf16_b4_t2048_h16_d128"),
    ("config 2", "varlen_bf16_n16_cap20480_h32_d128_c32"),
    ("config 3a", "dense_bf16_b1_t8192_h96_d128"),
    ("config 3b", "dense_bf16_b4_t4096_h64_d128"),
    ("config 4b", "dense_bf16_b8_t2048_h32_d256"),
    ("config 3b, non-safe gate", "dense_bf16_b4_t4096_h64_d128_nonsafe"),
    ("config 4b, non-safe gate", "dense_bf16_b8_t2048_h32_d256_nonsafe"),
)


def roofline_of(w, seconds, peaks):
    """Algorithmic bytes and flops of one forward of workload w and the fraction of the GB300
    roofline it reaches in `seconds`: the slower of the HBM time for the bytes and the bf16
    tensor time for the flops, over the measured time."""
    K, V, C = w.K, w.V, w.chunk_size
    ht = w.head_tokens()
    state_bytes = 0 if w.initial_state is None else 2 * w.initial_state.numel() * 4
    nbytes = algorithmic_bytes_per_head_token(K, V, w.q.element_size(), w.g.element_size()) * ht + state_bytes
    flops = algorithmic_flops_per_head_token(K, V, C) * ht
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_mma = flops / (peaks["bf16_tflops"] * 1e12)
    return {"bytes": nbytes, "flops": flops, "achieved_gbs": nbytes / seconds / 1e9,
            "tflops": flops / seconds / 1e12, "bound": "hbm" if t_hbm >= t_mma else "tensor",
            "frac": max(t_hbm, t_mma) / seconds}


def time_chunk_workload(kda, w, dev, steps, warmup, flush=None):
    """Median CUDA-event time of one kda_chunk_fwd call on workload w (inputs resident); with
    `flush` (a device buffer larger than L2) L2 is overwritten before every timed call."""
    import torch

    B, T, H, K, V, C = w.B, w.T, w.H, w.K, w.V, w.chunk_size
    o = torch.empty((B, T, H, V), device=dev, dtype=w.q.dtype)
    n_ws = 0 if w.cu_seqlens is None else w.n_seqs
    ws_bytes = kda.kda_chunk_workspace_bytes(w.q.dtype, B, T, H, K, V, C, n_ws, w.mode)
    ws = torch.empty(max(ws_bytes, 1), device=dev, dtype=torch.uint8)
    S_fin = None if w.initial_state is None else torch.empty_like(w.initial_state)
    n_launch = kda.kda_chunk_fwd_launches(w.q.dtype, B, T, H, K, V, C, n_ws, w.mode, o.dtype)

    def step():
        kda.kda_chunk_fwd(w.q, w.k, w.v, w.g, w.beta, w.A_log, w.dt_bias, w.mode, w.lower_bound,
                          w.initial_state, False, w.cu_seqlens, C, o=o, workspace=ws,
                          final_state=S_fin)

    for _ in range(max(warmup, 3)):
        step()
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(steps):
        if flush is not None:
            flush.add_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    return statistics.median(times), n_launch


def path_of(w):
    """The kernels kda_chunk_fwd runs for workload w (the library's dispatch rule): the fused
    kernel for bf16 K = V = 128, the two-pass kernels for bf16 K in {128, 256} with V a multiple
    of 128 otherwise, the stage-by-stage kernels for the rest."""
    import torch

    if w.q.dtype == torch.bfloat16 and w.K == w.V == 128:
        return "fused"
    if w.q.dtype == torch.bfloat16 and w.K in (128, 256) and w.V >= 128 and w.V % 128 == 0:
        return "two-pass"
    return "stage-by-stage"


def per_config_lines(kda, workloads, dev, peaks, steps):
    """One entry per configured workload: median time per forward (L2 flushed before each),
    head-tokens/s, TFLOP/s and the roofline fraction."""
    import torch

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, device=dev, dtype=torch.float32)
    out = []
    for label, name in PER_CONFIG:
        w = workloads.make(name, device=dev)
        sec, n_launch = time_chunk_workload(kda, w, dev, steps, 3, flush)
        r = roofline_of(w, sec, peaks)
        out.append({"config": label, "workload": name, "ms_per_step": 1e3 * sec,
                    "head_tokens_per_s": w.head_tokens() / sec, "tflops": r["tflops"],
                    "achieved_gbs": r["achieved_gbs"], "roofline_bound": r["bound"],
                    "roofline_frac": r["frac"], "launches_per_call": n_launch,
                    "path": path_of(w), "dtype": str(w.q.dtype).replace("torch.", "")})
        del w
        torch.cuda.empty_cache()
    del flush
    return out


def time_gate(kda, workloads, dev, peaks, steps):
    """kda_gate_fwd alone on the headline workload's gate (bf16 g, safe activation, 64-token
    chunk-local log2 cumsum, float32 out), inputs resident; L2 flushed before each call.
    Algorithmic bytes: g in (2 B) and the float32 cumsum out (4 B) per element."""
    import torch

    w = workloads.make(WORKLOAD, device=dev)
    out = torch.empty(w.g.shape, device=dev, dtype=torch.float32)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, device=dev, dtype=torch.float32)

    def call():
        kda.kda_gate_fwd(w.g, w.A_log, w.dt_bias, w.mode, w.lower_bound, None, w.chunk_size, out=out)

    for _ in range(3):
        call()
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(steps):
        flush.add_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    sec = statistics.median(times)
    nbytes = w.g.numel() * (w.g.element_size() + 4)
    res = {"workload": f"gate of {WORKLOAD} (bf16 g, safe, chunk 64, float32 out)",
           "ms": 1e3 * sec, "achieved_gbs": nbytes / sec / 1e9,
           "frac": nbytes / sec / 1e9 / peaks["hbm_gbs"], "bytes_per_element": 6}
    del w, out, flush
    torch.cuda.empty_cache()
    return res


def time_decode(kda, workloads, dev, stream, n_dec, d_steps):
    """Decode: n_dec packed one-token sequences, H=32, K=V=128, FP32 states in place; returns
    (seconds per step, algorithmic bytes per step)."""
    import torch

    Hd = 32
    S = workloads.decode_state(n_dec, Hd, device=dev)
    cu = workloads.decode_cu_seqlens(n_dec, device=dev)
    pool = [workloads.decode_step(i, n_dec, Hd, device=dev) for i in range(4)]
    od = torch.empty((1, n_dec, Hd, 128), device=dev, dtype=torch.bfloat16)

    def dstep(i):
        p = pool[i % len(pool)]
        kda.kda_recurrent_fwd(p.q, p.k, p.v, p.gate, p.beta, S, True, cu, o=od, final_state=S)

    for i in range(3):
        dstep(i)
    torch.cuda.synchronize()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for i in range(d_steps):
        dstep(i)
    d1.record(stream)
    torch.cuda.synchronize()
    dec_s = d0.elapsed_time(d1) / 1e3 / d_steps
    dec_bytes = 2 * S.numel() * 4 + n_dec * Hd * (3 * 128 * 2 + 128 * 4 + 2 + 128 * 2)
    return dec_s, dec_bytes


def run_gate_only(args, local):
    """kda_gate_fwd alone (the "gate" object of the full line), for profiling: one JSON line."""
    import torch

    import chunked_kda_gb300 as kda
    from chunked_kda_gb300 import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kda.load_library()
    peaks, _ = load_peaks()
    print(json.dumps(time_gate(kda, workloads, dev, peaks, args.steps)), flush=True)


def run_decode_only(args, local):
    """The decode step alone (kda_recurrent_fwd), for profiling: one JSON line."""
    import torch

    import chunked_kda_gb300 as kda
    from chunked_kda_gb300 import workloads

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kda.load_library()
    peaks, _ = load_peaks()
    dec_s, dec_bytes = time_decode(kda, workloads, dev, torch.cuda.current_stream(),
                                   args.decode_seqs, args.steps)
    print(json.dumps({"decode_seqs": args.decode_seqs, "heads": 32, "ms_per_step": 1e3 * dec_s,
                      "achieved_gbs": dec_bytes / dec_s / 1e9,
                      "frac_of_hbm": dec_bytes / dec_s / 1e9 / peaks["hbm_gbs"]}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload name (chunked_kda_gb300.workloads, dense or packed); default is "
                         "the one the metric is quoted on")
    ap.add_argument("--chunk-only", action="store_true",
                    help="time the chunked forward only (no e2e, decode or CPU leg); for profiling")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration timings that follow the headline step")
    ap.add_argument("--decode-only", action="store_true",
                    help="time the decode step only (kda_recurrent_fwd); for profiling")
    ap.add_argument("--gate-only", action="store_true",
                    help="time kda_gate_fwd alone on the headline workload's gate; for profiling")
    ap.add_argument("--decode-seqs", type=int, default=512,
                    help="one-token sequences of the decode step (32 heads each)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.decode_only:
        run_decode_only(args, local)
        return
    if args.gate_only:
        run_gate_only(args, local)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
