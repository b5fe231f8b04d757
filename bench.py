"""Benchmark of the STOF masked-attention hot path on GB300.

One step = the whole hot path over one batch of synthetic input already
resident in HBM: encode the dense mask into the two-level format, sync the
tile counts, select the kernel analytically, run the masked MHA forward.
Metric: effective TFLOP/s = 4 * d * (valid mask elements over all heads) /
step time.  The default workload is the 16k one (B=1, H=32, L=16384,
d=128, bf16, per-head causal AND Bernoulli(0.1) masks with the diagonal
forced), the configuration the throughput target is quoted on.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle, same metric

Prints one JSON line (rank 0).  Under torchrun every rank runs an
independent replica of the workload on its own GPU (the path needs no
exchange step); value = units of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_mask_transformer_gb300 import synth  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "masked-MHA fwd effective TFLOP/s (valid elems) and % of GB300 tensor peak"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


HOST_CODE_MARK = b"// ---------------------------------------------------------------- host side"


def _code_only(text: bytes) -> bytes:
    """C++ source without its comments and blank-line or trailing-space
    differences (string literals in these files hold no comment markers)."""
    text = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)
    text = re.sub(rb"//[^\n]*", b"", text)
    return b"\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash() -> str:
    """Hash of the block-wise kernel's device code, comments left out:
    blockwise.cu up to its host-side launch code, and the headers of device
    code it includes."""
    h = hashlib.sha256()
    for f in ("blockwise.cu", "blockwise_common.cuh", "sm100_ptx.cuh"):
        with open(os.path.join(ROOT, "sparse_mask_transformer_gb300", "csrc", f), "rb") as fh:
            text = fh.read()
        h.update(_code_only(text.split(HOST_CODE_MARK)[0] if f == "blockwise.cu" else text))
    return h.hexdigest()[:16]


def profiled(workload: str, key: str):
    """A figure (`key: value` line) of the committed ncu summary of the
    block-wise kernel on this workload, if it was taken on the current
    kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"blockwise_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    src = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    val = re.search(rf"{key}:\s*([0-9.eE+]+)", text)
    if not src or not val or src.group(1) != kernel_source_hash():
        return None
    return float(val.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling around the timed region.  The
    caller keeps the GPU under the step's own load for LEAD_S before and
    TAIL_S after the timed steps, so that every sample (one per 100 ms) sees
    the clocks of the loaded GPU, the timed region included."""
    LEAD_S = 0.4
    TAIL_S = 0.2
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, enabled: bool = True):
        self.index = index
        self.proc = None
        if not enabled:  # profiling runs: no sampler, no untimed lead and tail steps
            self.LEAD_S = self.TAIL_S = 0.0
        self.enabled = enabled

    def __enter__(self):
        if not self.enabled:
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


L2_BYTES = 129 * 2 ** 20  # GB300 L2


def l2_note(mask_bytes: int, qkv_bytes: int) -> str:
    """Whether a step's inputs exceed L2 (no flush needed between timed
    steps) or fit in it (not flushed: timed warm)."""
    sizes = "mask %.2f GB, Q/K/V %.2f GB" % (mask_bytes / 1e9, qkv_bytes / 1e9)
    if mask_bytes + qkv_bytes > L2_BYTES:
        return f"inputs larger than L2 ({sizes})"
    return f"inputs fit in L2 ({sizes}); not flushed between steps, so timed with a warm L2"


def run_for(step, seconds: float) -> int:
    """Untimed steps for about `seconds` of wall time; returns how many."""
    n, t_end = 0, time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        step()
        n += 1
    return n


def dist_setup(n_gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if _cuda_ok() else "gloo"
        dist.init_process_group(backend)
        return rank, world, local, dist
    return rank, world, local, None


def _cuda_ok() -> bool:
    import torch
    return torch.cuda.is_available()


def max_over_ranks(x: float, dist, device) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, dist, device) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- inputs

def device_inputs(w: synth.Workload, device):
    import torch
    from sparse_mask_transformer_gb300 import stof
    if w.pattern == "causal_bernoulli":
        mask = torch.empty(w.n_masks, w.L, w.L, dtype=torch.uint8, device=device)
        stof.stof_synth_causal_bernoulli_mask(mask, w.n_masks, w.L, w.seed,
                                              synth.bernoulli_threshold(synth.BERNOULLI_P))
    else:
        mask = torch.from_numpy(synth.make_mask(w)).to(device)
    q, k, v = (t.to(device) for t in synth.make_qkv(w.B, w.H, w.L, w.d, w.dtype, seed=w.seed))
    return mask, q, k, v


def heads_per_mask(w: synth.Workload) -> float:
    return w.B * w.H / w.n_masks


# ---------------------------------------------------------------- GPU arm

def run_gpu(args, w: synth.Workload):
    import torch
    from sparse_mask_transformer_gb300 import build, stof

    rank, world, local, dist = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    build.build()
    stof.load_library()
    peaks, peak_src = load_peaks()

    mask, q, k, v = device_inputs(w, device)
    o = torch.empty_like(q)
    bm = bn = 128
    ws = torch.empty(stof.stof_encode_workspace_bytes(w.n_masks, w.L, w.L, bm, bn), dtype=torch.uint8,
                     device=device)
    scale = 1.0 / math.sqrt(w.d)
    stream = torch.cuda.current_stream(device)
    fmt = stof.stof_format()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]

    def step(i=None):
        stof.stof_encode_mask(mask, bm, bn, ws, fmt)
        stof.stof_format_sync(fmt)                   # counts to host: feeds the selector
        if i is not None:
            ev[i][0].record(stream)
        stof.stof_mha_fwd(q, k, v, fmt, scale, w.stride_b, w.stride_h, stof.STOF_KERNEL_AUTO, o)
        if i is not None:
            ev[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    density = fmt.nnz / (w.n_masks * w.L * w.L)
    plan = stof.stof_mha_plan(fmt, w.B, w.H, w.L, w.d, stof.STOF_KERNEL_AUTO)
    chosen = plan.kernel
    valid = fmt.nnz * heads_per_mask(w)
    tiles = (fmt.n_full + fmt.n_part) * heads_per_mask(w)

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local, enabled=not args.no_clocks) as clk:
        run_for(step, clk.LEAD_S)  # untimed: the clocks are sampled under load
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        start.record(stream)
        for i in range(args.steps):
            step(i)
        end.record(stream)
        torch.cuda.synchronize()
        run_for(step, clk.TAIL_S)
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    step_ms_local = start.elapsed_time(end) / args.steps
    step_ms = max_over_ranks(step_ms_local, dist, device)
    mha_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    mha_ms = max_over_ranks(mha_ms, dist, device)
    clocks = clk.summary()

    flops_eff = 4.0 * w.d * valid
    flops_tile = 4.0 * w.d * 128 * 128 * tiles
    total_units = sum_over_ranks(flops_eff, dist, device)
    value = total_units / (step_ms * 1e-3) / 1e12

    # end to end through the same public API with host buffers
    e2e = None if args.no_e2e else run_e2e(args, w, mask, q, k, v, ws, fmt, scale, stream, device, dist)
    # the same step from the bit-packed mask (stof_encode_mask_bits)
    bitmask = None if args.no_bitmask else run_bitmask(args, w, mask, q, k, v, ws, scale, stream, device, dist)
    # the same step from the mask's rule, where the workload has one
    rules = None if args.no_bitmask else run_rules(args, w, q, k, v, ws, scale, stream, device, dist)
    # kernel-only times of both kernels and the encoder on all five workloads
    workloads = None
    if not args.no_workloads and not args.heads:
        workloads = run_workload_records(args, device, peaks, big=(w, mask, q, k, v))

    kern_name = "blockwise" if chosen == stof.STOF_KERNEL_BLOCKWISE else "rowwise"
    if chosen == stof.STOF_KERNEL_BLOCKWISE:
        achieved = flops_tile / (mha_ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        roofline = {"bound": "tensor", "kernel": "blockwise_kernel", "achieved": round(achieved, 2),
                    "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "traffic": profiled(w.name, "traffic_bytes_per_launch"),
                    "tensor_pipe_active_pct": profiled(w.name, "tensor_pipe_active_pct_of_active_cycles"),
                    "peak_source": f"{peak_src} bf16 burst",
                    "algorithmic": "4*d*128*128 FLOPs per listed outer tile per head"}
    else:
        bytes_alg = 4 * w.B * w.H * w.L * w.d * 2
        achieved = bytes_alg / (mha_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roofline = {"bound": "hbm", "kernel": "rowwise_kernel", "achieved": round(achieved, 1), "peak": peak,
                    "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                    "peak_source": f"{peak_src} copy", "algorithmic": "Q+K+V+O bytes per launch"}

    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "value_definition": ("4*d*(valid mask elements over all heads) / step time, one step being every row "
                             "of the hot path on one batch: encode the dense mask, sync the tile counts, "
                             "select the kernel, stof_mha_fwd.  The same metric over the stof_mha_fwd call "
                             "alone is breakdown.effective_tflops_mha_only; kernel-only times of both kernels "
                             "on all five workloads are under workloads"),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded masks and N(0,1) Q/K/V)",
        "config": {"workload": w.name + (f"(H={w.H})" if args.heads else ""), "B": w.B, "H": w.H, "L": w.L,
                   "d": w.d, "mask": w.describe,
                   "outer_tile": "128x128", "kernel": kern_name, "parallelism": f"replicas x{world}",
                   "l2": l2_note(w.mask_bytes, 3 * q.numel() * 2)},
        "breakdown": {"mha_ms": round(mha_ms, 4), "encode_and_sync_ms": round(step_ms - mha_ms, 4),
                      "effective_tflops_mha_only": round(flops_eff / (mha_ms * 1e-3) / 1e12, 3),
                      "tile_tflops": round(flops_tile / (mha_ms * 1e-3) / 1e12, 2),
                      "pct_of_tensor_peak_tile": round(100 * flops_tile / (mha_ms * 1e-3) / 1e12 /
                                                       peaks["bf16_tflops"], 2),
                      "pct_of_tensor_peak_effective": round(100 * value / peaks["bf16_tflops"], 3),
                      "density": round(density, 6), "nnz_per_mask_set": fmt.nnz,
                      "tiles_full": fmt.n_full, "tiles_partial": fmt.n_part},
        "roofline": roofline,
        "e2e": e2e,
        "bitmask": bitmask,
        "rules": rules,
        "workloads": workloads,
        "build": {"libstof_srchash": build.built_hash(), "sources_srchash": build.source_hash()},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w, args, mask, q, k, v)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# ---------------------------------------------------------------- per-workload records

def graph_ms(fn, n: int, flush=None) -> float:
    """Device time per call of fn() with no host work in it: n calls are
    captured into one CUDA graph and the replay is timed with events.  With
    `flush` (a buffer larger than L2), each call is preceded by a write of
    the buffer and the time of the flushes alone is subtracted, so every
    call starts with a cold L2."""
    import torch

    def timed(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                body()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    fn()
    torch.cuda.synchronize()
    if flush is None:
        return timed(fn)

    def both():
        flush.zero_()
        fn()
    return timed(both) - timed(flush.zero_)


def call_latency(lib_fn, args, reps: int = 15):
    """One C-ABI call on an idle GPU, timed by events recorded just before and
    after it on the stream (host argument checks, launch and kernel), median
    over reps; and the host time of the call alone (median, microseconds)."""
    import torch
    dev_ms, host_us = [], []
    for _ in range(reps):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        t0 = time.perf_counter_ns()
        st = lib_fn(*args)
        t1 = time.perf_counter_ns()
        b.record()
        torch.cuda.synchronize()
        if st != 0:
            raise RuntimeError(f"status {st}")
        dev_ms.append(a.elapsed_time(b))
        host_us.append((t1 - t0) / 1e3)
    return statistics.median(dev_ms), statistics.median(host_us)


def back_to_back(lib_fn, args, n: int = 20):
    """n C-ABI calls issued back to back (no synchronisation between them, as
    a pipeline issues them): event time per call on the stream and host time
    per call (microseconds)."""
    import torch
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    t0 = time.perf_counter_ns()
    for _ in range(n):
        if lib_fn(*args) != 0:
            raise RuntimeError("call failed")
    t1 = time.perf_counter_ns()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n, (t1 - t0) / 1e3 / n


def host_time_us(fn, args) -> float:
    """Host time of one C-ABI call through ctypes (microseconds)."""
    t0 = time.perf_counter_ns()
    fn(*args)
    return (time.perf_counter_ns() - t0) / 1e3


def workload_record(w: synth.Workload, mask, q, k, v, peaks, flush) -> dict:
    """Kernel-only device times of both attention kernels and of the encoder
    on one workload (CUDA-graph replay, warm and with a cold L2), the latency
    of one stof_mha_fwd call through the C ABI, and the analytic selector's
    choice against the measured times."""
    import ctypes

    import torch
    from sparse_mask_transformer_gb300 import stof
    lib = stof.load_library()
    n_masks = mask.shape[0]
    ws = torch.empty(stof.stof_encode_workspace_bytes(n_masks, w.L, w.L, 128, 128), dtype=torch.uint8,
                     device=q.device)
    fmt = stof.stof_format()
    enc = lambda: stof.stof_encode_mask(mask, 128, 128, ws, fmt)  # noqa: E731
    enc_ms = graph_ms(enc, 10)
    enc()
    stof.stof_format_sync(fmt)
    hpm = heads_per_mask(w)
    density = fmt.nnz / (n_masks * w.L * w.L)
    tiles = fmt.n_full + fmt.n_part
    eff_flops = 4.0 * w.d * fmt.nnz * hpm
    tile_flops = 4.0 * w.d * 128 * 128 * tiles * hpm
    n_rows = n_masks * (w.L // 128)
    fmt_bytes = 8 * (n_rows + 1) + 4 * tiles + 2048 * fmt.n_part
    enc_bytes = n_masks * w.L * w.L + fmt_bytes
    o = torch.empty_like(q)
    scale = 1.0 / math.sqrt(w.d)
    chosen = stof.stof_mha_plan(fmt, w.B, w.H, w.L, w.d, stof.STOF_KERNEL_AUTO).kernel
    rec = {"B": w.B, "H": w.H, "L": w.L, "d": w.d, "dtype": w.dtype, "density": round(density, 6),
           "tiles_full": fmt.n_full, "tiles_partial": fmt.n_part,
           "encode": {"ms": round(enc_ms, 5), "gbs": round(enc_bytes / (enc_ms * 1e-3) / 1e9, 1),
                      "frac_hbm": round(enc_bytes / (enc_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)},
           "selected": "blockwise" if chosen == stof.STOF_KERNEL_BLOCKWISE else "rowwise"}
    times = {}
    for name, which in (("rowwise", stof.STOF_KERNEL_ROWWISE), ("blockwise", stof.STOF_KERNEL_BLOCKWISE)):
        call = lambda: stof.stof_mha_fwd(q, k, v, fmt, scale, w.stride_b, w.stride_h, which, o)  # noqa: E731
        once = graph_ms(call, 2)
        n = max(3, min(40, int(60.0 / max(once, 1e-3))))
        warm = graph_ms(call, n)
        cold = graph_ms(call, n, flush=flush) if q.numel() * 6 < L2_BYTES else warm
        B, H, L, d = q.shape
        args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), 1 if q.dtype == torch.bfloat16 else 0, B, H, L, d,
                ctypes.c_float(scale), ctypes.byref(fmt), w.stride_b, w.stride_h, which, o.data_ptr(),
                torch.cuda.current_stream().cuda_stream)
        lat_ms, host_us = call_latency(lib.stof_mha_fwd, args)
        b2b_ms, b2b_host_us = back_to_back(lib.stof_mha_fwd, args, max(5, min(40, int(40.0 / max(warm, 1e-3)))))
        plan_args = (ctypes.byref(fmt), B, H, L, d, which, ctypes.byref(stof.stof_plan()))
        plan_us = statistics.median(host_time_us(lib.stof_mha_plan, plan_args) for _ in range(15))
        r = {"kernel_ms": round(warm, 5), "kernel_ms_cold_l2": round(cold, 5), "call_ms": round(lat_ms, 5),
             "call_minus_kernel_us": round((lat_ms - warm) * 1e3, 2), "host_us": round(host_us, 2),
             "plan_host_us": round(plan_us, 2),
             "back_to_back_ms_per_call": round(b2b_ms, 5), "back_to_back_host_us": round(b2b_host_us, 2),
             "back_to_back_minus_kernel_us": round((b2b_ms - warm) * 1e3, 2),
             "effective_tflops": round(eff_flops / (warm * 1e-3) / 1e12, 3)}
        if name == "blockwise":
            r["variant"] = ("persistent" if w.d == 64 and tiles / n_rows < 48 else "cta_per_query_tile")
            r["tile_tflops"] = round(tile_flops / (warm * 1e-3) / 1e12, 2)
            r["frac_tensor_peak_tile"] = round(tile_flops / (warm * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)
        else:
            alg = 4 * B * H * L * d * 2 + fmt_bytes
            r["gbs"] = round(alg / (warm * 1e-3) / 1e9, 1)
            r["frac_hbm"] = round(alg / (warm * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)
        rec[name] = r
        times[name] = warm
    rec["fastest"] = min(times, key=times.get)
    rec["selector_picks_fastest"] = rec["fastest"] == rec["selected"]
    # the measured choice (stof_tune: every candidate, cached) and what AUTO then runs
    wst = torch.empty(stof.stof_tune_workspace_bytes(n_masks, w.L), dtype=torch.uint8, device=q.device)
    stof.stof_tune_clear()
    tr = stof.stof_tune(mask, q, k, v, scale, w.stride_b, w.stride_h, wst, o)
    del wst
    names = ["rowwise_rpw1", "rowwise_rpw2", "rowwise_rpw4", "blockwise_st3", "blockwise_st2", "blockwise_st4",
             "blockwise_persistent_st4", "blockwise_persistent_st3", "blockwise_persistent_st2", "blockwise_128x64"]
    plan = stof.stof_mha_plan(fmt, w.B, w.H, w.L, w.d, stof.STOF_KERNEL_AUTO)
    rec["tuned"] = {"candidates_ms": {nm: round(float(t), 5) for nm, t in zip(names, tr.cand_ms) if t > 0},
                    "auto_after_tuning": {"kernel": "blockwise" if plan.kernel == stof.STOF_KERNEL_BLOCKWISE
                                          else "rowwise", "stages": plan.stages, "persistent": plan.persistent,
                                          "rows_per_warp": plan.rows_per_warp, "source": plan.source}}
    stof.stof_tune_clear()
    rec["l2"] = ("inputs fit in L2: kernel_ms warm (back to back), kernel_ms_cold_l2 with a 256 MB write "
                 "before each call" if q.numel() * 6 < L2_BYTES else "inputs larger than L2")
    del ws
    return rec


def run_workload_records(args, device, peaks, big=None) -> dict:
    """Sub-records for every workload; `big` = (workload, mask, q, k, v)
    reuses the headline run's device inputs for that workload."""
    import torch
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=device)
    out = {}
    for name in synth.WORKLOAD_ORDER:
        w = synth.WORKLOADS[name]
        if big is not None and big[0].name == name:
            _, mask, q, k, v = big
        else:
            mask, q, k, v = device_inputs(w, device)
        out[name] = workload_record(w, mask, q, k, v, peaks, flush)
        del mask, q, k, v
        torch.cuda.empty_cache()
    return out


OPROJ_SHAPES = {
    # name: (B, H, L, d, N) -- the output projection after the MHA of a layer
    "llama7b_16384tok": (1, 32, 16384, 128, 4096),
    "llama7b_4096tok": (1, 32, 4096, 128, 4096),
    "bert_base_16x512": (16, 12, 512, 64, 768),
}


def run_oproj(args):
    """The operator after the MHA: stof_oproj_fwd (y = concat_heads(O) W^T +
    bias + residual) on the shape named by --oproj, bf16, random inputs;
    kernel-only CUDA-event time over 20 calls against the measured bf16
    peak.  One JSON line."""
    import torch
    from sparse_mask_transformer_gb300 import build, stof
    torch.cuda.set_device(0)
    build.build()
    stof.load_library()
    peaks, peak_src = load_peaks()
    B, H, L, d, N = OPROJ_SHAPES[args.oproj]
    g = torch.Generator(device="cuda").manual_seed(0)
    o = torch.randn(B, H, L, d, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(N, H * d, device="cuda", generator=g) / (H * d) ** 0.5).to(torch.bfloat16)
    bias = torch.randn(N, device="cuda", generator=g).to(torch.bfloat16)
    res = torch.randn(B, L, N, device="cuda", generator=g).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(N, device="cuda", generator=g)).to(torch.bfloat16)
    beta = (0.1 * torch.randn(N, device="cuda", generator=g)).to(torch.bfloat16)
    y = torch.empty(B, L, N, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(stof.stof_oproj_ln_workspace_bytes(B, L, N), dtype=torch.uint8, device="cuda")

    def timed(call):
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            call()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps

    ms = timed(lambda: stof.stof_oproj_fwd(o, w, bias, res, y))
    ms_ln = timed(lambda: stof.stof_oproj_ln_fwd(o, w, bias, res, gamma, beta, 1e-5, y, ws))
    flops = 2.0 * B * L * N * H * d
    ln_bytes = 2 * B * L * N * 2  # the normalising pass reads and writes y
    print(json.dumps({"oproj": args.oproj, "B": B, "H": H, "L": L, "d": d, "N": N, "dtype": "bf16",
                      "ms": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
                      "frac_tensor_peak": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                      "with_layernorm": {"ms": round(ms_ln, 4), "ln_pass_ms": round(ms_ln - ms, 4),
                                         "ln_pass_gbs": round(ln_bytes / max(ms_ln - ms, 1e-6) / 1e6, 1)},
                      "peak_source": f"{peak_src} bf16 burst", "steps": args.steps, "warmup": args.warmup}),
          flush=True)


# The grid the selector's coefficients were fitted to ("fit") and a held-out
# grid of other lengths, densities, head counts and a block-sparse pattern
# ("holdout") that checks the fitted model out of sample.
SWEEPS = {
    "fit": {"L": (128, 256, 512, 1024, 2048), "density": (0.01, 0.02, 0.05, 0.1, 0.2, 0.4),
            "heads": (2, 16, 64), "patterns": ("random", "window")},
    "holdout": {"L": (384, 768, 1536, 3072), "density": (0.03, 0.07, 0.15, 0.3),
                "heads": (1, 8, 32), "patterns": ("random", "window", "blocks")},
}


def sweep_mask(pattern: str, L: int, density: float, seed: int):
    """One shared mask of the sweep: 'random' = i.i.d. Bernoulli(density)
    elements; 'window' = causal sliding window whose width gives about that
    density (at least 1 key per row)."""
    if pattern == "random":
        m = synth.random_mask(1, L, L, density, seed=seed)
    elif pattern == "blocks":  # 64 x 64 blocks kept with probability density (BigBird-like random blocks)
        nb = L // 64
        keep = np.random.default_rng(seed).random((nb, nb)) < density
        m = np.kron(keep, np.ones((64, 64), bool)).astype(np.uint8)[None]
    else:
        wdt = max(1, int(round(density * L)))
        i = np.arange(L)[:, None]
        j = np.arange(L)[None, :]
        m = ((i - j >= 0) & (i - j < wdt)).astype(np.uint8)[None]
    return m


def run_sweep(args):
    """Kernel-only times (CUDA-graph replay, warm L2) of the row-wise and the
    block-wise kernel over short sequences and low densities, with the
    analytic selector's choice: one JSON line per case, then a summary."""
    import torch
    from sparse_mask_transformer_gb300 import build, stof
    torch.cuda.set_device(0)
    build.build()
    stof.load_library()
    grid = SWEEPS[args.sweep_set]
    cases = 0
    agree = 0
    losses = []
    for d in (64, 128):
        for L in grid["L"]:
            fmts = {}
            for pattern in grid["patterns"]:
                for rho in grid["density"]:
                    mask = torch.from_numpy(sweep_mask(pattern, L, rho, seed=L + int(rho * 1000))).cuda()
                    ws = torch.empty(stof.stof_encode_workspace_bytes(1, L, L, 128, 128), dtype=torch.uint8,
                                     device="cuda")
                    fmt = stof.stof_encode_mask(mask, 128, 128, ws)
                    stof.stof_format_sync(fmt)
                    fmts[(pattern, rho)] = (fmt, ws)
            for H in grid["heads"]:
                q, k, v = (t.cuda() for t in synth.make_qkv(1, H, L, d, "bf16", seed=H))
                o = torch.empty_like(q)
                for (pattern, rho), (fmt, ws) in fmts.items():
                    density = fmt.nnz / (L * L)
                    t = {}
                    for name, which in (("rowwise", stof.STOF_KERNEL_ROWWISE),
                                        ("blockwise", stof.STOF_KERNEL_BLOCKWISE)):
                        call = lambda: stof.stof_mha_fwd(q, k, v, fmt, 1 / math.sqrt(d), 0, 0,  # noqa: E731
                                                         which, o)
                        t[name] = graph_ms(call, 20) * 1e3
                    rpw_us = {}
                    for rpw in (1, 2, 4):  # the row-wise kernel with each rows-per-warp setting
                        plan = stof.stof_plan(stof.STOF_KERNEL_ROWWISE, 0, 0, 0, rpw)
                        call = lambda: stof.stof_mha_fwd_plan(q, k, v, fmt, 1 / math.sqrt(d), 0, 0,  # noqa: E731
                                                              plan, o)
                        rpw_us[rpw] = round(graph_ms(call, 20) * 1e3, 2)
                    auto_rpw = stof.stof_mha_plan(fmt, 1, H, L, d, stof.STOF_KERNEL_ROWWISE).rows_per_warp
                    sel = "blockwise" if stof.stof_mha_plan(fmt, 1, H, L, d, stof.STOF_KERNEL_AUTO).kernel == \
                        stof.STOF_KERNEL_BLOCKWISE else "rowwise"
                    fastest = min(t, key=t.get)
                    cases += 1
                    agree += sel == fastest
                    losses.append(t[sel] / t[fastest])
                    print(json.dumps({"sweep": pattern, "L": L, "d": d, "H": H, "density": round(density, 5),
                                      "tiles": fmt.n_full + fmt.n_part, "rowwise_us": round(t["rowwise"], 2),
                                      "blockwise_us": round(t["blockwise"], 2), "selected": sel,
                                      "fastest": fastest, "rowwise_rpw_us": rpw_us, "auto_rpw": auto_rpw}),
                          flush=True)
    print(json.dumps({"sweep_summary": {"set": args.sweep_set, "cases": cases, "selector_picks_fastest": agree,
                                        "mean_time_over_fastest": round(float(np.mean(losses)), 4),
                                        "worst_time_over_fastest": round(float(np.max(losses)), 3)}}), flush=True)


def run_bitmask(args, w, mask, q, k, v, ws, scale, stream, device, dist):
    """The step with the mask given bit-packed (one bit per element, an
    eighth of the bytes): device-timed, and end to end from pinned host
    buffers of the packed mask and Q/K/V."""
    import torch
    from sparse_mask_transformer_gb300 import stof
    bits = stof.stof_synth_pack_bits(mask)
    fmt = stof.stof_format()
    o = torch.empty_like(q)

    def step():
        stof.stof_encode_mask_bits(bits, w.L, 128, 128, ws, fmt)
        stof.stof_format_sync(fmt)
        stof.stof_mha_fwd(q, k, v, fmt, scale, w.stride_b, w.stride_h, stof.STOF_KERNEL_AUTO, o)

    def timed(fn, n):
        fn()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(a.elapsed_time(b) / n, dist, device)

    enc_ms = timed(lambda: stof.stof_encode_mask_bits(bits, w.L, 128, 128, ws, fmt), args.steps)
    step_ms = timed(step, args.steps)
    valid = sum_over_ranks(4.0 * w.d * fmt.nnz * heads_per_mask(w), dist, device)
    out = {"mask_bytes": int(bits.numel()), "encode_ms": round(enc_ms, 4), "ms_per_step": round(step_ms, 4),
           "value": round(valid / (step_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s"}
    if not args.no_e2e:
        hb = torch.empty(bits.shape, dtype=torch.uint8, pin_memory=True).copy_(bits)
        hq, hk, hv = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in (q, k, v))
        ho = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)

        def e2e_step():
            bits.copy_(hb, non_blocking=True)
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            step()
            ho.copy_(o, non_blocking=True)

        ms = timed(e2e_step, max(1, min(args.steps, args.e2e_steps)))
        out["e2e"] = {"value": round(valid / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s", "ms_per_step": round(ms, 3),
                      "h2d_bytes_per_step": int(hb.numel() + 3 * hq.numel() * hq.element_size()),
                      "d2h_bytes_per_step": int(ho.numel() * ho.element_size())}
    del bits
    torch.cuda.empty_cache()
    return out


def run_rules(args, w, q, k, v, ws, scale, stream, device, dist):
    """The step with the mask given as a rule (stof_encode_rules: band,
    global tokens, blocks), for the workloads that have one: no mask is
    read, only the format is written."""
    import torch
    from sparse_mask_transformer_gb300 import stof
    rule = synth.workload_rule(w)
    if rule is None:
        return None
    bits = lambda a: None if a is None else stof.bitset_words(a, device)  # noqa: E731
    rules = [stof.MaskRule(rule["band_lo"], rule["band_hi"], bits(rule["global_rows"]), bits(rule["global_cols"]),
                           bits(rule["blocks"]), rule["block"])] * w.n_masks
    fmt = stof.stof_format()
    o = torch.empty_like(q)

    def step():
        stof.stof_encode_rules(rules, w.L, w.L, 128, 128, ws, fmt)
        stof.stof_format_sync(fmt)
        stof.stof_mha_fwd(q, k, v, fmt, scale, w.stride_b, w.stride_h, stof.STOF_KERNEL_AUTO, o)

    def timed(fn, n):
        fn()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(a.elapsed_time(b) / n, dist, device)

    enc_ms = timed(lambda: stof.stof_encode_rules(rules, w.L, w.L, 128, 128, ws, fmt), args.steps)
    step_ms = timed(step, args.steps)
    valid = sum_over_ranks(4.0 * w.d * fmt.nnz * heads_per_mask(w), dist, device)
    return {"encode_ms": round(enc_ms, 4), "ms_per_step": round(step_ms, 4),
            "value": round(valid / (step_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s"}


def run_e2e(args, w, mask, q, k, v, ws, fmt, scale, stream, device, dist):
    """Same metric through the public API from pinned host buffers: each
    step moves mask, Q, K, V host->device, runs the hot path and reads O
    back to the host.  The encoder reads the mask straight from pinned host
    memory (every byte once, over the host link, which bounds the step);
    Q, K and V are copied."""
    import torch
    from sparse_mask_transformer_gb300 import stof
    hm = torch.empty(mask.shape, dtype=mask.dtype, pin_memory=True)
    hm.copy_(mask)
    hq, hk, hv = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t) for t in (q, k, v))
    ho = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    o = torch.empty_like(q)
    steps = max(1, min(args.steps, args.e2e_steps))

    def step():
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        v.copy_(hv, non_blocking=True)
        stof.stof_encode_mask(hm, 128, 128, ws, fmt)
        stof.stof_format_sync(fmt)
        stof.stof_mha_fwd(q, k, v, fmt, scale, w.stride_b, w.stride_h, stof.STOF_KERNEL_AUTO, o)
        ho.copy_(o, non_blocking=True)

    step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1) / steps, dist, device)
    valid = fmt.nnz * heads_per_mask(w)
    total = sum_over_ranks(4.0 * w.d * valid, dist, device)
    h2d = hm.numel() + 3 * hq.numel() * hq.element_size()
    d2h = ho.numel() * ho.element_size()
    return {"value": round(total / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s", "ms_per_step": round(ms, 3),
            "steps": steps, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "mask_input": "pinned host memory, read by the encoder over the host link (no device copy)"}


# ---------------------------------------------------------------- CPU oracle

def oracle_sample(w: synth.Workload, budget_rows: int, seed: int = 0):
    """A bounded, seeded sample of the workload for the fp64 oracle: a few
    heads and query rows, plus the OT rows those queries fall in for the
    brute-force encoder."""
    rng = np.random.default_rng(seed)
    n_heads = min(w.B * w.H, 2)
    heads = [(int(x) // w.H, int(x) % w.H) for x in rng.choice(w.B * w.H, n_heads, replace=False)]
    rows = np.sort(rng.choice(w.L, min(w.L, budget_rows), replace=False))
    return heads, rows


def run_oracle_sample(w: synth.Workload, heads, rows, qkv64=None):
    """Times the oracle on the sample; returns (seconds, valid elements, threads)."""
    import oracle
    q, k, v = qkv64 if qkv64 is not None else (synth.to_float64(t) for t in synth.make_qkv(
        w.B, w.H, w.L, w.d, w.dtype, seed=w.seed))
    threads = oracle.default_threads()
    masks = {}
    for (b, h) in heads:
        m = synth.mask_index(w, b, h)
        masks[(b, h)] = synth.mask_rows(w, m, rows)
    bands = sorted({int(r) // 128 for r in rows[:4]})
    band_masks = [(synth.mask_index(w, *heads[0]), I) for I in bands]
    band_data = [synth.mask_rows(w, m, np.arange(I * 128, I * 128 + 128))[None] for m, I in band_masks]
    t0 = time.perf_counter()
    valid = 0
    for (b, h) in heads:
        oracle.attention(q[b, h, rows], k[b, h], v[b, h], masks[(b, h)], 1 / math.sqrt(w.d), threads)
        valid += int(masks[(b, h)].sum())
    for bd in band_data:
        oracle.encode(bd, 128, 128)
    return time.perf_counter() - t0, valid, threads


def cpu_baseline(w: synth.Workload, args, mask_dev, q, k, v):
    """The fp64 oracle, as it stands, on a bounded seeded sample of the
    same workload: all query rows of a seeded row sample, head after head
    until about --cpu-seconds of oracle time, plus the brute-force encoder
    on 4 OT rows scaled to the same fraction of the workload.  Mask rows and
    Q/K/V are copied from the device inputs (untimed)."""
    import oracle
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(w.L, min(w.L, args.cpu_rows), replace=False))
    order = rng.permutation(w.B * w.H)
    threads = oracle.default_threads()
    attn_s, valid, done = 0.0, 0, 0
    for x in order:
        b, h = int(x) // w.H, int(x) % w.H
        m = synth.mask_index(w, b, h)
        mrows = mask_dev[m, rows].cpu().numpy()
        qh = q[b, h, rows].double().cpu().numpy()
        kh, vh = k[b, h].double().cpu().numpy(), v[b, h].double().cpu().numpy()
        t0 = time.perf_counter()
        oracle.attention(qh, kh, vh, mrows, 1 / math.sqrt(w.d), threads)
        attn_s += time.perf_counter() - t0
        valid += int(mrows.sum())
        done += 1
        if attn_s >= args.cpu_seconds:
            break
    bands = [mask_dev[0, I * 128:(I + 1) * 128].cpu().numpy()[None] for I in rng.choice(w.L // 128, 4)]
    t0 = time.perf_counter()
    for bd in bands:
        oracle.encode(bd, 128, 128)
    enc_per_row = (time.perf_counter() - t0) / len(bands)
    frac = done * len(rows) / (w.B * w.H * w.L)
    enc_s = enc_per_row * w.n_masks * (w.L // 128) * frac
    return {"value": round(4.0 * w.d * valid / (attn_s + enc_s) / 1e12, 6), "unit": "TFLOP/s",
            "cores": threads, "kind": "oracle", "seconds": round(attn_s + enc_s, 3),
            "sample": f"{done} heads x {len(rows)} seeded query rows of {w.name} (fp64 C oracle over valid keys) "
                      f"+ brute-force encode of 4 OT rows scaled to the same {frac:.3f} of the workload"}


def run_reference(args, w: synth.Workload):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    heads, rows = oracle_sample(w, min(args.cpu_rows, 2048))
    qkv64 = tuple(synth.to_float64(t) for t in synth.make_qkv(w.B, w.H, w.L, w.d, w.dtype, seed=w.seed))
    for _ in range(args.warmup):
        run_oracle_sample(w, heads, rows[:64], qkv64)
    secs, valid = 0.0, 0
    threads = 1
    for _ in range(args.steps):
        s, vld, threads = run_oracle_sample(w, heads, rows, qkv64)
        secs += s
        valid += vld
    value = 4.0 * w.d * valid / secs / 1e12
    ms = secs / args.steps * 1e3
    sample = f"{len(heads)} heads x {len(rows)} query rows of {w.name} per step + brute-force encode of 4 OT rows"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded masks and N(0,1) Q/K/V)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d, "mask": w.describe},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="bernoulli_L16384", choices=list(synth.WORKLOADS))
    ap.add_argument("--impl", default="stof", choices=["stof", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--cpu-rows", type=int, default=8192, help="query rows per head in the oracle sample")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle time budget of the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-bitmask", action="store_true", help="skip the bit-packed-mask and mask-rule measurements")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the bench line: kernel-only times of both kernels over short, sparse cases")
    ap.add_argument("--sweep-set", default="fit", choices=list(SWEEPS),
                    help="the grid the selector was fitted to, or a held-out grid")
    ap.add_argument("--oproj", default="", choices=[""] + list(OPROJ_SHAPES),
                    help="instead of the bench line: time the output projection after the MHA on this shape")
    ap.add_argument("--no-clocks", action="store_true",
                    help="profiling runs: no clock sampling and no untimed steps around the timed ones")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-workload kernel-only records of both kernels")
    ap.add_argument("--heads", type=int, default=0,
                    help="profiling only: run the workload with this many heads (one mask per head "
                         "for per-head masks)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = synth.WORKLOADS[args.workload]
    if args.heads:
        import dataclasses
        per_head = w.n_masks == w.B * w.H
        w = dataclasses.replace(w, H=args.heads, n_masks=w.B * args.heads if per_head else w.n_masks,
                                stride_b=args.heads if per_head else w.stride_b)
    if args.sweep:
        run_sweep(args)
    elif args.oproj:
        run_oproj(args)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
