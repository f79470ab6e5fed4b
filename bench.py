#!/usr/bin/env python
"""Benchmark of the GB300 MoE expert path (route -> L1 -> SwiGLU/requant -> L2 -> combine).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill|decode|tiny|mid|skewed|...]
                    [--impl ours|reference]

Prints one JSON line. The default workload is prefill (T = 16384 tokens, the
largest one-GPU configuration, tensor bound); with it, the decode workload
(T = 8, weight-stream bound) is timed in the same process after it and
reported under "decode". A step is one mm_run over the workload's batch with all
inputs resident in HBM (weights generated in device memory); L2 is flushed
between steps (a 256 MB write, outside the timed events). `value` is tokens per
second over all ranks. `e2e` repeats the measurement through the public Python
API with the step's activations and routing copied from pinned host memory and
the output copied back inside the timed region. `--impl reference` times the CPU
oracle on the host cores on a bounded sample of the same workload.

Under torchrun (N > 1) every rank runs an independent replica of the workload
(tokens are independent; there is no data-path collective); a barrier and a
max-reduction of the elapsed time are the only cross-rank operations.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "MoE-layer tokens/s and TFLOP/s on 1 GB300; % of HBM or FP8xFP4 tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio (4.5 / 2.25 PFLOP/s)

# DRAM bytes (read + write) per launch of the dominant kernel from one ncu
# capture, keyed by workload, valid only while the GEMM sources hash to `src`
# (gemm_source_hash) and for the kernel named (fused "gemm" or "l1_gemm").
NCU_TRAFFIC = {
    # decode (fused GEMM): E=64 capture (42 experts touched, 988,569,856 bytes) scaled to the 61
    # experts one launch touches
    "decode": {"src": "e7f04684463aacd7", "kernel": "gemm", "bytes": 1435780029},
    # prefill (split schedule, per-expert widths: every expert above 112 rows, so both linears
    # run the 224-token tiles, one CTA per tile; the light-class launches are empty): T=2048/E=32
    # capture of the four GEMM launches (16384 rows; L1 666,591,232 + L2 483,426,304 bytes) scaled
    # x8 to 131072 rows
    "prefill": {"src": "e7f04684463aacd7", "kernel": "gemms", "bytes": 9200140288},
}


def gemm_source_hash() -> str:
    """sha256 prefix of the GEMM kernel's sources (kernel, constants, PTX helpers)."""
    h = hashlib.sha256()
    for name in ("mm_gemm.cu", "mm_common.cuh", "mm_internal.h", "mm_ptx.cuh"):
        with open(os.path.join(ROOT, "moe_expert_layer_scan_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def algorithmic(w, counts):
    """Algorithmic work of one step from the routing counts (per-expert rows)."""
    counts = np.asarray(counts)
    R = int(counts.sum())
    touched = int((counts > 0).sum())
    wsf, asf = w.w_sf_bytes, w.a_sf_bytes                       # scale bytes per element
    w1 = touched * 2 * w.I * w.H * (w.w_elem_bytes + wsf)
    w2 = touched * w.H * w.I * (w.w_elem_bytes + wsf)
    l1_act = R * w.H * (1 + asf) + R * w.I * (1 + asf)        # pool rows in, FP8 L2 operand out
    l2_act = R * w.I * (1 + asf) + R * w.H * 2                  # FP8 L2 operand in, BF16 slot rows out
    return dict(rows=R, touched=touched, flops=6.0 * w.H * w.I * R, l1_flops=4.0 * w.H * w.I * R,
                l2_flops=2.0 * w.H * w.I * R, l1_bytes=w1 + l1_act, l2_bytes=w2 + l2_act,
                weight_bytes=w1 + w2)


class Clocks:
    """nvidia-smi sampling (every 20 ms) of SM clock, power and throttle reasons
    over the whole run; `summary(windows)` keeps the samples taken inside the
    timed windows (host wall-clock intervals)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.idx = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.path = None
        self.rows = []

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)  # the sampler's first rows precede the first timed window
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    self.rows.append(parts)
        os.unlink(self.path)

    @staticmethod
    def _epoch(ts: str):
        try:
            import datetime
            return datetime.datetime.strptime(ts, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self, windows):
        """Median SM clock, max clock and the throttle reasons seen in the
        samples inside the timed windows [(t0, t1), ...]; with no sample inside
        a window (a window shorter than the sampling interval) the sample
        nearest to each window stands in, and `in_window` says how many were
        inside."""
        if not self.rows:
            return None
        num = lambda v: float(v) if v.replace(".", "").isdigit() else None
        samples = [(self._epoch(r[0]), num(r[2]), num(r[3]), r) for r in self.rows]
        samples = [x for x in samples if x[0] is not None]
        inside = [x for x in samples if any(a <= x[0] <= b for a, b in windows)]
        picked = list(inside)
        if not inside:
            for a, b in windows:
                mid = (a + b) / 2
                near = min(samples, key=lambda x: abs(x[0] - mid), default=None)
                if near is not None and near not in picked:
                    picked.append(near)
        if not picked:
            return None
        sm = [x[1] for x in picked if x[1] is not None]
        mx = [x[2] for x in picked if x[2] is not None]
        reasons = sorted({self.REASONS[i] for x in picked for i in range(4) if x[3][6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(picked), "in_window": len(inside),
                "interval_ms": self.interval_ms, "timed_windows_s": round(sum(b - a for a, b in windows), 4)}


def max_over_ranks(dist, total_ms, e2e_ms, device):
    """Slowest rank's elapsed times (the job's wall time): an all-reduce MAX of
    (device-timed total, end-to-end total); e2e_ms None on every rank stays None."""
    import torch
    t = torch.tensor([total_ms, -1.0 if e2e_ms is None else e2e_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0]), (float(t[1]) if t[1] >= 0 else None)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------- CPU oracle timing
def oracle_sample(w, n_tokens):
    """Inputs of a bounded sample (the first n_tokens tokens) for the oracle:
    the sub-problem over only the experts those tokens touch."""
    tokens = list(range(min(n_tokens, w.T)))
    idx, wt = workloads.routing(w)
    xs = [workloads.x_host(w, t, t + 1) for t in tokens]
    routed = sorted({int(e) for e in idx[tokens].ravel()})
    remap = {e: i for i, e in enumerate(routed)}
    sub_idx = np.vectorize(remap.get)(idx[tokens]).astype(np.int32)
    experts = routed + list(range(w.E, w.E + w.S))
    parts1 = [workloads.w_host(w, workloads.TAG_W1, e, e + 1) for e in experts]
    parts2 = [workloads.w_host(w, workloads.TAG_W2, e, e + 1) for e in experts]
    cat = lambda ps, i: np.ascontiguousarray(np.concatenate([p[i] for p in ps]))
    dims = dict(T=len(tokens), H=w.H, I=w.I, E=len(routed), k=w.k, S=w.S, clamp=w.clamp, w_fmt=w.w_fmt)
    args = (np.concatenate([a for a, _ in xs]), np.concatenate([b for _, b in xs]), sub_idx,
            np.ascontiguousarray(wt[tokens]), cat(parts1, 0), cat(parts1, 1), cat(parts2, 0), cat(parts2, 1))
    return dims, args, len(tokens), len(experts)


def time_oracle(w, n_tokens, reps=1):
    import oracle
    o = oracle.get()
    dims, args, nt, ne = oracle_sample(w, n_tokens)
    cores = os.cpu_count() or 1
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        o.forward(dims, *args, nthreads=cores)
        times.append(time.perf_counter() - t0)
    return times, nt, ne, cores


def sample_tokens_for(w):
    """Tokens per oracle step: about 10-30 s of CPU work on a 16-core host for one sample."""
    per_token = 6.0 * w.H * w.I * w.Kp
    return int(max(1, min(w.T, round(2.0e10 / per_token))))


def run_reference(args, world, rank):
    if rank != 0:
        return
    w = workloads.CONFIGS[args.workload]
    n_tok = max(1, min(w.T, sample_tokens_for(w) // 4))  # one step: a quarter of the CPU-baseline sample
    times, nt, ne, cores = time_oracle(w, n_tok, reps=args.warmup + args.steps)
    timed = times[args.warmup:]
    step_s = sum(timed) / len(timed)
    value = nt / step_s
    sample = f"first {nt} of {w.T} tokens of the {w.name} workload ({nt * w.Kp} slot rows, {ne} experts), per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype_of(w), "data": "synthetic",
            "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def dtype_of(w):
    return {0: "fp8xfp4", 1: "fp8xfp8", 2: "fp8xfp8 float-scaled"}[w.w_fmt] + " (fp32 accumulate)"


def workload_config(w):
    return {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "E": w.E, "topk": w.k, "shared": w.S,
            "swiglu_clamp": w.clamp, "routing": f"zipf({w.zipf})" if w.zipf else "uniform", "seed": w.seed,
            "weights": {0: "MXFP4 (E2M1 + UE8M0/32)", 1: "MXFP8 (E4M3 + UE8M0/32)",
                        2: "FP8 E4M3 + float32 scale per 128x128 block (activations float32 per 128)"}[w.w_fmt],
            "l2": "flushed between steps (256 MB write outside the timed events)"}


# ----------------------------------------------------------------------------- our arm
def measure(args, w, dist, steps, warmup, with_e2e, windows):
    """Times one workload: K whole forwards device-timed (nothing recorded
    between their kernels), K more with an event between kernels (per-kernel
    durations), then optionally the end-to-end pass. Appends the host
    wall-clock interval of every timed pass to `windows` (for the clock
    record). Returns the timings and the algorithmic work of one step."""
    import torch
    import moe_expert_layer_scan_gb300 as mm

    d = workloads.device_inputs(w)
    moe = mm.MegaMoE(w.E, w.H, w.I, w.k, w.S, swiglu_clamp=w.clamp, schedule=args.schedule, weight_format=w.w_fmt,
                     tiles=args.tiles)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    moe.workspace(w.T)
    # weight preparation, once, outside every timed region: the weight scales
    # in the tensor core's copy layout (UE8M0 formats with H and I multiples of 512)
    try:
        moe.transform_weight_scales(d["w1_sf"], d["w2_sf"])
        scales = "transformed before timing (mm_transform_weight_scales)"
    except mm.MMError:
        scales = "as given"
    torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ins = (d["x"], d["x_sf"], d["topk_idx"], d["topk_w"], d["w1"], d["w1_sf"], d["w2"], d["w2_sf"])

    for _ in range(warmup):
        flush.zero_()
        moe.run(*ins, out=out)
    torch.cuda.synchronize()
    if moe.status() != 0:
        raise RuntimeError(f"device status {moe.status()} after warm-up")
    v = moe.views(w.T)
    off = v.counts - moe.ws.data_ptr()
    counts = moe.ws[off:off + 4 * w.Ep].view(torch.int32).cpu().numpy()
    alg = algorithmic(w, counts)

    # device-resident timing: K whole forwards, nothing recorded between their kernels
    # (so each kernel's prologue overlaps its predecessor's tail as in production) ...
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_host = time.time()
    for i in range(steps):
        flush.zero_()
        e0[i].record()
        moe.run(*ins, out=out)
        e1[i].record()
    torch.cuda.synchronize()
    windows.append((t_host, time.time()))
    # ... then K more with an event between every two kernels, for the per-kernel durations
    mm.mm_profile_enable(moe.h, True)
    per_kernel = []
    t_host = time.time()
    for i in range(steps):
        flush.zero_()
        moe.run(*ins, out=out)
        per_kernel.append(mm.mm_profile_stages(moe.h))
    torch.cuda.synchronize()
    windows.append((t_host, time.time()))
    mm.mm_profile_enable(moe.h, False)
    if dist:
        dist.barrier()
    total_ms = sum(a.elapsed_time(b) for a, b in zip(e0, e1))
    if moe.status() != 0:
        raise RuntimeError(f"device status {moe.status()} after the timed steps")

    e2e_ms, h2d, d2h = None, 0, 0
    if with_e2e:
        e2e_ms, h2d, d2h = measure_e2e(args, w, d, moe, out, dist, steps, windows)
    res = dict(total_ms=total_ms, e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, per_kernel=per_kernel, alg=alg,
               tile_width=mm.mm_token_tile_width(moe.h, w.T), launches=moe.launches(w.T), weight_scales=scales)
    del moe, d, out, flush
    torch.cuda.empty_cache()
    return res


def run_ours(args, world, rank, local):
    import torch

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w = workloads.CONFIGS[args.workload]
    clocks = Clocks(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
    windows, dec_windows = [], []
    main = measure(args, w, dist, args.steps, args.warmup, not args.no_e2e, windows)
    dec = None
    if world == 1 and w.name == "prefill" and not args.no_decode_record:
        # the decode-shape line timed in the same process (both targets of the method in one run)
        dw = workloads.CONFIGS["decode"]
        dec = measure(args, dw, None, DECODE_RECORD_STEPS, args.warmup, False, dec_windows)
        dec["w"] = dw
    if clocks:
        clocks.stop()
    total_ms, e2e_ms = main["total_ms"], main["e2e_ms"]
    if dist:
        total_ms, e2e_ms = max_over_ranks(dist, total_ms, e2e_ms, device="cuda")
    if rank != 0:
        return
    main["total_ms"], main["e2e_ms"] = total_ms, e2e_ms
    clk = clocks.summary(windows) if clocks else None
    dclk = clocks.summary(dec_windows) if clocks and dec else None
    report(args, w, world, main, clk, dec=dec, dec_clk=dclk)


# steps of the decode-shape record (its forwards take ~0.26 ms: 200 of them fill a few clock samples)
DECODE_RECORD_STEPS = 200


def measure_e2e(args, w, d, moe, out, dist, steps, windows):
    """Throughput through the public call with the inputs in pinned host memory:
    every step copies its inputs host->device, runs the forward and copies the
    output device->host. As a serving loop would, the copies run on two copy
    streams (inputs, outputs) with double-buffered device tensors, so step
    i+1's inputs and step i-1's output move while step i computes; events order
    each step's forward after its inputs and each output copy after its forward.
    Timed: wall time of the K steps, first input copy to last output copy. No
    L2 flush between steps (they overlap): every step streams far more than L2
    (the touched weights and the activations)."""
    import torch
    pin = lambda t: t.cpu().pin_memory()
    hx, hxs, hidx, hw = pin(d["x"]), pin(d["x_sf"]), pin(d["topk_idx"]), pin(d["topk_w"])
    hout = [torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dins = [tuple(torch.empty_like(d[k]) for k in ("x", "x_sf", "topk_idx", "topk_w")) for _ in range(2)]
    douts = [out, torch.empty_like(out)]
    h2d = sum(t.numel() * t.element_size() for t in (hx, hxs, hidx, hw))
    d2h = hout[0].numel() * hout[0].element_size()
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    h2d_done = [ev(), ev()]
    comp_done = [ev(), ev()]
    d2h_done = [ev(), ev()]
    used = [False, False]

    def step(i):
        b = i & 1
        dx, dxs, didx, dw = dins[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(comp_done[b])  # the forward two steps back has read these inputs
            dx.copy_(hx, non_blocking=True)
            dxs.copy_(hxs, non_blocking=True)
            didx.copy_(hidx, non_blocking=True)
            dw.copy_(hw, non_blocking=True)
            h2d_done[b].record(s_in)
        comp.wait_event(h2d_done[b])
        if used[b]:
            comp.wait_event(d2h_done[b])  # the output copy two steps back has read this buffer
        moe.run(dx, dxs, didx, dw, d["w1"], d["w1_sf"], d["w2"], d["w2_sf"], out=douts[b])
        comp_done[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            hout[b].copy_(douts[b], non_blocking=True)
            d2h_done[b].record(s_out)
        used[b] = True

    for i in range(max(1, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host = time.time()
    t0.record(s_in)
    for i in range(steps):
        step(i)
    s_out.wait_stream(comp)
    t1.record(s_out)
    torch.cuda.synchronize()
    windows.append((t_host, time.time()))
    if dist:
        dist.barrier()
    e2e_ms = t0.elapsed_time(t1)
    last = (steps - 1) & 1
    assert torch.equal(hout[last], douts[last].cpu()), "end-to-end output differs from the device output"
    return e2e_ms, h2d, d2h


def roofline_of(w, alg, kern, ms_step):
    """Roofline records of one step: the dominant kernel's (the fused grouped
    GEMM, or with one launch per linear the L1 GEMM, which holds two thirds of
    the weights and FLOPs) from its mean event duration, and the whole
    forward's (all launches) from the step time. Bound by whichever of bytes
    over HBM bandwidth and FLOPs over the FP8 tensor peak takes longer for the
    dominant kernel."""
    peaks, peak_src = load_peaks()
    # "gemm": both linears in one launch; "gemms": both linears as the two
    # concurrent per-expert-width launch pairs (timed together)
    fused = "gemm" in kern or "gemms" in kern
    k_name = ("gemm" if "gemm" in kern else "gemms") if fused else "l1_gemm"
    k_ms = kern.get(k_name)
    k_bytes = alg["l1_bytes"] + alg["l2_bytes"] if fused else alg["l1_bytes"]
    k_flops = alg["flops"] if fused else alg["l1_flops"]
    hbm = float(peaks["hbm_gbs"])
    fp8_peak = float(peaks["bf16_tflops"]) * FP8_OVER_BF16
    tensor_bound = k_flops / k_bytes >= fp8_peak * 1e12 / (hbm * 1e9)
    hbm_src = f"{peak_src} hbm_gbs (STREAM-style copy)"
    tc_src = f"{peak_src} bf16_tflops (burst) x {FP8_OVER_BF16} nominal FP8/BF16 ratio"

    def rec(bytes_, flops, ms):
        if tensor_bound:
            a = flops / (ms / 1e3) / 1e12
            return {"bound": "tensor", "achieved": a, "peak": fp8_peak, "unit": "TFLOP/s", "frac": a / fp8_peak,
                    "peak_source": tc_src}
        a = bytes_ / (ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": a, "peak": hbm, "unit": "GB/s", "frac": a / hbm, "peak_source": hbm_src}

    roof = rec(k_bytes, k_flops, k_ms)
    tr = NCU_TRAFFIC.get(w.name)
    roof["traffic"] = tr["bytes"] if tr and tr.get("src") == gemm_source_hash() and tr.get("kernel") == k_name \
        else None
    roof["kernel"] = ("gemm_kernel<fused> (mm_gemm.cu): L1 then L2 tiles in one launch" if k_name == "gemm"
                      else "gemm_kernel<L1>, <L2> (mm_gemm.cu): both linears, light and heavy experts on "
                           "concurrent launches" if k_name == "gemms" else "gemm_kernel<L1> (mm_gemm.cu)")
    roof["scope"] = "dominant kernel, mean CUDA-event duration over the per-kernel pass"
    roof["algorithmic_bytes_per_launch"] = k_bytes
    roof["algorithmic_flops_per_launch"] = k_flops
    roof["kernel_ms"] = k_ms
    step = rec(alg["l1_bytes"] + alg["l2_bytes"], alg["flops"], ms_step)
    step["scope"] = ("whole forward (route, gather, both grouped GEMMs, combine) over ms_per_step: "
                     "the fraction of the roofline the fused MoE path reaches")
    step["algorithmic_bytes"] = alg["l1_bytes"] + alg["l2_bytes"]
    step["algorithmic_flops"] = alg["flops"]
    return roof, step, ("fused" if k_name == "gemm" else "split, per-expert widths" if k_name == "gemms" else "split")


def clock_record(clk, ms):
    if not clk:
        return clk
    clk = dict(clk)
    if clk.get("sm_mhz"):
        clk["ms_per_step_x_sm_mhz"] = ms * clk["sm_mhz"]
    return clk


def report(args, w, world, main, clk, dec=None, dec_clk=None):
    steps = args.steps
    ms = main["total_ms"] / steps
    tokens = w.T * world
    value = tokens / (ms / 1e3)
    alg = main["alg"]
    kern = {n: statistics.mean(p[n] for p in main["per_kernel"]) for n in main["per_kernel"][0]}
    roof, roof_step, sched = roofline_of(w, alg, kern, ms)
    e2e_ms = main["e2e_ms"]
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype_of(w), "data": "synthetic",
            "config": workload_config(w),
            "parallelism": f"{world} independent replicas" if world > 1 else "1 GPU",
            "gemm_schedule": sched + (" (auto)" if args.schedule == "auto" else ""),
            "token_tiles": ("per expert (112 / 224)" if args.tiles == 0
                            else "224 on CTA pairs" if args.tiles == -2 else f"{main['tile_width']}")
                           + (" (auto)" if args.tiles == -1 else ""),
            "weight_scales": main.get("weight_scales", "as given"),
            "tflops": alg["flops"] * world / (ms / 1e3) / 1e12,
            "hbm_gbs_whole_step": (alg["l1_bytes"] + alg["l2_bytes"]) / (ms / 1e3) / 1e9,
            "kernels_ms": kern,
            "kernels_ms_note": "mean per kernel over a second pass of the same steps with a CUDA event between "
                               "kernels (which serialises them); ms_per_step is the pass without those events",
            "rows": alg["rows"], "experts_touched": alg["touched"],
            "roofline": roof,
            "roofline_step": roof_step,
            "e2e": None if e2e_ms is None else
            {"value": tokens / (e2e_ms / steps / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": main["h2d"],
             "d2h_bytes_per_step": main["d2h"], "ms_per_step": e2e_ms / steps,
             "method": "pinned host inputs and output; per step input copy, forward, output copy, the copies on "
                       "two streams overlapping the neighbouring steps' forwards; wall time over the steps; no L2 "
                       "flush (every step streams more than L2)"},
            "gpu_launches": main["launches"] * steps,
            "clocks": clock_record(clk, ms)}
    if dec is not None:
        dw = dec["w"]
        dsteps = DECODE_RECORD_STEPS
        dms = dec["total_ms"] / dsteps
        dkern = {n: statistics.mean(p[n] for p in dec["per_kernel"]) for n in dec["per_kernel"][0]}
        droof, dstep, dsched = roofline_of(dw, dec["alg"], dkern, dms)
        line["decode"] = {"config": workload_config(dw), "steps": dsteps, "warmup": args.warmup, "ms_per_step": dms,
                          "tokens_per_s": dw.T / (dms / 1e3), "gemm_schedule": dsched,
                          "token_tiles": f"{dec['tile_width']}", "kernels_ms": dkern,
                          "rows": dec["alg"]["rows"], "experts_touched": dec["alg"]["touched"],
                          "roofline": droof, "roofline_step": dstep, "gpu_launches": dec["launches"] * dsteps,
                          "clocks": clock_record(dec_clk, dms),
                          "note": "the decode workload timed in the same process after the main line, same method "
                                  "(device-timed forwards, L2 flushed between steps; per-kernel pass after)"}
    if world == 1 and not args.no_cpu_baseline:
        n_tok = sample_tokens_for(w)
        times, nt, ne, cores = time_oracle(w, n_tok, reps=1)
        line["cpu_baseline"] = {"value": nt / times[0], "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"first {nt} of {w.T} tokens ({nt * w.Kp} slot rows, {ne} experts), "
                                          f"{times[0]:.1f} s wall"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="prefill", choices=list(workloads.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) measurement")
    ap.add_argument("--no-decode-record", action="store_true",
                    help="with the prefill workload, skip the decode-shape record timed after it")
    ap.add_argument("--tiles", type=int, default=-1, choices=[-2, -1, 0, 16, 64, 112, 224],
                    help="token-tile width (-1: the library's choice; 0: per expert, by its routed rows; "
                         "-2: 224-token tiles on CTA pairs)")
    ap.add_argument("--schedule", default="auto", choices=["auto", "fused", "split"],
                    help="GEMM schedule: one persistent launch for both linears, one per linear, or the "
                         "library's choice from the rows per expert (default)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (smaller cases for profiler captures; not a bench line)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (smaller cases for profiler captures; not a bench line)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    world, rank, local = dist_setup()
    w = workloads.CONFIGS[args.workload]
    if args.experts or args.tokens:
        w = w.replace(E=args.experts or w.E, T=args.tokens or w.T, name=w.name + "-capture")
        workloads.CONFIGS[w.name] = w
        args.workload = w.name
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
