#!/usr/bin/env python
"""Benchmark of the GB300 MoE expert path (route -> L1 -> SwiGLU/requant -> L2 -> combine).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload decode|tiny|mid|skewed|prefill]
                    [--impl ours|reference]

Prints one JSON line. A step is one mm_run over the workload's batch with all
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
    # decode (fused GEMM): E=64 capture (42 experts touched) scaled to the 61 experts one launch touches
    "decode": {"src": "be902d7cc0cdd9f4", "kernel": "gemm", "bytes": 1441261244},
    # prefill (L1 GEMM of the split schedule, 224-token tiles, one CTA per tile): T=2048/E=32
    # capture (16384 rows) scaled x8 to 131072 rows
    "prefill": {"src": "be902d7cc0cdd9f4", "kernel": "l1_gemm", "bytes": 5241108480},
}


def gemm_source_hash() -> str:
    """sha256 prefix of the GEMM kernel's sources (kernel, constants, PTX helpers)."""
    h = hashlib.sha256()
    for name in ("mm_gemm.cu", "mm_internal.h", "mm_ptx.cuh"):
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
    sf = 1.0 / 32.0
    w1 = touched * 2 * w.I * w.H * (w.w_elem_bytes + sf)
    w2 = touched * w.H * w.I * (w.w_elem_bytes + sf)
    l1_act = R * w.H * (1 + sf) + R * w.I * (1 + sf)          # pool rows in, FP8 L2 operand out
    l2_act = R * w.I * (1 + sf) + R * w.H * 2                  # FP8 L2 operand in, BF16 slot rows out
    return dict(rows=R, touched=touched, flops=6.0 * w.H * w.I * R, l1_flops=4.0 * w.H * w.I * R,
                l2_flops=2.0 * w.H * w.I * R, l1_bytes=w1 + l1_act, l2_bytes=w2 + l2_act,
                weight_bytes=w1 + w2)


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


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
    return ("fp8xfp8" if w.w_fmt else "fp8xfp4") + " (fp32 accumulate)"


def workload_config(w):
    return {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "E": w.E, "topk": w.k, "shared": w.S,
            "swiglu_clamp": w.clamp, "routing": f"zipf({w.zipf})" if w.zipf else "uniform", "seed": w.seed,
            "weights": "MXFP8 (E4M3 + UE8M0/32)" if w.w_fmt else "MXFP4 (E2M1 + UE8M0/32)",
            "l2": "flushed between steps (256 MB write outside the timed events)"}


# ----------------------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import torch
    import moe_expert_layer_scan_gb300 as mm

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w = workloads.CONFIGS[args.workload]
    d = workloads.device_inputs(w)
    moe = mm.MegaMoE(w.E, w.H, w.I, w.k, w.S, swiglu_clamp=w.clamp, schedule=args.schedule, weight_format=w.w_fmt,
                     tiles=args.tiles)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    moe.workspace(w.T)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ins = (d["x"], d["x_sf"], d["topk_idx"], d["topk_w"], d["w1"], d["w1_sf"], d["w2"], d["w2_sf"])

    for _ in range(args.warmup):
        flush.zero_()
        moe.run(*ins, out=out)
    torch.cuda.synchronize()
    if moe.status() != 0:
        raise RuntimeError(f"device status {moe.status()} after warm-up")
    counts = torch.empty(w.Ep, dtype=torch.int32)
    v = moe.views(w.T)
    counts.copy_(moe.ws[v.counts - moe.ws.data_ptr():v.counts - moe.ws.data_ptr() + 4 * w.Ep].view(torch.int32).cpu())
    alg = algorithmic(w, counts.numpy())

    # ---- device-resident timing: K whole forwards, nothing recorded between their kernels
    # (so each kernel's prologue overlaps its predecessor's tail as in production) ...
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = Clocks(torch.cuda.current_device()) if rank == 0 else None
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    for i in range(args.steps):
        flush.zero_()
        e0[i].record()
        moe.run(*ins, out=out)
        e1[i].record()
    torch.cuda.synchronize()
    # ... then K more with an event between every two kernels, for the per-kernel durations
    mm.mm_profile_enable(moe.h, True)
    per_kernel = []
    for i in range(args.steps):
        flush.zero_()
        moe.run(*ins, out=out)
        per_kernel.append(mm.mm_profile_stages(moe.h))
    torch.cuda.synchronize()
    mm.mm_profile_enable(moe.h, False)
    clk = clocks.stop() if clocks else None
    if dist:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(e0, e1)]
    total_ms = sum(step_ms)
    if moe.status() != 0:
        raise RuntimeError(f"device status {moe.status()} after the timed steps")

    # ---- end-to-end through the public API with host buffers
    e2e_ms, h2d, d2h = None, 0, 0
    if not args.no_e2e:
        e2e_ms, h2d, d2h = measure_e2e(args, w, d, moe, out, flush, dist)
    if dist:
        total_ms, e2e_ms = max_over_ranks(dist, total_ms, e2e_ms, device="cuda")
    if rank != 0:
        return
    report(args, w, world, total_ms, e2e_ms, h2d, d2h, per_kernel, alg, moe, clk)


def measure_e2e(args, w, d, moe, out, flush, dist):
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
    t0.record(s_in)
    for i in range(args.steps):
        step(i)
    s_out.wait_stream(comp)
    t1.record(s_out)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e2e_ms = t0.elapsed_time(t1)
    last = (args.steps - 1) & 1
    assert torch.equal(hout[last], douts[last].cpu()), "end-to-end output differs from the device output"
    return e2e_ms, h2d, d2h


def report(args, w, world, total_ms, e2e_ms, h2d, d2h, per_kernel, alg, moe, clk):
    import moe_expert_layer_scan_gb300 as mm
    ms = total_ms / args.steps
    tokens = w.T * world
    value = tokens / (ms / 1e3)
    kern = {n: statistics.mean(p[n] for p in per_kernel) for n in per_kernel[0]}
    peaks, peak_src = load_peaks()
    # the dominant kernel: the fused grouped GEMM (both linears in one launch)
    # or, with one launch per linear, the L1 GEMM (two thirds of the weights and FLOPs)
    fused = "gemm" in kern
    k_name = "gemm" if fused else "l1_gemm"
    k_ms = kern.get(k_name)
    k_bytes = alg["l1_bytes"] + alg["l2_bytes"] if fused else alg["l1_bytes"]
    k_flops = alg["flops"] if fused else alg["l1_flops"]
    hbm = float(peaks["hbm_gbs"])
    fp8_peak = float(peaks["bf16_tflops"]) * FP8_OVER_BF16
    balance = fp8_peak * 1e12 / (hbm * 1e9)
    if k_flops / k_bytes < balance:
        achieved = k_bytes / (k_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)"}
    else:
        achieved = k_flops / (k_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak,
                "peak_source": f"{peak_src} bf16_tflops (burst) x {FP8_OVER_BF16} nominal FP8/BF16 ratio"}
    tr = NCU_TRAFFIC.get(w.name)
    roof["traffic"] = tr["bytes"] if tr and tr.get("src") == gemm_source_hash() and tr.get("kernel") == k_name \
        else None
    roof["kernel"] = ("gemm_kernel<fused> (mm_gemm.cu): L1 then L2 tiles in one launch" if fused
                      else "gemm_kernel<L1> (mm_gemm.cu)")
    roof["algorithmic_bytes_per_launch"] = k_bytes
    roof["algorithmic_flops_per_launch"] = k_flops
    roof["kernel_ms"] = k_ms

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype_of(w), "data": "synthetic",
            "config": dict(workload_config(w), parallelism=f"{world} independent replicas" if world > 1 else "1 GPU",
                           gemm_schedule=("fused" if "gemm" in kern else "split")
                           + (" (auto)" if args.schedule == "auto" else ""),
                           token_tiles=f"{mm.mm_token_tile_width(moe.h, w.T)}"
                           + (" (auto)" if args.tiles == -1 else "")),
            "tflops": alg["flops"] * world / (ms / 1e3) / 1e12,
            "hbm_gbs_whole_step": (alg["l1_bytes"] + alg["l2_bytes"]) / (ms / 1e3) / 1e9,
            "kernels_ms": kern,
            "kernels_ms_note": "mean per kernel over a second pass of the same steps with a CUDA event between "
                               "kernels (which serialises them); ms_per_step is the pass without those events",
            "rows": alg["rows"], "experts_touched": alg["touched"],
            "roofline": roof,
            "e2e": None if e2e_ms is None else
            {"value": tokens / (e2e_ms / args.steps / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
             "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps,
             "method": "pinned host inputs and output; per step input copy, forward, output copy, the copies on "
                       "two streams overlapping the neighbouring steps' forwards; wall time over the steps; no L2 "
                       "flush (every step streams more than L2)"},
            "gpu_launches": moe.launches(w.T) * args.steps,
            "clocks": clk}
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
    ap.add_argument("--workload", default="decode", choices=list(workloads.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) measurement")
    ap.add_argument("--tiles", type=int, default=-1, choices=[-1, 16, 64, 112, 224],
                    help="token-tile width (-1: the library's choice)")
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
