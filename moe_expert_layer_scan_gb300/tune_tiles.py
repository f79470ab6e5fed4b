"""Measures the token-tile crossovers of the grouped GEMMs on this GPU.

    python -m moe_expert_layer_scan_gb300.tune_tiles [--workload prefill] [--tokens 64,128,256,384,512]
                                                     [--widths 16,64,112,224]

For each token count, runs the whole forward with each token-tile width
(schedule chosen by the library) on seeded synthetic inputs of the workload's
shape (weights generated in device memory), L2 flushed between steps, and
prints the median step time of each and the mean routed rows per expert. The
library's automatic policy switches from 16-token tiles above
MM_TILES16_MAX_ROWS_PER_EXPERT rows per expert (to 64-token tiles up to
MM_TILES64_MAX_ROWS_PER_EXPERT when the call has no shared expert, then
112-token tiles) and to 224-token tiles at MM_TILES224_MIN_ROWS_PER_EXPERT,
the crossovers this measures.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import workloads  # noqa: E402

import moe_expert_layer_scan_gb300 as mm  # noqa: E402


def measure(moe, args, out, flush, steps=10, warmup=3):
    import torch
    for _ in range(warmup):
        flush.zero_()
        moe.run(*args, out=out)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        flush.zero_()
        a.record()
        moe.run(*args, out=out)
        b.record()
    torch.cuda.synchronize()
    if moe.status() != 0:
        raise RuntimeError(f"device status {moe.status():#x}")
    return float(np.median([a.elapsed_time(b) for a, b in ev]))


def main():
    import torch
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="prefill", choices=list(workloads.CONFIGS))
    ap.add_argument("--tokens", default="64,128,256,320,384,448,512,1024")
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--widths", default="16,112")
    a = ap.parse_args()
    base = workloads.CONFIGS[a.workload]
    Ts = [int(t) for t in a.tokens.split(",")]
    widths = [int(x) for x in a.widths.split(",")]
    d = workloads.device_inputs(base.replace(T=max(Ts)))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    print(f"# {base.name} shape: H={base.H} I={base.I} E={base.E} top-{base.k} shared={base.S}")
    print("tokens  rows/expert  " + "  ".join(f"ms({b}-token tiles)" for b in widths) + "  faster")
    for T in Ts:
        w = base.replace(T=T, name=f"{base.name}_T{T}")
        idx, wt = workloads.routing(w)
        args = (d["x"][:T], d["x_sf"][:T], torch.from_numpy(idx).cuda(), torch.from_numpy(wt).cuda(),
                d["w1"], d["w1_sf"], d["w2"], d["w2_sf"])
        out = torch.empty((T, w.H), dtype=torch.bfloat16, device="cuda")
        ms = {}
        for tiles in widths:
            moe = mm.MegaMoE(w.E, w.H, w.I, w.k, w.S, swiglu_clamp=w.clamp, weight_format=w.w_fmt, tiles=tiles)
            ms[tiles] = measure(moe, args, out, flush, steps=a.steps)
            del moe
        rows = T * w.Kp / w.Ep
        best = min(widths, key=lambda b: ms[b])
        print(f"{T:6d}  {rows:11.2f}  " + "  ".join(f"{ms[b]:18.4f}" for b in widths) + f"  {best}")
        print(json.dumps({"T": T, "rows_per_expert": rows, **{f"ms{b}": ms[b] for b in widths}}), file=sys.stderr)


if __name__ == "__main__":
    main()
