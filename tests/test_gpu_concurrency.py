"""Two forwards of the fused schedule running at the same time on two streams,
with separate handles and workspaces.

In the fused schedule an L2 tile waits for L1 tiles that other CTAs hold. The
CTAs claim tiles from a per-launch counter in index order, so every L1 tile is
claimed by a running CTA before any L2 tile and the waits end even when two
launches share the GPU's SMs. The wait limit is set short (MM_DEVICE_TIMEOUT_MS),
so that a schedule that did depend on the whole grid being resident would
report MM_DEV_TIMEOUT here quickly instead of holding the GPU.
"""
import os

import numpy as np
import pytest

import gpu_util as G
import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

CASES = [Workload("conc_a", T=64, H=2048, I=1024, E=32, k=8, seed=401),
         Workload("conc_b", T=48, H=1536, I=768, E=24, k=6, S=1, clamp=3.0, seed=402)]


def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_two_fused_forwards_on_two_streams(orc, monkeypatch):
    import torch

    monkeypatch.setenv("MM_DEVICE_TIMEOUT_MS", "200")
    runs = [G.DeviceRun(w, schedule="fused") for w in CASES]
    serial = [_bits(r.run()) for r in runs]           # each alone first
    for r in runs:
        assert r.status() == 0
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda") for w in CASES]
    torch.cuda.synchronize()
    for _ in range(20):                                # interleaved enqueues: the launches overlap
        for r, s, o in zip(runs, streams, outs):
            d = r.d
            r.moe.run(d["x"], d["x_sf"], d["topk_idx"], d["topk_w"], d["w1"], d["w1_sf"], d["w2"], d["w2_sf"],
                      out=o, stream=s)
    torch.cuda.synchronize()
    for r, s, o, ref, w in zip(runs, streams, outs, serial, CASES):
        assert r.status(stream=s) == 0, f"{w.name}: device status 0x{r.status(stream=s):x}"
        assert np.array_equal(_bits(o), ref), f"{w.name}: concurrent result differs from the serial one"
        h = workloads.host_inputs(w)
        want = orc.forward(dict(T=w.T, H=w.H, I=w.I, E=w.E, k=w.k, S=w.S, clamp=w.clamp), h["x"], h["x_sf"],
                           h["topk_idx"], h["topk_w"], h["w1"], h["w1_sf"], h["w2"], h["w2_sf"])["out"]
        G.assert_out_close(ref, want, f"{w.name} vs oracle")
