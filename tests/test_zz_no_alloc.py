"""The allocation-free entry point, mm_run_noalloc.

Some callers cannot allocate device memory where they run the layer: plugin
hosts that own every device allocation and forbid allocating inside their
execute callback, and latency-critical loops that avoid cudaMalloc/cudaFree
because those calls can synchronise the device. mm_run_noalloc serves them by
taking its scratch from a fixed 32 MiB array inside the library.

The test calls it through the C ABI twice in a row, first on a larger call
(100 tokens, 112-token tiles) and then on a smaller one with other inputs and
other routing (8 tokens, 16-token tiles), so that the second call finds the
first call's routing tables, arrival counters and intermediates left in the
shared array. Each output must equal, bit for bit, the output of the regular
mm_run (caller workspace) on the same inputs: the two run the same kernels on
the same data. A call whose workspace would exceed the array is rejected. This
file is collected last and passes both alone and after the other tests.
"""
import numpy as np
import pytest

import gpu_util as G
import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_noalloc_equals_mm_run_on_a_large_then_a_small_call():
    import torch
    import moe_expert_layer_scan_gb300 as mm

    large = Workload("noalloc_large", T=100, H=7168, I=2048, E=16, k=8, seed=301)
    small = Workload("noalloc_small", T=8, H=7168, I=2048, E=16, k=8, seed=302)
    run = G.DeviceRun(large)
    h = run.moe.h
    assert mm.mm_workspace_bytes(h, large.T) <= 32 << 20
    assert mm.mm_token_tile_width(h, large.T) != mm.mm_token_tile_width(h, small.T)
    s = torch.cuda.current_stream().cuda_stream
    for w in (large, small):
        d = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in workloads.host_inputs(w).items()}
        ref = _bits(run.run(**d))                                  # regular entry point, caller workspace
        assert run.status() == 0
        out = torch.full((w.T, w.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = mm.mm_run_noalloc(h, w.T, d["x"].data_ptr(), d["x_sf"].data_ptr(), d["topk_idx"].data_ptr(),
                               d["topk_w"].data_ptr(), d["w1"].data_ptr(), d["w1_sf"].data_ptr(), d["w2"].data_ptr(),
                               d["w2_sf"].data_ptr(), out.data_ptr(), s)
        assert rc == 0, mm.mm_status_string(rc)
        torch.cuda.synchronize()
        got = _bits(out)
        assert np.array_equal(got, ref), f"{w.name}: mm_run_noalloc differs from mm_run " \
                                         f"on {int((got != ref).sum())} of {got.size} elements"


def test_noalloc_rejects_calls_beyond_its_scratch():
    import moe_expert_layer_scan_gb300 as mm

    moe = mm.MegaMoE(256, 7168, 2048, 8, 0)
    assert mm.mm_workspace_bytes(moe.h, 144) > 32 << 20
    rc = mm.mm_run_noalloc(moe.h, 144, *([0] * 9), 0)
    assert rc == 3  # MM_ERR_WORKSPACE_TOO_SMALL
