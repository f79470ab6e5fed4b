"""The allocation-free entry point, mm_run_noalloc.

Some callers cannot allocate device memory where they run the layer — plugin
hosts that own every device allocation and forbid allocating inside their
execute callback, or latency-critical loops that avoid cudaMalloc/cudaFree
because those calls can synchronise the device. mm_run_noalloc serves them by
taking its scratch from a fixed 32 MiB array inside the library. This test
calls it through the C ABI twice in a row, on two different inputs, and checks
each result against the regular mm_run (caller-provided workspace) with the
output tolerance the other GPU tests use. It also checks that a call whose
workspace would exceed the array is rejected. This file is collected last and
passes both on its own and after the other tests.
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


def test_noalloc_matches_mm_run_on_two_calls_in_a_row():
    import torch
    import moe_expert_layer_scan_gb300 as mm

    w = Workload("noalloc", T=8, H=7168, I=2048, E=16, k=8, seed=301)
    run = G.DeviceRun(w)
    inputs = [run.d, {k: torch.from_numpy(np.ascontiguousarray(v)).cuda()
                      for k, v in workloads.host_inputs(w.replace(seed=302)).items()}]
    s = torch.cuda.current_stream().cuda_stream
    for d in inputs:
        ref = _bits(run.run(**d))                                  # regular entry point, caller workspace
        out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
        rc = mm.mm_run_noalloc(run.moe.h, w.T, d["x"].data_ptr(), d["x_sf"].data_ptr(), d["topk_idx"].data_ptr(),
                               d["topk_w"].data_ptr(), d["w1"].data_ptr(), d["w1_sf"].data_ptr(), d["w2"].data_ptr(),
                               d["w2_sf"].data_ptr(), out.data_ptr(), s)
        assert rc == 0, mm.mm_status_string(rc)
        torch.cuda.synchronize()
        G.assert_out_close(_bits(out), ref, "mm_run_noalloc vs mm_run")


def test_noalloc_rejects_calls_beyond_its_scratch():
    import moe_expert_layer_scan_gb300 as mm

    moe = mm.MegaMoE(256, 7168, 2048, 8, 0)
    assert mm.mm_workspace_bytes(moe.h, 144) > 32 << 20
    rc = mm.mm_run_noalloc(moe.h, 144, *([0] * 9), 0)
    assert rc == 3  # MM_ERR_WORKSPACE_TOO_SMALL
