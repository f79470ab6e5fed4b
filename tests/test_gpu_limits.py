"""Limits of the supported shapes and reuse under CUDA-graph replay: the most
experts and slots the handle accepts, the gather's chunk-width boundary, the
routing boundary between the one-CTA and the multi-CTA routing kernels, the
largest hidden and intermediate sizes, and a forward captured into a CUDA
graph and replayed."""
import numpy as np
import pytest

import gpu_util as G
import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu


def dims(w):
    return dict(T=w.T, H=w.H, I=w.I, E=w.E, k=w.k, S=w.S, clamp=w.clamp, w_fmt=w.w_fmt)


def bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_out(orc, w, h):
    return orc.forward(dims(w), h["x"], h["x_sf"], h["topk_idx"], h["topk_w"], h["w1"], h["w1_sf"], h["w2"],
                       h["w2_sf"])


def test_most_experts_and_slots(orc):
    """E + S = 1024 experts (4 shared) and topk + S = 16 slots per token."""
    w = Workload("max_experts", T=24, H=256, I=128, E=1020, k=12, S=4, seed=401)
    h = workloads.host_inputs(w)
    run = G.DeviceRun(w, inputs=h)
    out = bits(run.run())
    ref = oracle_out(orc, w, h)
    inter = run.intermediates(w.T)
    assert inter["status"] == 0
    assert np.array_equal(inter["counts"], ref["counts"]) and np.array_equal(inter["offsets"], ref["offsets"])
    G.assert_out_close(out, ref["out"])


@pytest.mark.parametrize("T,S", [(511, 0), (512, 0), (512, 1), (37, 1)])
def test_gather_pool_rows_bit_exact(T, S):
    """The gather copies each routed slot's token row and scale row into its
    expert-sorted pool row byte for byte, on both sides of the switch between
    1 KB and 4 KB chunks per warp (512 tokens), with rows of 7168 bytes (several
    chunks per row) and with a shared expert (nine slots per token)."""
    w = Workload(f"gather_{T}_{S}", T=T, H=7168, I=128, E=16, k=8, S=S, seed=404)
    h = workloads.host_inputs(w)
    run = G.DeviceRun(w, inputs=h)
    run.run()
    inter = run.intermediates(w.T, pool=True)
    assert inter["status"] == 0
    tok = inter["perm"] // w.Kp
    assert np.array_equal(inter["pool_x"], np.asarray(h["x"]).reshape(w.T, w.H)[tok])
    assert np.array_equal(inter["pool_sf"], np.asarray(h["x_sf"]).reshape(w.T, w.H // 32)[tok])


@pytest.mark.parametrize("T", [2048, 2049])
def test_routing_boundary_single_and_multi_cta(orc, T):
    """16384 slots are routed by one CTA, 16392 by the three-pass multi-CTA
    routing: both bit-exact, both outputs within tolerance."""
    w = Workload(f"route_{T}", T=T, H=256, I=128, E=64, k=8, seed=402)
    h = workloads.host_inputs(w)
    run = G.DeviceRun(w, inputs=h)
    out = bits(run.run())
    ref = oracle_out(orc, w, h)
    inter = run.intermediates(w.T)
    n = int(ref["offsets"][-1])
    assert inter["status"] == 0
    assert np.array_equal(inter["counts"], ref["counts"])
    assert np.array_equal(inter["offsets"], ref["offsets"])
    assert np.array_equal(inter["perm"], ref["perm"][:n])
    assert np.array_equal(inter["pos"], ref["pos"])
    G.assert_out_close(out, ref["out"])


@pytest.mark.parametrize("H,I", [(16384, 256), (512, 16384)])
def test_largest_hidden_and_intermediate(orc, H, I):
    w = Workload(f"big_{H}_{I}", T=5, H=H, I=I, E=2, k=1, S=1, seed=403)
    h = workloads.host_inputs(w)
    run = G.DeviceRun(w, inputs=h)
    G.assert_out_close(bits(run.run()), oracle_out(orc, w, h)["out"])


@pytest.mark.parametrize("T", [8, 64])
def test_cuda_graph_capture_and_replay(orc, T):
    """The whole forward (its launches overlapped by programmatic dependent
    launch) captured into a CUDA graph: replays with new input contents
    reproduce the eager results bit for bit."""
    import torch
    w = Workload(f"graph_{T}", T=T, H=1024, I=512, E=16, k=4, seed=404)
    a = workloads.host_inputs(w)
    b = workloads.host_inputs(w.replace(seed=405))
    run = G.DeviceRun(w, inputs=a)
    eager_a = bits(run.run())
    static = run.d
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run.moe(static["x"], static["x_sf"], static["topk_idx"], static["topk_w"], static["w1"], static["w1_sf"],
                static["w2"], static["w2_sf"], out=out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run.moe(static["x"], static["x_sf"], static["topk_idx"], static["topk_w"], static["w1"], static["w1_sf"],
                static["w2"], static["w2_sf"], out=out)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), eager_a)
    for k in ("x", "x_sf", "topk_idx", "topk_w"):  # new activations and routing, same weights
        static[k].copy_(torch.from_numpy(np.ascontiguousarray(b[k])).cuda())
    g.replay()
    torch.cuda.synchronize()
    hb = dict(a, x=b["x"], x_sf=b["x_sf"], topk_idx=b["topk_idx"], topk_w=b["topk_w"])
    G.assert_out_close(bits(out), oracle_out(orc, w, hb)["out"])
    assert run.status() == 0
