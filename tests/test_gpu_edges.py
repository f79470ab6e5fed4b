"""Edge cases of the CUDA path: empty and single-token calls, disabled and
out-of-range slots, duplicate experts, hot experts spanning many token tiles,
workspace reuse, determinism, fast-math SiLU and the bounded-wait status."""
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


def ref_out(orc, w, h):
    return orc.forward(dims(w), h["x"], h["x_sf"], h["topk_idx"], h["topk_w"], h["w1"], h["w1_sf"], h["w2"],
                       h["w2_sf"])


def test_zero_tokens():
    import torch
    w = Workload("t0", T=0, H=256, I=128, E=4, k=2, seed=201)
    run = G.DeviceRun(w)
    out = run.run()
    assert out.shape == (0, 256)
    assert run.status() == 0
    assert run.moe.launches(0) == 1


@pytest.mark.parametrize("T", [1, 17])
def test_single_and_boundary_token_counts(orc, T):
    w = Workload(f"t{T}", T=T, H=512, I=256, E=8, k=2, S=1, seed=202)
    h = workloads.host_inputs(w)
    run = G.DeviceRun(w, inputs=h)
    G.assert_out_close(bits(run.run()), ref_out(orc, w, h)["out"])


def test_disabled_and_out_of_range_slots(orc):
    w = Workload("bad", T=20, H=256, I=128, E=6, k=3, S=1, seed=203)
    h = workloads.host_inputs(w)
    idx = h["topk_idx"].copy()
    idx[0, :] = -1            # token 0: only the shared expert
    idx[3, 1] = 6             # out of range
    idx[5, 0] = -9            # out of range
    h["topk_idx"] = idx
    ref = ref_out(orc, w, h)
    assert ref["bad"] == 2
    run = G.DeviceRun(w, inputs=h)
    out = bits(run.run())
    assert run.status() & 0x1
    G.assert_out_close(out, ref["out"])


def test_all_slots_disabled_gives_zero():
    w = Workload("none", T=5, H=256, I=128, E=3, k=2, seed=204)
    h = workloads.host_inputs(w)
    h["topk_idx"] = np.full_like(h["topk_idx"], -1)
    run = G.DeviceRun(w, inputs=h)
    out = bits(run.run())
    assert (out == 0).all() and run.status() == 0


def test_duplicate_experts_small_variant(orc):
    """Every slot on one expert: 64 rows over four 16-token tiles."""
    w = Workload("dup", T=16, H=512, I=256, E=4, k=4, seed=205)
    h = workloads.host_inputs(w)
    h["topk_idx"] = np.full_like(h["topk_idx"], 2)
    run = G.DeviceRun(w, inputs=h, tiles=16)
    G.assert_out_close(bits(run.run()), ref_out(orc, w, h)["out"])


@pytest.mark.parametrize("tiles", [-1, 64, 224])
def test_hot_expert_many_tiles(orc, tiles):
    """One expert receives every token: several full token tiles plus a ragged
    tail (112-token tiles by the automatic policy, or 64- or 224-token tiles)."""
    w = Workload("hot", T=300, H=256, I=256, E=4, k=1, seed=206)
    h = workloads.host_inputs(w)
    h["topk_idx"] = np.zeros_like(h["topk_idx"])
    run = G.DeviceRun(w, inputs=h, tiles=tiles)
    G.assert_out_close(bits(run.run()), ref_out(orc, w, h)["out"])


def test_workspace_reuse_and_determinism():
    w = Workload("reuse", T=40, H=512, I=256, E=6, k=2, S=1, seed=207)
    a = workloads.host_inputs(w)
    b = workloads.host_inputs(w.replace(seed=208))
    run = G.DeviceRun(w, inputs=a)
    first = bits(run.run())
    import torch
    bd = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in b.items()}
    other = bits(run.run(**bd))
    again = bits(run.run())
    assert np.array_equal(first, again)          # no pollution from the previous call, deterministic
    fresh = G.DeviceRun(w, inputs=b)
    assert np.array_equal(other, bits(fresh.run()))


def test_fast_math_silu(orc):
    w = Workload("fast", T=24, H=512, I=256, E=4, k=2, seed=209)
    h = workloads.host_inputs(w)
    run = G.DeviceRun(w, inputs=h, fast_math=True)
    G.assert_out_close(bits(run.run()), ref_out(orc, w, h)["out"])


def test_bounded_wait_reports_timeout_and_gpu_stays_usable(orc):
    import torch
    import moe_expert_layer_scan_gb300 as mm
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    mm.mm_debug_timeout_probe(ws.data_ptr(), 5_000_000, s)   # 5 ms
    torch.cuda.synchronize()
    status = int(ws[:4].view(torch.int32).item())
    assert status & 0x2
    w = Workload("after", T=8, H=256, I=128, E=4, k=2, seed=210)
    h = workloads.host_inputs(w)
    run = G.DeviceRun(w, inputs=h)
    G.assert_out_close(bits(run.run()), ref_out(orc, w, h)["out"])


def test_schedule_choice_and_validation():
    """AUTO runs both GEMMs in one launch up to 128 routed rows per expert on
    average and one launch per linear above; explicit choices are honoured and
    out-of-range values rejected."""
    import moe_expert_layer_scan_gb300 as mm
    moe = mm.MegaMoE(256, 7168, 2048, 8, 0)
    small = mm.mm_launches_per_run(moe.h, 8)          # 64 rows over 256 experts: fused
    at = mm.mm_launches_per_run(moe.h, 4096)          # 128 rows per expert: still fused
    above = mm.mm_launches_per_run(moe.h, 4097)       # just above: split, per-expert widths
    assert above == at + 3                            # (two launch pairs instead of one fused launch)
    n_big = mm.mm_launches_per_run(moe.h, 16384)      # 512 rows per expert: split
    mm.mm_set_schedule(moe.h, "fused")
    assert mm.mm_launches_per_run(moe.h, 16384) == n_big - 3
    assert mm.mm_launches_per_run(moe.h, 8) == small
    mm.mm_set_schedule(moe.h, "split")
    assert mm.mm_launches_per_run(moe.h, 8) == small + 1
    with pytest.raises(mm.MMError):
        mm.mm_set_schedule(moe.h, 2)
    with pytest.raises(mm.MMError):
        mm.mm_set_schedule(moe.h, -2)


def test_weight_format_validation_and_switch(orc):
    """Switching the weight format re-describes the cached weight layout: the
    same handle runs an MXFP4, an MXFP8 and a float-scale FP8 problem correctly."""
    import torch
    import moe_expert_layer_scan_gb300 as mm
    w4 = Workload("fmt4", T=6, H=256, I=128, E=4, k=2, seed=305)
    w8 = w4.replace(name="fmt8", w_fmt=1)
    run = G.DeviceRun(w4)
    out4 = bits(run.run())
    G.assert_out_close(out4, ref_out(orc, w4, workloads.host_inputs(w4))["out"])
    h8 = workloads.host_inputs(w8)
    mm.mm_set_weight_format(run.moe.h, mm.MM_WEIGHTS_MXFP8)
    d8 = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in h8.items()}
    out8 = bits(run.run(**d8))
    G.assert_out_close(out8, ref_out(orc, w8, h8)["out"])
    # and to the float-scale format (float32 scale tensors of other shapes)
    wf = w4.replace(name="fmtf", w_fmt=2)
    hf = workloads.host_inputs(wf)
    mm.mm_set_weight_format(run.moe.h, mm.MM_WEIGHTS_FP8_F128)
    df = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in hf.items()}
    outf = bits(run.run(**df))
    G.assert_out_close(outf, ref_out(orc, wf, hf)["out"])
    with pytest.raises(mm.MMError):
        mm.mm_set_weight_format(run.moe.h, 3)


def test_tile_policy_validation():
    """The four widths, the per-expert widths and the automatic policy are
    accepted, anything else rejected; 64-token tiles exist for at most 300
    experts, larger calls run 112-token tiles."""
    import moe_expert_layer_scan_gb300 as mm
    moe = mm.MegaMoE(8, 512, 256, 2, 0)
    for t in (mm.MM_TILES_16, mm.MM_TILES_64, mm.MM_TILES_112, mm.MM_TILES_224, mm.MM_TILES_PER_EXPERT,
              mm.MM_TILES_AUTO):
        mm.mm_set_tile_policy(moe.h, t)
    for bad in (1, 32, 128, 200, 256):
        with pytest.raises(mm.MMError):
            mm.mm_set_tile_policy(moe.h, bad)
    mm.mm_set_tile_policy(moe.h, mm.MM_TILES_64)
    assert mm.mm_token_tile_width(moe.h, 64) == 64
    for e, s, width in ((299, 1, 64), (300, 1, 112), (512, 0, 112)):
        big = mm.MegaMoE(e, 512, 256, 2, s, tiles=mm.MM_TILES_64)
        assert mm.mm_token_tile_width(big.h, 64) == width, (e, s)


def test_token_tile_width_policy():
    """AUTO: 16-token tiles up to 12 routed rows per expert on average, 224
    above 112 (per-expert widths, reported as 224, when the call runs split),
    64 up to 48 without a shared expert, 112 between; a fixed policy is
    reported as set."""
    import moe_expert_layer_scan_gb300 as mm
    moe = mm.MegaMoE(256, 7168, 2048, 8, 0)
    assert mm.mm_token_tile_width(moe.h, 8) == 16          # decode: 0.25 rows per expert
    assert mm.mm_token_tile_width(moe.h, 384) == 16        # 12 rows per expert
    assert mm.mm_token_tile_width(moe.h, 385) == 64
    assert mm.mm_token_tile_width(moe.h, 1536) == 64       # 48 rows per expert
    assert mm.mm_token_tile_width(moe.h, 1537) == 112
    with_shared = mm.MegaMoE(256, 7168, 2048, 8, 1)
    assert mm.mm_token_tile_width(with_shared.h, 1024) == 112  # 36 rows per expert, one shared expert
    many = mm.MegaMoE(512, 7168, 2048, 8, 0)
    assert mm.mm_token_tile_width(many.h, 2048) == 112     # 32 rows per expert, above 300 experts
    assert mm.mm_token_tile_width(moe.h, 3584) == 112      # 112 rows per expert
    assert mm.mm_token_tile_width(moe.h, 3585) == 224      # fused, above 112
    assert mm.mm_token_tile_width(moe.h, 4096) == 224      # 128: still fused
    assert mm.mm_token_tile_width(moe.h, 4097) == 224      # split from here: per-expert widths
    assert mm.mm_token_tile_width(moe.h, 16384) == 224     # prefill: 512 rows per expert
    skewed = mm.MegaMoE(256, 7168, 2048, 8, 1)
    assert mm.mm_token_tile_width(skewed.h, 4096) == 224   # 143 rows per expert, split, per expert
    assert mm.mm_launches_per_run(skewed.h, 4096) == mm.mm_launches_per_run(moe.h, 4097)
    mm.mm_set_schedule(moe.h, "split")
    assert mm.mm_token_tile_width(moe.h, 4096) == 224      # 128 rows per expert, split: per expert
    assert mm.mm_token_tile_width(moe.h, 3584) == 112      # 112 rows per expert, split: one width
    mm.mm_set_schedule(moe.h, "auto")
    mm.mm_set_tile_policy(moe.h, mm.MM_TILES_112)
    assert mm.mm_token_tile_width(moe.h, 16384) == 112
    mm.mm_set_tile_policy(moe.h, mm.MM_TILES_16)
    assert mm.mm_token_tile_width(moe.h, 16384) == 16
