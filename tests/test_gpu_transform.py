"""The weight-scale transform (the SM100 weight transform's scale transpose,
"MegaMoE research report" sec. 6.4 and "MEGAMOE_SM90_DESIGN" sec. 15.2): the
transformed copy's byte layout, and forwards that read it giving the same
bits as forwards that read the scale tensors themselves."""
import numpy as np
import pytest

import gpu_util as G
import workloads
from workloads import Workload

pytestmark = pytest.mark.gpu

CASES = {
    # 16-token tiles (fused), 112-token tiles with a shared expert, 224-token
    # tiles (split), E4M3 weights, both width classes of a skewed load
    "t_decode": Workload("t_decode", T=8, H=1024, I=512, E=16, k=4, seed=501),
    "t_mid": Workload("t_mid", T=300, H=1024, I=512, E=4, k=2, S=1, clamp=2.0, seed=502),
    "t_wide": Workload("t_wide", T=600, H=512, I=1024, E=2, k=1, seed=503),
    "t_fp8w": Workload("t_fp8w", T=200, H=512, I=512, E=4, k=2, seed=504, w_fmt=1),
    "t_mix": Workload("t_mix", T=256, H=512, I=512, E=16, k=4, S=1, zipf=1.2, seed=505),
}


def transformed_layout(sf: np.ndarray, K: int) -> np.ndarray:
    """The transformed copy written out from its definition: for 128-row block
    b and K step s (128 along K), byte 16 l + 4 i + j of piece (b, s) is scale
    byte 4 s + j of row 128 b + 32 i + l."""
    rows = sf.shape[0]
    steps = K // 128
    x = sf.reshape(rows // 128, 4, 32, steps, 4)          # [b][i][l][s][j]
    return np.ascontiguousarray(x.transpose(0, 3, 2, 1, 4)).reshape(-1)  # [b][s][l][i][j]


def test_transformed_layout():
    import torch
    import moe_expert_layer_scan_gb300 as mm
    w = CASES["t_mid"]
    h = workloads.host_inputs(w)
    moe = mm.MegaMoE(w.E, w.H, w.I, w.k, w.S)
    d1 = torch.from_numpy(np.ascontiguousarray(h["w1_sf"])).cuda()
    d2 = torch.from_numpy(np.ascontiguousarray(h["w2_sf"])).cuda()
    moe.transform_weight_scales(d1, d2)
    torch.cuda.synchronize()
    got = moe.tsf.cpu().numpy()
    ep = w.E + w.S
    n1 = ep * 2 * w.I * (w.H // 32)
    assert got.size == n1 + ep * w.H * (w.I // 32)
    exp1 = transformed_layout(np.asarray(h["w1_sf"]).reshape(ep * 2 * w.I, w.H // 32), w.H)
    exp2 = transformed_layout(np.asarray(h["w2_sf"]).reshape(ep * w.H, w.I // 32), w.I)
    assert np.array_equal(got[:n1], exp1)
    assert np.array_equal(got[n1:], exp2)


@pytest.mark.parametrize("name", list(CASES))
def test_transformed_scales_bit_equal(name, orc):
    """Forwards that read the transformed copy equal, bit for bit, those that
    read the scale tensors (same scales in the same TMEM columns), on both
    schedules; and match the oracle."""
    w = CASES[name]
    h = workloads.host_inputs(w)
    ref = orc.forward(dict(T=w.T, H=w.H, I=w.I, E=w.E, k=w.k, S=w.S, clamp=w.clamp, w_fmt=w.w_fmt), h["x"],
                      h["x_sf"], h["topk_idx"], h["topk_w"], h["w1"], h["w1_sf"], h["w2"], h["w2_sf"])
    for schedule in ("fused", "split"):
        plain = G.DeviceRun(w, inputs=h, schedule=schedule)
        a = plain.run()
        ia = plain.intermediates(w.T)
        tr = G.DeviceRun(w, inputs=h, schedule=schedule)
        tr.moe.transform_weight_scales(tr.d["w1_sf"], tr.d["w2_sf"])
        b = tr.run()
        ib = tr.intermediates(w.T)
        assert ia["status"] == 0 and ib["status"] == 0
        ob = G_bits(b)
        assert np.array_equal(G_bits(a), ob), f"{name} {schedule}: output differs with transformed scales"
        for k in ("l2a", "l2a_sf", "z"):
            assert np.array_equal(ia[k], ib[k]), f"{name} {schedule}: {k}"
        G.assert_out_close(ob, ref["out"])


def test_transform_registration():
    """A run whose scale pointers are not the registered ones reads its own
    arguments; dst = NULL unregisters; unsupported formats and shapes are
    refused."""
    import torch
    import moe_expert_layer_scan_gb300 as mm
    w = CASES["t_mid"]
    h = workloads.host_inputs(w)
    run = G.DeviceRun(w, inputs=h)
    ref = G_bits(run.run())
    # register a copy made from other scales (every code 127), then run with the real tensors: not used
    z1 = torch.full_like(run.d["w1_sf"], 127)
    z2 = torch.full_like(run.d["w2_sf"], 127)
    run.moe.transform_weight_scales(z1, z2)
    assert np.array_equal(G_bits(run.run()), ref)
    # the real ones registered, then unregistered
    run.moe.transform_weight_scales(run.d["w1_sf"], run.d["w2_sf"])
    assert np.array_equal(G_bits(run.run()), ref)
    mm.mm_transform_weight_scales(run.moe.h, 0, 0, 0, 0, 0)
    assert np.array_equal(G_bits(run.run()), ref)
    assert run.intermediates(w.T)["status"] == 0
    # refused: the float-scale format, and H not a multiple of 512
    f = mm.MegaMoE(4, 512, 512, 2, 0, weight_format=mm.MM_WEIGHTS_FP8_F128)
    with pytest.raises(mm.MMError):
        f.transform_weight_scales(run.d["w1_sf"], run.d["w2_sf"])
    o = mm.MegaMoE(4, 384, 512, 2, 0)
    with pytest.raises(mm.MMError):
        o.transform_weight_scales(run.d["w1_sf"], run.d["w2_sf"])


def G_bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)
