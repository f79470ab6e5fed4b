"""Expert-parallel-ready routing outputs on the GPU: the per-destination-rank
row ranges of the sorted order and the cumulative per-expert receive counts,
checked against the oracle's routing (stable counting sort)."""
import numpy as np
import pytest

import gpu_util as G
import workloads
from workloads import CONFIGS, Workload

pytestmark = pytest.mark.gpu


def _grab(run, ptr, n, dtype):
    ws = run.moe.ws
    off = ptr - ws.data_ptr()
    nbytes = n * np.dtype(dtype).itemsize
    assert 0 <= off and off + nbytes <= ws.numel()
    return ws[off:off + nbytes].cpu().numpy().view(dtype).copy()


@pytest.mark.parametrize("name,ranks", [("decode", 1), ("decode", 8), ("decode", 256), ("skewed_small", 4),
                                        ("skewed_small", 16)])
def test_rank_offsets_follow_expert_blocks(orc, name, ranks):
    w = CONFIGS.get(name) or Workload("skewed_small", T=48, H=1024, I=512, E=16, k=8, S=1, zipf=1.2, seed=103)
    run = G.DeviceRun(w, device_weights=True)
    run.mm.mm_set_ep_ranks(run.moe.h, ranks)
    run.run()
    v = run.moe.views(w.T)
    got = _grab(run, v.rank_offsets, ranks + 1, np.int32)
    idx, _ = workloads.routing(w)
    r = orc.route(idx, w.E, w.S)
    per = w.E // ranks
    want = np.array([r["offsets"][g * per] for g in range(ranks)] + [r["offsets"][w.E]], np.int32)
    assert np.array_equal(got, want)
    # every row in rank g's range belongs to an expert rank g owns
    perm = r["perm"]
    for g in range(ranks):
        slots = perm[want[g]:want[g + 1]]
        j = slots % w.Kp
        experts = idx[slots // w.Kp, np.minimum(j, w.k - 1)]
        assert ((experts // per) == g).all() and (j < w.k).all()


def test_expert_stats_accumulate_over_calls(orc):
    import torch
    w = Workload("stats", T=40, H=512, I=256, E=8, k=2, S=1, seed=301)
    run = G.DeviceRun(w)
    stats = torch.full((w.Ep,), 5, dtype=torch.int32, device="cuda")
    run.mm.mm_set_expert_stats(run.moe.h, stats.data_ptr())
    for _ in range(3):
        run.run()
    idx, _ = workloads.routing(w)
    counts = orc.route(idx, w.E, w.S)["counts"].astype(np.int64)
    assert np.array_equal(stats.cpu().numpy(), 5 + 3 * counts)
    # disabled: no further change
    run.mm.mm_set_expert_stats(run.moe.h, None)
    run.run()
    assert np.array_equal(stats.cpu().numpy(), 5 + 3 * counts)
    assert run.status() == 0


def test_expert_stats_skip_disabled_slots(orc):
    import torch
    w = Workload("stats_masked", T=16, H=256, I=128, E=4, k=2, seed=302)
    h = workloads.host_inputs(w)
    idx = h["topk_idx"].copy()
    idx[::3, 1] = -1
    h["topk_idx"] = idx
    run = G.DeviceRun(w, inputs=h)
    stats = torch.zeros(w.Ep, dtype=torch.int32, device="cuda")
    run.mm.mm_set_expert_stats(run.moe.h, stats.data_ptr())
    run.run()
    assert np.array_equal(stats.cpu().numpy(), orc.route(idx, w.E, w.S)["counts"])


def test_ep_ranks_validation():
    import moe_expert_layer_scan_gb300 as mm
    moe = mm.MegaMoE(12, 256, 128, 2, 0)
    for bad, code in ((0, 1), (13, 1), (5, 2)):
        with pytest.raises(mm.MMError) as e:
            mm.mm_set_ep_ranks(moe.h, bad)
        assert e.value.code == code
    mm.mm_set_ep_ranks(moe.h, 4)
