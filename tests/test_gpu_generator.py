"""The device build of the input generator writes the same bytes as the host
build, so oracle inputs (host) and CUDA-path inputs (HBM) are identical."""
import numpy as np
import pytest

import workloads
from workloads import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", list(CONFIGS))
def test_device_generator_matches_host(name):
    import torch
    w = CONFIGS[name]
    tdt = lambda dt: torch.float32 if dt == np.float32 else torch.uint8
    x = torch.empty((w.T, w.H), dtype=torch.uint8, device="cuda")
    shape, dt = workloads.x_sf_shape(w, w.T)
    xs = torch.empty(shape, dtype=tdt(dt), device="cuda")
    workloads.x_device(w, x, xs)
    rows = sorted({0, w.T // 2, w.T - 1})
    for t in rows:
        hx, hs = workloads.x_host(w, t, t + 1)
        assert np.array_equal(x[t:t + 1].cpu().numpy(), hx) and np.array_equal(xs[t:t + 1].cpu().numpy(), hs)
    for which in (workloads.TAG_W1, workloads.TAG_W2):
        rows_w, K = workloads.weight_shape(w, which)
        for e in sorted({0, w.Ep - 1}):
            c = torch.empty((1, rows_w, workloads.code_bytes(w, K)), dtype=torch.uint8, device="cuda")
            shape, dt = workloads.w_sf_shape(w, which, 1)
            s = torch.empty(shape, dtype=tdt(dt), device="cuda")
            workloads.w_device(w, which, c, s, e, e + 1)
            hc, hs = workloads.w_host(w, which, e, e + 1)
            assert np.array_equal(c.cpu().numpy(), hc), f"W{which - 1} expert {e} codes differ"
            assert np.array_equal(s.cpu().numpy(), hs), f"W{which - 1} expert {e} scales differ"
