"""The seeded input generator: determinism, counter-based access, distributions."""
import numpy as np

import workloads


def test_routing_is_deterministic_and_valid():
    for w in workloads.CONFIGS.values():
        a, wa = workloads.routing(w)
        b, wb = workloads.routing(w)
        assert np.array_equal(a, b) and np.array_equal(wa, wb)
        assert a.min() >= 0 and a.max() < w.E
        assert all(len(set(row)) == w.k for row in a[:256])        # without replacement
        assert np.allclose(wa.sum(axis=1), 1.0, atol=1e-5)


def test_zipf_routing_is_skewed():
    w = workloads.CONFIGS["skewed"]
    idx, _ = workloads.routing(w)
    c = np.sort(np.bincount(idx.ravel(), minlength=w.E))[::-1]
    assert c[0] > 1000 and c[-1] < 32 and c[0] > 100 * c[-1]


def test_counter_based_rows_match_full_generation():
    w = workloads.CONFIGS["tiny"]
    x, s = workloads.x_host(w)
    x2, s2 = workloads.x_host(w, 5, 9)
    assert np.array_equal(x[5:9], x2) and np.array_equal(s[5:9], s2)
    c, cs = workloads.w_host(w, workloads.TAG_W1)
    c2, cs2 = workloads.w_host(w, workloads.TAG_W1, 3, 5, nthreads=3)
    assert np.array_equal(c[3:5], c2) and np.array_equal(cs[3:5], cs2)


def test_normal_moments():
    lib = workloads._lib_host()
    key = lib.syn_key(7, 1)
    v = np.array([lib.syn_normal_at(key, i) for i in range(200000)])
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.01


def test_fp8_weights_quantise_the_same_values():
    """The MXFP8 weight variant draws the same N(0, 1/K) values as MXFP4 and
    quantises each 32-group to E4M3 with the smallest power-of-two scale >=
    amax/448: dequantised FP8 weights agree with the FP4 ones to FP4's error."""
    import pins
    w4 = workloads.Workload("g4", T=4, H=256, I=128, E=2, k=1, seed=9)
    w8 = w4.replace(name="g8", w_fmt=1)
    c4, s4 = workloads.w_host(w4, workloads.TAG_W1)
    c8, s8 = workloads.w_host(w8, workloads.TAG_W1)
    assert c8.shape == (2, 256, 256) and c4.shape == (2, 256, 128)
    v4, v8 = pins.deq_w(c4, s4, 0), pins.deq_w(c8, s8, 1)
    # FP8: relative error of E4M3 (<= 2^-4 of the value above the subnormal range)
    amax = np.abs(v8).reshape(-1, 32).max(axis=1)
    sc = pins.deq_ue8m0(s8.reshape(-1))
    assert (amax <= 448 * sc).all() and (amax >= 224 * sc).all()
    err = np.abs(v8 - v4).max()
    assert err <= 0.5 * np.abs(v4).max()   # same draws (FP4 is the coarse one)
    assert np.corrcoef(v4.ravel(), v8.ravel())[0, 1] > 0.98


def test_float_recipe_inputs_follow_their_definition():
    """Float-scale recipe inputs, rebuilt from single normal draws: each
    activation group of 128 has the scale float32(amax) / 448 and torch's E4M3
    cast of v / scale; each 128 x 128 weight block has a scale in
    [std * 5/448, 2 * std * 5/448) and the E4M3 cast of w / scale."""
    import torch
    lib = workloads._lib_host()
    w = workloads.Workload("gf", T=3, H=256, I=128, E=2, k=1, seed=11, w_fmt=2)
    x, xs = workloads.x_host(w)
    assert x.shape == (3, 256) and xs.shape == (3, 2) and xs.dtype == np.float32
    key = lib.syn_key(w.seed, 1)
    raw = np.array([lib.syn_normal_at(key, i) for i in range(3 * 256)], np.float32)
    v = torch.from_numpy(raw).to(torch.bfloat16).to(torch.float32).numpy().reshape(3, 2, 128)
    sc = np.abs(v).max(axis=2) / np.float32(448.0)
    assert np.array_equal(xs, sc.astype(np.float32))
    codes = torch.from_numpy(np.clip(v / sc[..., None], -448, 448)).to(torch.float8_e4m3fn)
    assert np.array_equal(x.reshape(3, 2, 128), codes.view(torch.uint8).numpy())
    c, s = workloads.w_host(w, workloads.TAG_W1)
    assert c.shape == (2, 256, 256) and s.shape == (2, 2, 2) and s.dtype == np.float32
    lo = np.float32(w.std1) * np.float32(5.0 / 448.0)
    assert (s >= lo * (1 - 1e-6)).all() and (s < 2 * lo).all()
    assert len(np.unique(s)) == s.size                       # an independent draw per block
    wkey = lib.syn_key(w.seed, workloads.TAG_W1)
    for e, n, kk in ((0, 0, 0), (1, 200, 130), (1, 255, 255), (0, 129, 7)):
        idx = (e * 256 + n) * 256 + kk
        val = np.float32(lib.syn_normal_at(wkey, idx)) * np.float32(w.std1)
        q = torch.tensor([np.clip(val / s[e, n // 128, kk // 128], -448, 448)]).to(torch.float8_e4m3fn)
        assert c[e, n, kk] == q.view(torch.uint8).item()
