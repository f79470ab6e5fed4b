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
