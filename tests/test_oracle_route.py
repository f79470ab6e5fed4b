"""Oracle routing pinned to NumPy's stable argsort and the counting-sort invariants."""
import numpy as np

import pins
import workloads


def test_route_matches_stable_argsort(orc):
    assert pins.pin_route(orc) == []


def test_route_invariants_on_every_workload(orc):
    for w in workloads.CONFIGS.values():
        idx, _ = workloads.routing(w)
        r = orc.route(idx, w.E, w.S)
        R = w.T * w.Kp
        assert r["counts"].sum() == R                       # every slot valid in the configs
        assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(r["counts"])]))
        assert np.array_equal(np.sort(r["perm"]), np.arange(R))      # a permutation
        assert np.array_equal(r["pos"][r["perm"]], np.arange(R))     # pos is its inverse
        ex = pins.slot_experts(idx, w.E, w.S)
        for e in range(w.Ep):
            seg = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
            assert (ex[seg] == e).all() and (np.diff(seg) > 0).all()  # stable, ascending slots
        if w.S:
            assert r["counts"][w.E] == w.T                  # the shared expert sees every token


def test_route_skips_disabled_and_counts_bad_ids(orc):
    idx = np.array([[0, -1], [5, 1], [-7, 1]], np.int32)
    r = orc.route(idx, E=3, S=1)
    assert r["bad"] == 2
    assert list(r["counts"]) == [1, 2, 0, 3]
    assert list(r["pos"]) == [0, -1, 3, -1, 1, 4, -1, 2, 5]
    assert list(r["perm"][:6]) == [0, 4, 7, 2, 5, 8]
