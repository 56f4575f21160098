"""Regression record of the oracle (tests/golden/, written by
tests/golden/make_golden.py through the oracle alone) and properties of the
seeded input generators."""
import json
import os

import numpy as np
import pytest

import oracle as O
from finite_volume_shallow_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("fname,make", [
    ("dam128_oracle.json", lambda: I.make_workload("dam128")),
    ("hills96x80_oracle.json", lambda: I.make_workload("hills2048", nx=96, ny=80)),
])
def test_oracle_matches_its_record(fname, make):
    rec = json.load(open(os.path.join(GOLDEN, fname)))
    d = make()
    W, dts, st = O.run_grid(d, nsteps=rec["steps"])
    assert st == O.OM_OK
    np.testing.assert_allclose(dts, rec["dts"], rtol=1e-14)
    for i, k in enumerate(("h", "qx", "qy", "hC")):
        got = W[i][rec["cells"]]
        scale = max(np.abs(W[i]).max(), 1e-30)
        assert np.abs(got - np.array(rec["fields"][k])).max() <= 1e-13 * scale


def test_generators_are_deterministic_and_wet():
    a = I.make_workload("hills2048", nx=300, ny=257)
    b = I.make_workload("hills2048", nx=300, ny=257)
    for k in ("H", "h", "qx", "qy", "hC"):
        assert np.array_equal(a[k], b[k])
        assert a[k].shape == (300 * 257,)
    assert a["h"].min() >= 0.5
    C = a["hC"] / a["h"]
    assert 0.0 <= C.min() and C.max() <= 1.0
    # C constant on 16 x 16 blocks
    Cb = C.reshape(257, 300)
    assert np.allclose(Cb[:16, :16], Cb[0, 0], rtol=1e-15, atol=0)
    assert not np.isclose(Cb[0, 0], Cb[0, 16])
    # surface is 5 m plus bumps of at most 3 x 0.5 m
    eta = a["h"] - a["H"]
    assert eta.min() >= 5.0 - 1e-12 and eta.max() <= 6.5


def test_lake_at_rest_generator():
    d = I.make_workload("hills2048", nx=64, ny=40, lake_at_rest=True)
    assert np.allclose(d["h"] - d["H"], 5.0, rtol=0, atol=1e-14)
    assert np.all(d["qx"] == 0) and np.all(d["qy"] == 0)
    assert d["H"].min() < -0.01                      # hills present


def test_pulses_velocities_small():
    d = I.make_workload("pulses8192", nx=128, ny=96)
    u = np.hypot(d["qx"], d["qy"]) / d["h"]
    assert u.max() <= 0.1 + 1e-12 and u.max() > 0.05


def test_dam128_shape():
    d = I.make_workload("dam128")
    h = d["h"].reshape(128, 128)
    assert h[64, 64] == 2.0 and h[0, 0] == 1.0
    assert np.array_equal(h, h.T) and np.array_equal(h, h[::-1, ::-1])
    assert d["steps"] == 100 and d["precision"] == 64


def test_full_size_records_are_consistent():
    # the full-size records come from one deterministic oracle: each names
    # its workload's own step count (or a shorter run), holds one dt per
    # step and a value per sampled cell and field; the 100-step record of
    # the mesh repeats the first 100 dt of the 500-step one bit for bit and
    # samples the same cells
    golden = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    recs = {}
    for f in sorted(os.listdir(golden)):
        if f.startswith("full_") and f.endswith(".json"):
            r = json.load(open(os.path.join(golden, f)))
            recs[f] = r
            assert len(r["dts"]) == r["steps"], f
            assert all(d > 0 for d in r["dts"]), f
            assert abs(sum(r["dts"]) - r["t"]) <= 1e-12 * r["t"], f
            for nm in r["fields"]:
                assert len(r["values"][nm]) == len(r["cells"]), (f, nm)
                assert len(r["block_means"][nm]) == 1024, (f, nm)
            if "steps.json" not in f:
                assert r["steps"] == I.WORKLOADS[r["workload"]]["steps"], f
    long, short = recs["full_tri1024_fp32.json"], recs["full_tri1024_fp32_100steps.json"]
    assert short["steps"] == 100
    assert short["dts"] == long["dts"][:100]
    assert short["cells"] == long["cells"]
