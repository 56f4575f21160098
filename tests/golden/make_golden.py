"""Writes the stored expected values under tests/golden/ by calling only the
CPU oracle (``oracle/``) on seeded workloads.  The pages print no worked
numerical example for the IR-Roe step, so these files are a regression record
of the oracle, not an independent pin: they freeze the circular dam break's
per-step dt and a seeded sample of cells after 100 steps (An MPI-CUDA
implementation of an improved Roe method for two-layer shallow water
systems, Sec. 2.2, eq. (4)-(5), one layer plus pollutant).

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
from finite_volume_shallow_gb300 import inputs as I  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def record(name, d, nsteps, n_sample=64, seed=7):
    W, dts, st = O.run_grid(d, nsteps=nsteps)
    assert st == O.OM_OK
    n = d["nx"] * d["ny"]
    cells = np.sort(np.random.default_rng(seed).choice(n, n_sample, replace=False))
    out = {
        "workload": name, "nx": d["nx"], "ny": d["ny"], "dx": d["dx"], "dy": d["dy"],
        "g": d["g"], "cfl": d["cfl"], "steps": nsteps,
        "source": "oracle/swe_oracle.c via tests/golden/make_golden.py",
        "dts": [float(x) for x in dts],
        "cells": [int(c) for c in cells],
        "fields": {k: [float(W[i][c]) for c in cells] for i, k in enumerate(("h", "qx", "qy", "hC"))},
        "sums": {k: float(W[i].sum()) for i, k in enumerate(("h", "qx", "qy", "hC"))},
    }
    with open(os.path.join(HERE, f"{name}_oracle.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    record("dam128", I.make_workload("dam128"), 100)
    record("hills96x80", I.make_workload("hills2048", nx=96, ny=80), 100)
