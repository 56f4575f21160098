"""Writes the full-size, full-length expected values under tests/golden/ by
calling only the CPU oracle (``oracle/``) on the seeded workloads at their own
sizes and step counts:

    hills2048   2048 x 2048 grid, one layer + pollutant, 1000 steps, fp64 and fp32
    pulses8192  8192 x 8192 grid, one layer + pollutant,  200 steps, fp32
    tri1024     2,097,152 triangles, two layers,           500 steps, fp32
    flood2048   2048 x 2048 grid, one layer + pollutant with wet/dry fronts and
                the entropy fix,                           500 steps, fp64

An fp32 record is the fp64 oracle started from the inputs rounded to fp32 (the
values the fp32 GPU run starts from).  Each record holds the dt of every step
(eq. (5) of An MPI-CUDA implementation of an improved Roe method for two-layer
shallow water systems, Sec. 2.2), the final state at a seeded sample of cells
(walls and corners included), each field's scale (the larger of its maximum
magnitude at the start and at the end), each field's area-weighted sum at the
start and at the end, and the mean of each field over 32 x 32 blocks of the
grid (over 1024 consecutive ranges of cell numbers on the mesh), all after the
update of eq. (4) with the flux of steps 1-4.

The runs take from half an hour (2048^2) to about three hours (the mesh) of
one CPU core each.  Run from the repository root, one record per process:

    python tests/golden/make_full_size.py hills2048 64
    python tests/golden/make_full_size.py hills2048 32
    python tests/golden/make_full_size.py pulses8192 32
    python tests/golden/make_full_size.py tri1024 32
    python tests/golden/make_full_size.py flood2048 64

A third argument records a shorter run of the same workload
(full_<name>_fp<precision>_<steps>steps.json), e.g. the two-layer mesh over
100 steps, where the fp32 bounds are stated:

    python tests/golden/make_full_size.py tri1024 32 100
"""
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
from finite_volume_shallow_gb300 import inputs as I  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
N_RANDOM = 2048
N_WALL = 256
N_BLOCKS = 32


def record_path(name, precision, steps=None):
    tail = f"_{steps}steps" if steps else ""
    return os.path.join(HERE, f"full_{name}_fp{precision}{tail}.json")


def _grid_sample(nx, ny, rng):
    n = nx * ny
    i = np.arange(n) % nx
    j = np.arange(n) // nx
    wall = np.nonzero((i == 0) | (i == nx - 1) | (j == 0) | (j == ny - 1))[0]
    corners = np.array([0, nx - 1, (ny - 1) * nx, n - 1])
    cells = np.concatenate([rng.choice(n, N_RANDOM, replace=False),
                            rng.choice(wall, N_WALL, replace=False), corners])
    return np.unique(cells)


def _grid_block_means(W, nx, ny):
    out = []
    for w in W:
        a = w.reshape(ny, nx)
        bj, bi = ny // N_BLOCKS, nx // N_BLOCKS
        out.append(a.reshape(N_BLOCKS, bj, N_BLOCKS, bi).mean(axis=(1, 3)).reshape(-1))
    return out


def _chunk_means(W):
    return [np.array([c.mean() for c in np.array_split(w, N_BLOCKS * N_BLOCKS)]) for w in W]


def make(name, precision, steps=None):
    d = I.make_workload(name)
    own = steps is None
    steps = d["steps"] if own else steps
    dr = I.rounded(d, np.float32) if precision == 32 else d
    rng = np.random.default_rng(20_000 + precision)
    t0 = time.time()
    if name == "tri1024":
        names = I.TWO_LAYER_FIELDS
        W0 = I.fields2_of(dr)
        m = O.tri_mesh(d["xy"], d["tri"])
        W, dts, st = O.run2(m, dr["H"], W0, d["g"], d["r"], d["cfl"], steps)
        area = m.area
        wall = np.nonzero((m.nbr < 0).reshape(-1, 3).any(axis=1))[0]
        n = d["n_cells"]
        cells = np.unique(np.concatenate([rng.choice(n, N_RANDOM, replace=False),
                                          rng.choice(wall, N_WALL, replace=False)]))
        blocks = _chunk_means(W)
        geo = {"n_cells": int(n)}
    else:
        names = ("h", "qx", "qy", "hC")
        W0 = I.fields_of(dr)
        nx, ny = d["nx"], d["ny"]
        with O.wet_dry(d.get("h_dry", 0.0), on=bool(d.get("wet_dry", 0))), \
                O.entropy_fix(d.get("entropy_fix", 0)):
            W, dts, st = O.grid_run1(nx, ny, d["dx"], d["dy"], dr["H"], W0, d["g"], d["cfl"],
                                     steps)
        area = np.full(nx * ny, d["dx"] * d["dy"])
        cells = _grid_sample(nx, ny, rng)
        blocks = _grid_block_means(W, nx, ny)
        geo = {"nx": nx, "ny": ny, "dx": d["dx"], "dy": d["dy"]}
    assert st == O.OM_OK, st
    assert len(dts) == steps
    out = {
        "workload": name, "precision": precision, "steps": steps, "g": d["g"],
        "cfl": d["cfl"], **geo,
        "source": "oracle/ via tests/golden/make_full_size.py (fp64, one thread)",
        "oracle_seconds": round(time.time() - t0, 1),
        "fields": list(names),
        "dts": [float(x) for x in dts],
        "t": float(np.sum(dts)),
        "scale": {k: float(max(np.abs(W[i]).max(), np.abs(W0[i]).max()))
                  for i, k in enumerate(names)},
        "sum0": {k: float(W0[i].dot(area)) for i, k in enumerate(names)},
        "sum": {k: float(W[i].dot(area)) for i, k in enumerate(names)},
        "cells": [int(c) for c in cells],
        "values": {k: [float(W[i][c]) for c in cells] for i, k in enumerate(names)},
        "block_means": {k: [float(x) for x in blocks[i]] for i, k in enumerate(names)},
    }
    with open(record_path(name, precision, None if own else steps), "w") as f:
        json.dump(out, f, separators=(",", ":"))


if __name__ == "__main__":
    make(sys.argv[1], int(sys.argv[2]), int(sys.argv[3]) if len(sys.argv) > 3 else None)
