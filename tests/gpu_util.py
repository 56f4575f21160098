"""Helpers shared by the GPU tests: run a workload through the C ABI and
through the oracle on the same seeded inputs, and compare."""
import numpy as np

import oracle as O
from finite_volume_shallow_gb300 import inputs as I
from finite_volume_shallow_gb300 import swe as S

# tolerances: max |gpu - oracle| / max |oracle| per field, and relative dt
TOL = {
    64: {"h": 1e-10, "qx": 1e-10, "qy": 1e-10, "hC": 1e-10, "dt": 1e-12},
    32: {"h": 1e-4, "qx": 1e-3, "qy": 1e-3, "hC": 1e-3, "dt": 1e-6},
}


def np_dtype(precision):
    return np.float32 if precision == 32 else np.float64


def gpu_create(d, precision, cfl=None, stream=None):
    dt = np_dtype(precision)
    return S.swe_create_grid(d["nx"], d["ny"], d["dx"], d["dy"], d["H"].astype(dt),
                             [f.astype(dt) for f in I.fields_of(d)], precision=precision,
                             g=d["g"], cfl=d["cfl"] if cfl is None else cfl, stream=stream,
                             entropy_fix=d.get("entropy_fix", 0), wet_dry=d.get("wet_dry", 0),
                             h_dry=d.get("h_dry", 0.0))


def gpu_run(d, precision, nsteps, use_run=False):
    """(fields as fp64, dts, t) after nsteps GPU steps."""
    st = gpu_create(d, precision)
    if use_run:
        S.swe_run(st, nsteps)
        dts = S.swe_get_dt_history(st, nsteps)
    else:
        dts = np.array([S.swe_step(st, d["cfl"]) for _ in range(nsteps)])
    W, t = S.swe_get_state(st)
    S.swe_destroy(st)
    return [w.astype(np.float64) for w in W], np.asarray(dts), t


def oracle_run(d, precision, nsteps):
    """The oracle on the same inputs (rounded to the GPU's precision)."""
    dr = I.rounded(d, np_dtype(precision)) if precision == 32 else d
    with O.entropy_fix(d.get("entropy_fix", 0)):
        W, dts, st = O.grid_run1(d["nx"], d["ny"], d["dx"], d["dy"], dr["H"], I.fields_of(dr),
                                 d["g"], d["cfl"], nsteps)
    assert st == O.OM_OK, st
    return W, dts


def rel_errors(W_gpu, W_ref, W_init=None):
    """max |gpu - oracle| per field, relative to the field's scale: the larger
    of its max magnitude in the oracle's final state and in the initial state
    (a field that decays towards zero keeps the scale it started with)."""
    out = {}
    for i, (k, a, b) in enumerate(zip(("h", "qx", "qy", "hC"), W_gpu, W_ref)):
        scale = np.abs(b).max()
        if W_init is not None:
            scale = max(scale, np.abs(W_init[i]).max())
        out[k] = float(np.abs(a - b).max() / max(scale, 1e-30))
    return out


def assert_parity(d, precision, nsteps, use_run=False):
    Wg, dtg, tg = gpu_run(d, precision, nsteps, use_run=use_run)
    Wo, dto = oracle_run(d, precision, nsteps)
    tol = TOL[precision]
    errs = rel_errors(Wg, Wo, I.fields_of(d))
    for k in ("h", "qx", "qy", "hC"):
        assert errs[k] <= tol[k], (k, errs)
    assert len(dtg) == len(dto) == nsteps
    dte = float(np.abs(dtg / dto - 1.0).max())
    assert dte <= tol["dt"], dte
    assert abs(tg - dto.sum()) <= tol["dt"] * dto.sum()
    return errs, dte


# ---- two layers -------------------------------------------------------------
TOL2 = {
    64: {"h1": 1e-10, "q1x": 1e-10, "q1y": 1e-10, "h2": 1e-10, "q2x": 1e-10, "q2y": 1e-10,
         "dt": 1e-12},
    32: {"h1": 1e-4, "q1x": 1e-3, "q1y": 1e-3, "h2": 1e-4, "q2x": 1e-3, "q2y": 1e-3, "dt": 1e-6},
}


def gpu_create2(d, precision, stream=None):
    dt = np_dtype(precision)
    return S.swe_create_grid(d["nx"], d["ny"], d["dx"], d["dy"], d["H"].astype(dt),
                             [f.astype(dt) for f in I.fields2_of(d)], precision=precision,
                             g=d.get("g", 9.81), cfl=d.get("cfl", 0.9), stream=stream,
                             n_layers=2, pollutant=0, r=d["r"],
                             entropy_fix=d.get("entropy_fix", 0))


def gpu_run2(d, precision, nsteps):
    st = gpu_create2(d, precision)
    S.swe_run(st, nsteps)
    dts = S.swe_get_dt_history(st, nsteps)
    W, t = S.swe_get_state(st)
    S.swe_destroy(st)
    return [w.astype(np.float64) for w in W], np.asarray(dts), t


def oracle_run2(d, precision, nsteps):
    dr = I.rounded(d, np_dtype(precision)) if precision == 32 else d
    with O.entropy_fix(d.get("entropy_fix", 0)):
        W, dts, st = O.grid_run2(d["nx"], d["ny"], d["dx"], d["dy"], dr["H"], I.fields2_of(dr),
                                 d.get("g", 9.81), d["r"], d.get("cfl", 0.9), nsteps)
    assert st == O.OM_OK, st
    return W, dts


def rel_errors2(W_gpu, W_ref, W_init):
    out = {}
    for i, k in enumerate(I.TWO_LAYER_FIELDS):
        scale = max(np.abs(W_ref[i]).max(), np.abs(W_init[i]).max(), 1e-30)
        out[k] = float(np.abs(W_gpu[i] - W_ref[i]).max() / scale)
    return out


def assert_parity2(d, precision, nsteps):
    Wg, dtg, tg = gpu_run2(d, precision, nsteps)
    Wo, dto = oracle_run2(d, precision, nsteps)
    tol = TOL2[precision]
    errs = rel_errors2(Wg, Wo, I.fields2_of(d))
    for k in I.TWO_LAYER_FIELDS:
        assert errs[k] <= tol[k], (k, errs)
    assert len(dtg) == len(dto) == nsteps
    dte = float(np.abs(dtg / dto - 1.0).max())
    assert dte <= tol["dt"], dte
    return errs, dte


# ---- triangle meshes ----------------------------------------------------------
def mesh_fields(d, dtype=np.float64):
    return I.fields2_of(d, dtype) if d["n_layers"] == 2 else I.fields_of(d, dtype)


def gpu_create_mesh(d, precision, reorder=1, stream=None):
    dt = np_dtype(precision)
    two = d["n_layers"] == 2
    return S.swe_create_mesh(d["xy"], d["tri"], d["H"].astype(dt), mesh_fields(d, dt),
                             precision=precision, g=d.get("g", 9.81), cfl=d.get("cfl", 0.9),
                             stream=stream, n_layers=d["n_layers"], pollutant=0 if two else 1,
                             r=d.get("r", 0.0), reorder=reorder,
                             entropy_fix=d.get("entropy_fix", 0))


def gpu_run_mesh(d, precision, nsteps, reorder=1):
    st = gpu_create_mesh(d, precision, reorder=reorder)
    S.swe_run(st, nsteps)
    dts = S.swe_get_dt_history(st, nsteps)
    W, t = S.swe_get_state(st)
    S.swe_destroy(st)
    return [w.astype(np.float64) for w in W], np.asarray(dts), t


def oracle_run_mesh(d, precision, nsteps):
    dr = I.rounded(d, np_dtype(precision)) if precision == 32 else d
    m = O.tri_mesh(d["xy"], d["tri"])
    if d["n_layers"] == 2:
        with O.entropy_fix(d.get("entropy_fix", 0)):
            W, dts, st = O.run2(m, dr["H"], mesh_fields(dr), d.get("g", 9.81), d["r"],
                                d.get("cfl", 0.9), nsteps)
    else:
        with O.entropy_fix(d.get("entropy_fix", 0)):
            W, dts, st, _ = O.run1(m, dr["H"], mesh_fields(dr), d.get("g", 9.81),
                                   d.get("cfl", 0.9), nsteps)
    assert st == O.OM_OK, st
    return W, dts


def assert_parity_mesh(d, precision, nsteps, reorder=1):
    Wg, dtg, tg = gpu_run_mesh(d, precision, nsteps, reorder=reorder)
    Wo, dto = oracle_run_mesh(d, precision, nsteps)
    if d["n_layers"] == 2:
        tol = TOL2[precision]
        errs = rel_errors2(Wg, Wo, mesh_fields(d))
        names = I.TWO_LAYER_FIELDS
    else:
        tol = TOL[precision]
        errs = rel_errors(Wg, Wo, mesh_fields(d))
        names = ("h", "qx", "qy", "hC")
    for k in names:
        assert errs[k] <= tol[k], (k, errs)
    assert len(dtg) == len(dto) == nsteps
    dte = float(np.abs(dtg / dto - 1.0).max())
    assert dte <= tol["dt"], dte
    assert abs(tg - dto.sum()) <= tol["dt"] * dto.sum()
    return errs, dte
