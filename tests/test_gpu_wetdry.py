"""The one-layer step with wet/dry fronts (swe_params.wet_dry = 1) on the GPU,
through the C ABI, against the oracle with its wet/dry treatment on (dry
cells, emerged banks as walls after Brufau, Vazquez-Cendon and
Garcia-Navarro 2002; draining-time positivity after Bollermann, Chen,
Kurganov and Noelle 2013), element by element on the same seeded inputs.

Tolerances as for the plain scheme: fp64 1e-10 per field (relative to its
scale) and 1e-12 on dt; fp32 1e-4 on h, 1e-3 on q and hC, 1e-6 on dt, the
oracle starting from the fp32-rounded inputs.  Where a depth crosses h_dry
the dry/wet decision is a branch, so the fp32 cases are ones whose
decisions stay clear of the threshold.
"""
import math

import numpy as np
import pytest

import oracle as O
from finite_volume_shallow_gb300 import inputs as I
from finite_volume_shallow_gb300 import swe as S
from gpu_util import TOL, np_dtype, rel_errors

pytestmark = pytest.mark.gpu

H_DRY = 1e-4


def _create(d, precision, efix, h_dry=H_DRY):
    dt = np_dtype(precision)
    return S.swe_create_grid(d["nx"], d["ny"], d["dx"], d["dy"], d["H"].astype(dt),
                             [f.astype(dt) for f in I.fields_of(d)], precision=precision,
                             g=9.81, cfl=0.9, entropy_fix=efix, wet_dry=1, h_dry=h_dry)


def _gpu(d, precision, efix, nsteps):
    st = _create(d, precision, efix)
    S.swe_run(st, nsteps)
    dts = S.swe_get_dt_history(st, nsteps)
    W, t = S.swe_get_state(st)
    S.swe_destroy(st)
    return [w.astype(np.float64) for w in W], np.asarray(dts), t


def _oracle(d, precision, efix, nsteps):
    dr = I.rounded(d, np_dtype(precision)) if precision == 32 else d
    with O.wet_dry(H_DRY), O.entropy_fix(efix):
        W, dts, st = O.grid_run1(d["nx"], d["ny"], d["dx"], d["dy"], dr["H"], I.fields_of(dr),
                                 9.81, 0.9, nsteps)
    assert st == O.OM_OK, st
    return W, dts


def _parity(d, precision, efix, nsteps, at_rest=False):
    Wg, dtg, tg = _gpu(d, precision, efix, nsteps)
    Wo, dto = _oracle(d, precision, efix, nsteps)
    W0 = I.fields_of(d)
    if at_rest:
        # discharges stay at rounding level on both sides: measure them
        # against the discharge scale h sqrt(g h) of the deepest water
        hm = d["h"].max()
        W0 = [W0[0], np.full_like(W0[1], hm * math.sqrt(9.81 * hm)),
              np.full_like(W0[2], hm * math.sqrt(9.81 * hm)), W0[3]]
    errs = rel_errors(Wg, Wo, W0)
    tol = TOL[precision]
    for k in ("h", "qx", "qy", "hC"):
        assert errs[k] <= tol[k], (k, errs)
    assert len(dtg) == nsteps
    dte = float(np.abs(dtg / dto - 1.0).max())
    assert dte <= tol["dt"], dte
    assert abs(tg - dto.sum()) <= tol["dt"] * dto.sum()
    assert Wg[0].min() >= 0.0
    return Wg, Wo


@pytest.mark.parametrize("efix", [1, 0])
def test_ritter_dry_bed_dam_break(efix):
    d = I.dry_dam_1d(400)
    _parity(d, 64, efix, 150)


def test_ritter_dry_bed_dam_break_fp32():
    d = I.dry_dam_1d(300, ny=3)
    _parity(d, 32, 1, 60)


@pytest.mark.parametrize("precision", [64, 32])
def test_lake_at_rest_against_emerged_hills(precision):
    d = I.emerged_hills(97, 61)
    Wg, Wo = _parity(d, precision, 0, 100, at_rest=True)
    h0 = d["h"].astype(np_dtype(precision)).astype(np.float64)
    scale = h0.max()
    if precision == 64:
        assert np.abs(Wg[0] - h0).max() <= 1e-13 * scale
        assert np.abs(Wg[1]).max() <= 1e-13 * scale * math.sqrt(9.81 * scale)
    assert np.array_equal(Wg[0][h0 == 0.0], h0[h0 == 0.0])


@pytest.mark.parametrize("efix", [1, 0])
@pytest.mark.parametrize("nx,ny", [(60, 44), (131, 37)])
def test_flooding_dry_land(efix, nx, ny):
    d = I.emerged_hills(nx, ny, column=(200.0, 220.0, 80.0, 2.0))
    Wg, _ = _parity(d, 64, efix, 200)
    W0 = I.fields_of(d)
    assert abs(Wg[0].sum() / W0[0].sum() - 1.0) <= 1e-12
    assert abs(Wg[3].sum() / W0[3].sum() - 1.0) <= 1e-12
    dry = Wg[0] <= H_DRY
    assert np.all(Wg[1][dry] == 0.0) and np.all(Wg[2][dry] == 0.0)


@pytest.mark.parametrize("nx,ny", [(1, 1), (1, 9), (9, 1), (33, 9), (32, 8)])
def test_small_and_ragged_grids(nx, ny):
    d = I.emerged_hills(nx, ny, dx=40.0, column=(0.5 * nx * 40.0, 0.5 * ny * 40.0, 60.0, 1.0))
    _parity(d, 64, 1, 20)


def test_anisotropic_cells():
    d = I.emerged_hills(48, 30, column=(200.0, 150.0, 80.0, 2.0))
    d["dy"] = 17.0
    _parity(d, 64, 1, 60)


def test_all_wet_is_the_plain_scheme():
    # with no dry cell and no cell draining within a step, the wet/dry path
    # (its own kernels, flux form) agrees with the fused step to rounding
    d = I.dam_break_1d(300)
    Wg, dtg, _ = _gpu(d, 64, 0, 80)
    st = S.swe_create_grid(d["nx"], d["ny"], d["dx"], d["dy"], d["H"], I.fields_of(d),
                           precision=64)
    S.swe_run(st, 80)
    Wp, _ = S.swe_get_state(st)
    dtp = S.swe_get_dt_history(st, 80)
    S.swe_destroy(st)
    errs = rel_errors(Wg, Wp, I.fields_of(d))
    assert max(errs.values()) <= 1e-12, errs
    assert np.abs(dtg / dtp - 1).max() <= 1e-13


def test_restart_is_bitwise():
    d = I.emerged_hills(50, 40, column=(200.0, 200.0, 80.0, 2.0))
    st = _create(d, 64, 1)
    S.swe_run(st, 30)
    W, t = S.swe_get_state(st)
    S.swe_run(st, 20)
    Wa, ta = S.swe_get_state(st)
    S.swe_set_state(st, W, t)
    S.swe_run(st, 20)
    Wb, tb = S.swe_get_state(st)
    S.swe_destroy(st)
    assert ta == tb
    for a, b in zip(Wa, Wb):
        assert np.array_equal(a, b)


def test_per_kernel_timing_lists_the_wet_dry_kernels():
    d = I.emerged_hills(64, 48, column=(200.0, 200.0, 80.0, 2.0))
    st = _create(d, 32, 0)
    S.swe_set_timing(st, True)
    S.swe_run(st, 5)
    tm = S.swe_get_timing(st)
    S.swe_destroy(st)
    assert list(tm) == ["wd_speed_kernel", "wd_tile_kernel"]
    assert all(v[0] == 5 and v[1] > 0 for v in tm.values())


def test_errors_and_unsupported_requests():
    d = I.emerged_hills(16, 12)
    z = np.zeros(16 * 12)
    # an all-dry domain has no finite time step
    st = S.swe_create_grid(16, 12, 10.0, 10.0, d["H"], [z, z, z, z], wet_dry=1, h_dry=H_DRY)
    with pytest.raises(S.SweError) as e:
        S.swe_step(st, 0.9)
    assert e.value.status == S.SWE_ERR_NONFINITE
    S.swe_destroy(st)
    # a negative depth is refused even with the wet/dry treatment
    h = d["h"].copy()
    h[5] = -1e-3
    with pytest.raises(S.SweError) as e:
        S.swe_create_grid(16, 12, 10.0, 10.0, d["H"], [h, z, z, z], wet_dry=1, h_dry=H_DRY)
    assert e.value.status == S.SWE_ERR_ARG
    # two layers and triangle meshes have no wet/dry treatment here
    with pytest.raises(S.SweError) as e:
        S.swe_create_grid(16, 12, 10.0, 10.0, d["H"], [d["h"] + 1, z, z, d["h"] + 1, z, z],
                          n_layers=2, pollutant=0, r=0.5, wet_dry=1, h_dry=H_DRY)
    assert e.value.status == S.SWE_ERR_UNSUPPORTED
    m = I.tri_workload1(6, 5, seed=3)
    with pytest.raises(S.SweError) as e:
        S.swe_create_mesh(m["xy"], m["tri"], m["H"], I.fields_of(m), wet_dry=1, h_dry=H_DRY)
    assert e.value.status == S.SWE_ERR_UNSUPPORTED
