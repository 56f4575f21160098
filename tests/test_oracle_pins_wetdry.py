"""Pins of the oracle's wet/dry treatment (one layer), each against what the
mathematics or a published solution fixes, never against the oracle itself.

The pages give no wet/dry treatment (An MPI-CUDA implementation of an
improved Roe method for two-layer shallow water systems, Sec. 2.2, keeps
depths positive); the oracle's is the combination of Brufau, Vazquez-Cendon
and Garcia-Navarro (2002: dry cells, emerged banks as walls) and the
draining time of Bollermann, Chen, Kurganov and Noelle (2013: positivity).
  - Ritter's dry-bed dam break: with the Harten-Hyman entropy fix (its fan is
    transonic) the L1 errors of depth and discharge against the analytic
    solution fall by at least 1.4 per doubling of the resolution; without
    the fix the error stalls (an expansion shock sits at the dam);
  - water at rest against emerged hills stays at rest (the banks act as
    walls), to rounding;
  - mass and pollutant are conserved to 1e-12 and depths stay >= 0 while a
    column of water floods dry land between hills;
  - with every cell wet and no cell draining within a step the treatment
    changes nothing: the result is bitwise the plain scheme's;
  - an all-dry domain has no finite time step.
"""
import math

import numpy as np
import pytest

import oracle as O
import ritter
from finite_volume_shallow_gb300 import inputs as I

G = 9.81
H_DRY = 1e-4


def _ritter_errors(nx, efix, t_end=40.0):
    d = I.dry_dam_1d(nx)
    W = I.fields_of(d)
    t = 0.0
    with O.wet_dry(H_DRY), O.entropy_fix(efix):
        while t < t_end:
            dt = O.grid_dt1(nx, d["ny"], d["dx"], d["dy"], d["H"], W, G, 0.9)
            W, st = O.grid_update1(nx, d["ny"], d["dx"], d["dy"], d["H"], W, G, dt)
            assert st == O.OM_OK
            t += dt
    x = (np.arange(nx) + 0.5) * d["dx"]
    he, ue = ritter.solution(x, t, 1000.0, 2.0, G)
    h = W[0].reshape(d["ny"], nx)
    q = W[1].reshape(d["ny"], nx)
    assert np.array_equal(h, np.tile(h[0], (d["ny"], 1)))  # no y dependence
    assert h.min() >= 0.0
    return (np.abs(h[0] - he).sum() * d["dx"], np.abs(q[0] - he * ue).sum() * d["dx"])


def test_ritter_dry_bed_dam_break_converges_with_the_entropy_fix():
    errs = [_ritter_errors(nx, 1) for nx in (200, 400, 800, 1600)]
    for (eh0, eq0), (eh1, eq1) in zip(errs, errs[1:]):
        assert eh0 / eh1 >= 1.4, errs
        assert eq0 / eq1 >= 1.4, errs
    assert errs[-1][0] < 6.0  # m^2 of depth error over a 2000 m channel


def test_ritter_without_the_fix_keeps_an_expansion_shock():
    e400, _ = _ritter_errors(400, 0)
    e1600, _ = _ritter_errors(1600, 0)
    assert e400 / e1600 < 1.6  # two doublings: the fixed scheme gains > 2.4
    assert e1600 > 2.0 * _ritter_errors(1600, 1)[0]


def test_ritter_front_position_converges():
    # where the depth falls to 1 cm: x0 + (2 c0 - 3 sqrt(g 0.01)) t exactly;
    # the first-order front lags behind it by less at every doubling
    lags = []
    for nx in (400, 800, 1600):
        d = I.dry_dam_1d(nx)
        W = I.fields_of(d)
        t = 0.0
        with O.wet_dry(H_DRY), O.entropy_fix():
            while t < 30.0:
                dt = O.grid_dt1(nx, d["ny"], d["dx"], d["dy"], d["H"], W, G, 0.9)
                W, st = O.grid_update1(nx, d["ny"], d["dx"], d["dy"], d["H"], W, G, dt)
                assert st == O.OM_OK
                t += dt
        wet = np.nonzero(W[0].reshape(d["ny"], nx)[0] > 0.01)[0]
        x_num = (wet.max() + 1) * d["dx"]
        x_exact = 1000.0 + (2.0 * math.sqrt(G * 2.0) - 3.0 * math.sqrt(G * 0.01)) * t
        lags.append((x_exact - x_num) / (x_exact - 1000.0))
    assert lags[0] > lags[1] > lags[2] > 0.0, lags
    assert lags[2] < 0.1, lags


def test_lake_at_rest_against_emerged_hills():
    d = I.emerged_hills(60, 44)
    h0 = d["h"].copy()
    dry = h0 == 0.0
    assert 0.05 < dry.mean() < 0.5  # hill tops stick out of the water
    with O.wet_dry(H_DRY):
        W, dts, st = O.grid_run1(d["nx"], d["ny"], d["dx"], d["dy"], d["H"], I.fields_of(d), G,
                                 0.9, 200)
    assert st == O.OM_OK
    scale = h0.max()
    qscale = scale * math.sqrt(G * scale)
    assert np.abs(W[0] - h0).max() <= 1e-13 * scale
    assert np.abs(W[1]).max() <= 1e-13 * qscale and np.abs(W[2]).max() <= 1e-13 * qscale
    assert np.array_equal(W[0][dry], h0[dry])


@pytest.mark.parametrize("efix", [0, 1])
def test_flooding_dry_land_conserves_mass_and_keeps_depths_positive(efix):
    d = I.emerged_hills(60, 44, column=(200.0, 220.0, 80.0, 2.0))
    W0 = I.fields_of(d)
    m0, c0 = W0[0].sum(), W0[3].sum()
    with O.wet_dry(H_DRY), O.entropy_fix(efix):
        W, dts, st = O.grid_run1(d["nx"], d["ny"], d["dx"], d["dy"], d["H"], W0, G, 0.9, 300)
    assert st == O.OM_OK
    assert abs(W[0].sum() - m0) <= 1e-12 * m0
    assert abs(W[3].sum() - c0) <= 1e-12 * c0
    assert W[0].min() >= 0.0
    assert W[3].min() >= -1e-12 * W0[3].max()
    # the flood reached cells that were dry, and dry cells carry no discharge
    assert ((W0[0] == 0.0) & (W[0] > H_DRY)).any()
    dry = W[0] <= H_DRY
    assert np.all(W[1][dry] == 0.0) and np.all(W[2][dry] == 0.0)
    # the time step stays physical: no film is driven to absurd speeds
    assert dts.min() > 0.2 * dts.max()


def test_all_wet_without_draining_is_the_plain_scheme():
    d = I.dam_break_1d(400)
    W = I.fields_of(d)
    plain, dts_p, st_p = O.grid_run1(d["nx"], d["ny"], d["dx"], d["dy"], d["H"], W, G, 0.9, 100)
    with O.wet_dry(H_DRY):
        wd, dts_w, st_w = O.grid_run1(d["nx"], d["ny"], d["dx"], d["dy"], d["H"], W, G, 0.9,
                                      100)
    assert st_p == st_w == O.OM_OK
    assert np.array_equal(dts_p, dts_w)
    for a, b in zip(plain, wd):
        assert np.array_equal(a, b)


def test_an_all_dry_domain_has_no_time_step():
    z = np.zeros(16)
    with O.wet_dry(H_DRY):
        W, dts, st = O.grid_run1(4, 4, 1.0, 1.0, z, [z, z, z, z], G, 0.9, 1)
    assert st == O.OM_ERR_NONFINITE


def test_the_flux_at_a_dry_bank_is_a_wall():
    # wet cell i (surface 0.5 above the reference) next to a dry cell whose
    # bed rises to 1.0: the edge passes no mass and the wet side feels the
    # hydrostatic wall pressure 1/2 g h^2 (water at rest)
    Wi = np.array([1.5, 0.0, 0.0, 0.3])
    Wj = np.array([0.0, 0.0, 0.0, 0.0])
    with O.wet_dry(H_DRY):
        F, D = O.flux1(Wi, Wj, 1.0, -1.0, (1.0, 0.0), G)
        Fj, Dj = O.flux1(Wj, Wi, -1.0, 1.0, (-1.0, 0.0), G)
    assert F[0] == 0.0 and F[3] == 0.0
    assert F[1] == pytest.approx(0.5 * G * 1.5 ** 2, rel=1e-15)
    assert D == pytest.approx(math.sqrt(G * 1.5), rel=1e-15)
    assert np.all(Fj == 0.0) and Dj == 0.0
    # the same dry cell below the wet surface is flooded: mass flows into it
    with O.wet_dry(H_DRY):
        F2, _ = O.flux1(Wi, Wj, 1.0, 0.8, (1.0, 0.0), G)
    assert F2[0] > 0.0
