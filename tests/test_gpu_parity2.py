"""Two-layer step on the GPU (through the C ABI) against the two-layer oracle
(An MPI-CUDA implementation of an improved Roe method for two-layer shallow
water systems, Sec. 2.2 with the 4x4 Roe matrix), same seeded inputs,
element by element; plus the properties that hold at any size, on the
2048 x 2048 interface dam break itself.

Tolerances as for one layer: fp64 <= 1e-10 per field and dt <= 1e-12; fp32
<= 1e-4 on depths, <= 1e-3 on discharges, dt <= 1e-6 (relative to each
field's scale).
"""
import numpy as np
import pytest

import oracle as O
from finite_volume_shallow_gb300 import inputs as I
from finite_volume_shallow_gb300 import swe as S
from gpu_util import (TOL2, assert_parity2, gpu_create2, gpu_run2, np_dtype, oracle_run2,
                      rel_errors2)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("precision", [64, 32])
@pytest.mark.parametrize("nx,ny", [(96, 20), (70, 33)])
def test_interface_dam_break(precision, nx, ny):
    d = I.make_workload("interface2048", nx=nx, ny=ny)
    assert_parity2(d, precision, 40)


@pytest.mark.parametrize("precision", [64, 32])
def test_moving_layers_over_hills(precision):
    d = I.two_layer_hills(53, 41, umax=0.05, bump=0.5)
    assert_parity2(d, precision, 30)


@pytest.mark.parametrize("precision", [64, 32])
@pytest.mark.parametrize("r", [0.01, 0.1])
def test_small_density_ratio_near_double_roots(precision, r):
    """Layers of nearly equal depth at a small density ratio: u1 + c1 and
    u2 + c2 nearly coincide, so the two largest eigenvalues of A_ij sit close
    together, where the outer Newton iteration converges slowly."""
    d = I.two_layer_hills(41, 29, interface_depth=6.5, umax=0.05, bump=0.3, r=r)
    c1 = np.sqrt(9.81 * d["h1"])
    c2 = np.sqrt(9.81 * d["h2"])
    assert np.min(np.abs(c1 - c2) / c1) < 1e-2
    assert_parity2(d, precision, 20)


@pytest.mark.parametrize("precision", [64, 32])
@pytest.mark.parametrize("nx,ny", [(1, 1), (1, 7), (7, 1), (33, 9), (32, 8), (31, 5)])
def test_small_and_ragged_grids(precision, nx, ny):
    d = I.two_layer_hills(nx, ny, umax=0.05, bump=0.3)
    assert_parity2(d, precision, 12)


def test_anisotropic_cells():
    d = I.two_layer_hills(45, 26, umax=0.05, bump=0.5)
    d["dy"] = 25.0
    assert_parity2(d, 64, 20)


def test_two_layer_lake_at_rest():
    d = I.two_layer_hills(300, 200)
    W, _, _ = gpu_run2(d, 64, 100)
    for i, k in ((0, "h1"), (3, "h2")):
        assert np.abs(W[i] - d[k]).max() <= 1e-13 * d[k].max()
    qs = d["h2"].max() * np.sqrt(9.81 * d["h2"].max())
    for i in (1, 2, 4, 5):
        assert np.abs(W[i]).max() <= 1e-13 * qs


@pytest.mark.parametrize("precision", [64, 32])
def test_full_size_interface_dam_rows_match_strip(precision):
    # the 2048^2 interface dam break is y-invariant with walls: every row of
    # the full grid must equal the oracle on a walled 2048 x 4 strip, over the
    # workload's own 500 steps
    d = I.make_workload("interface2048")
    steps = d["steps"]
    assert steps == 500
    Wg, dtg, _ = gpu_run2(d, precision, steps)
    strip = I.make_workload("interface2048", ny=4)
    Wo, dto = oracle_run2(strip, precision, steps)
    tol = TOL2[precision]
    for i, k in enumerate(I.TWO_LAYER_FIELDS):
        rows = Wg[i].reshape(2048, 2048)
        ref = Wo[i].reshape(4, 2048)[0]
        scale = max(np.abs(ref).max(), np.abs(d[k]).max())
        assert np.abs(rows - ref[None, :]).max() <= tol[k] * scale, k
    assert np.abs(dtg / dto - 1).max() <= tol["dt"]
    # layer masses conserved over the full grid
    for i, k in ((0, "h1"), (3, "h2")):
        assert abs(Wg[i].sum() - d[k].astype(np_dtype(precision)).astype(np.float64).sum()) \
            / d[k].sum() <= (1e-12 if precision == 64 else 2e-6)


def test_loss_of_hyperbolicity_is_reported():
    # opposite currents in the two layers, strong enough to make the inner
    # eigenvalues of the Roe matrix complex
    nx, ny = 40, 8
    d = I.interface_dam(nx, ny)
    d["h1"] = np.full(nx * ny, 3.0)
    d["h2"] = np.full(nx * ny, 7.0)
    d["q1x"] = 3.0 * 2.0 * np.ones(nx * ny)
    d["q2x"] = -7.0 * 2.0 * np.ones(nx * ny)
    s = gpu_create2(d, 64)
    with pytest.raises(S.SweError) as e:
        S.swe_step(s, 0.9)
    assert e.value.status == S.SWE_ERR_HYPERBOLIC
    # the error is sticky
    with pytest.raises(S.SweError):
        S.swe_run(s, 1)


def test_two_layer_restart_and_history():
    d = I.two_layer_hills(64, 48, umax=0.05, bump=0.5)
    a = gpu_create2(d, 32)
    S.swe_run(a, 30)
    Wa, ta = S.swe_get_state(a)
    b = gpu_create2(d, 32)
    S.swe_run(b, 12)
    Wm, tm = S.swe_get_state(b)
    S.swe_set_state(b, Wm, tm)
    S.swe_run(b, 18)
    Wb, tb = S.swe_get_state(b)
    for x, y in zip(Wa, Wb):
        assert np.array_equal(x, y)
    assert len(S.swe_get_dt_history(a)) == 30
    info = S.swe_get_info(a)
    assert info["n_layers"] == 2 and info["steps"] == 30


@pytest.mark.parametrize("precision", [32, 64])
def test_fused_run_equals_single_steps(precision):
    """A run applies each step's update inside the next step's flux pass;
    steps taken one call at a time apply it in a separate pass.  Both round
    the same way: states, clocks and dt histories agree bit for bit, also for
    a run split into pieces."""
    d = I.two_layer_hills(72, 40, umax=0.05, bump=0.5)
    a = gpu_create2(d, precision)
    S.swe_run(a, 17)
    b = gpu_create2(d, precision)
    for _ in range(17):
        S.swe_step(b, d.get("cfl", 0.9))
    c = gpu_create2(d, precision)
    for n in (2, 1, 5, 9):
        S.swe_run(c, n)
    (Wa, ta), (Wb, tb), (Wc, tc) = (S.swe_get_state(x) for x in (a, b, c))
    for x, y, z in zip(Wa, Wb, Wc):
        assert np.array_equal(x, y) and np.array_equal(x, z)
    assert ta == tb == tc
    ha, hb, hc = (S.swe_get_dt_history(x) for x in (a, b, c))
    assert len(ha) == 17 and np.array_equal(ha, hb) and np.array_equal(ha, hc)
    for x in (a, b, c):
        S.swe_destroy(x)


@pytest.mark.parametrize("precision", [64, 32])
def test_y_independent_state_stays_so_bitwise(precision):
    """The interface dam break does not depend on y, and neither does the
    scheme's answer: over hundreds of steps every row stays bitwise equal to
    the first and q_y exactly 0.  Each edge's Newton iteration stops on its
    own convergence, so identical edges give identical results whichever
    warp or tile evaluates them."""
    d = I.make_workload("interface2048", nx=200, ny=24)
    W, _, _ = gpu_run2(d, precision, 300)
    for k, w in zip(I.TWO_LAYER_FIELDS, W):
        rows = w.reshape(d["ny"], d["nx"])
        assert np.array_equal(rows, np.broadcast_to(rows[0], rows.shape)), k
    assert not W[2].any() and not W[5].any()


def test_two_layer_arguments():
    d = I.interface_dam(16, 8)
    with pytest.raises(S.SweError) as e:   # two layers carry no pollutant
        S.swe_create_grid(16, 8, 10.0, 10.0, d["H"], I.fields2_of(d), precision=64,
                          n_layers=2, pollutant=1, r=0.98)
    assert e.value.status == S.SWE_ERR_UNSUPPORTED
    with pytest.raises(S.SweError) as e:   # r must lie in [0, 1)
        S.swe_create_grid(16, 8, 10.0, 10.0, d["H"], I.fields2_of(d), precision=64,
                          n_layers=2, pollutant=0, r=1.0)
    assert e.value.status == S.SWE_ERR_ARG
    bad = dict(d)
    bad["h2"] = d["h2"].copy()
    bad["h2"][5] = -1.0
    with pytest.raises(S.SweError) as e:
        gpu_create2(bad, 64)
    assert e.value.status == S.SWE_ERR_ARG


@pytest.mark.parametrize("precision", [64, 32])
def test_cfl_limit_two_layers(precision):
    d = I.two_layer_hills(53, 41, umax=0.05, bump=0.5)
    d["cfl"] = 1.0
    assert_parity2(d, precision, 30)


def test_grid_taller_than_a_launch_dimension():
    # the march puts all its units in the launch's x dimension: a strip of
    # 530,000 rows (more than 65,535 blocks of 8 rows) runs and matches the
    # oracle
    d = I.two_layer_hills(2, 530_000, umax=0.05, bump=0.5)
    assert_parity2(d, 32, 3)


@pytest.mark.parametrize("precision", [32, 64])
@pytest.mark.parametrize("nx,ny", [(30, 17), (60, 9), (61, 23), (91, 40), (29, 70)])
def test_band_borders_of_the_march(precision, nx, ny):
    # widths at and around multiples of the march's 30-column bands: a band
    # whose halo lane sits on the east wall, a band with one column, and
    # row segments of a few rows each
    d = I.two_layer_hills(nx, ny, umax=0.05, bump=0.5)
    assert_parity2(d, precision, 15)
