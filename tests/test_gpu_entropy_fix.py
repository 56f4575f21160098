"""Parity of the step with the Harten-Hyman entropy fix switched on
(swe_params.entropy_fix = 1) against the oracle with its fix switched on, on
flows that have sonic points.  One layer: a transonic dam break (h_r / h_l = 0.05, the
fan crosses the critical speed at the dam), a strong radial dam break on a
grid and on triangles, and supercritical flow leaving a wall (the mirror
ghost then makes the fix act on the wall edges).  Tolerances as in the other parity
tests.  Also checks that the fix is what the kernel ran: the transonic result
differs from the plain scheme's by far more than rounding.
"""
import numpy as np
import pytest

from finite_volume_shallow_gb300 import inputs as I
from finite_volume_shallow_gb300 import swe as S
from gpu_util import (TOL, assert_parity, assert_parity2, assert_parity_mesh, gpu_create,
                      gpu_run, gpu_run2, np_dtype, rel_errors)

pytestmark = pytest.mark.gpu


def _transonic(nx=400):
    d = I.dam_break_1d(nx, h_left=10.0, h_right=0.5)
    d.update(g=9.81, cfl=0.9, entropy_fix=1)
    return d


@pytest.mark.parametrize("precision", [64, 32])
def test_transonic_dam_break(precision):
    assert_parity(_transonic(), precision, 150)


def test_fix_changes_the_transonic_solution():
    d = _transonic()
    Wf, _, _ = gpu_run(d, 64, 150)
    d0 = dict(d, entropy_fix=0)
    Wp, _, _ = gpu_run(d0, 64, 150)
    assert np.abs(Wf[0] - Wp[0]).max() > 1e-3 * np.abs(Wp[0]).max()


@pytest.mark.parametrize("precision", [64, 32])
def test_strong_radial_dam_break(precision):
    d = I.circular_dam(150, 70, dx=1.0, radius=18.0, h_in=10.0, h_out=0.5)
    d.update(g=9.81, cfl=0.9, entropy_fix=1)
    assert_parity(d, precision, 60)


@pytest.mark.parametrize("precision", [64, 32])
def test_strong_dam_break_on_anisotropic_cells(precision):
    # dx != dy runs the anisotropic variant of the step with the fix
    d = I.circular_dam(120, 64, dx=1.0, dy=2.5, radius=25.0, centre=(50.0, 70.0), h_in=10.0,
                       h_out=0.5)
    d.update(g=9.81, cfl=0.9, entropy_fix=1)
    assert_parity(d, precision, 60)


@pytest.mark.parametrize("precision", [64, 32])
def test_supercritical_departure_from_a_wall(precision):
    # u = 3.6 m/s > sqrt(g h) = 3.1 m/s leaving the left wall: against its
    # mirror ghost the 2-speed of the wall edge has spread delta = u > c, so
    # the fix acts on the wall edges (and only there: the interior flow is
    # uniform along x).  Roe's linearised middle state h (1 - u / c) is
    # negative here, so within a few steps the wall cells run dry; 4 steps
    # keep every depth above 0.1 m.
    import oracle as O

    nx, ny = 130, 70
    y = np.repeat((np.arange(ny) + 0.5)[:, None], nx, axis=1)
    h = 1.0 + 0.1 * np.sin(2 * np.pi * y / ny)
    z = np.zeros(nx * ny)
    d = dict(nx=nx, ny=ny, dx=1.0, dy=1.0, H=z, h=h.reshape(-1), qx=3.6 * h.reshape(-1),
             qy=(0.3 * np.cos(2 * np.pi * y / ny) * h).reshape(-1),
             hC=((np.arange(nx)[None, :] % 7 == 0) * h).reshape(-1), g=9.81, cfl=0.9,
             entropy_fix=1)
    runs = []
    for fix in (0, 1):
        with O.entropy_fix(fix):
            W, _, st = O.grid_run1(nx, ny, 1.0, 1.0, z, I.fields_of(d), 9.81, 0.9, 4)
        assert st == O.OM_OK
        runs.append(W[0].reshape(ny, nx))
    assert np.abs(runs[0] - runs[1])[:, 0].max() > 1e-2   # the wall edges are fixed
    assert_parity(d, precision, 4)


@pytest.mark.parametrize("precision", [64, 32])
def test_strong_dam_break_on_triangles(precision):
    xy, tri = I.square_tri_mesh(40, 30, jitter=0.2, seed=77)
    c = I.tri_centroids(xy, tri)
    inside = (c[:, 0] - 20.0) ** 2 + (c[:, 1] - 15.0) ** 2 < 8.0 ** 2
    h = np.where(inside, 10.0, 0.5)
    z = np.zeros_like(h)
    d = dict(xy=xy, tri=tri, n_cells=tri.shape[0], n_layers=1, mesh=True, g=9.81, cfl=0.9,
             H=z, h=h, qx=z.copy(), qy=z.copy(), hC=h * inside, entropy_fix=1)
    assert_parity_mesh(d, precision, 60)


@pytest.mark.parametrize("precision", [32, 64])
def test_fix_through_the_no_alloc_entry_point(precision):
    import torch

    d = _transonic(260)
    nx, ny = d["nx"], d["ny"]
    npdt = np_dtype(precision)
    tdt = torch.float32 if precision == 32 else torch.float64
    pitch = S.noalloc_pitch(nx)

    def padded(values):
        t = torch.zeros(((ny + 4) * pitch,), dtype=tdt, device="cuda")
        if values is not None:
            t.view(ny + 4, pitch)[2:ny + 2, 2:nx + 2] = torch.from_numpy(
                values.astype(npdt).reshape(ny, nx)).to("cuda")
        return t

    H = padded(d["H"])
    Wa = [padded(f) for f in I.fields_of(d)]
    Wb = [padded(None) for _ in range(4)]
    torch.cuda.synchronize()
    dts = S.swe_run_noalloc(nx, ny, d["dx"], d["dy"], H.data_ptr(), [w.data_ptr() for w in Wa],
                            [w.data_ptr() for w in Wb], pitch, 90, precision=precision,
                            g=d["g"], cfl=d["cfl"], entropy_fix=1)
    ref = gpu_create(d, precision)
    S.swe_run(ref, 90)
    W_ref, _ = S.swe_get_state(ref)
    dts_ref = S.swe_get_dt_history(ref, 90)
    S.swe_destroy(ref)
    W = [w.view(ny + 4, pitch)[2:ny + 2, 2:nx + 2].cpu().numpy().reshape(-1).astype(np.float64)
         for w in Wa]
    errs = rel_errors(W, [w.astype(np.float64) for w in W_ref], I.fields_of(d))
    for k in ("h", "qx", "qy", "hC"):
        assert errs[k] <= TOL[precision][k], errs
    assert np.abs(dts / dts_ref - 1.0).max() <= TOL[precision]["dt"]


# ---- two layers: a transonic dam break in the lower layer under a thick
# upper layer with a flat surface (the fix acts on the lower layer's waves) --
def _two_layer_dam(d, r, upper=60.0):
    h2 = d["h"]
    z = np.zeros(h2.size)
    out = dict(nx=d["nx"], ny=d["ny"], dx=d["dx"], dy=d["dy"], H=d["H"], r=r, n_layers=2,
               g=9.81, cfl=0.9, entropy_fix=1)
    for k, v in (("h1", upper - h2), ("q1x", z), ("q1y", z), ("h2", h2), ("q2x", z),
                 ("q2y", z)):
        out[k] = np.ascontiguousarray(v, dtype=np.float64)
    return out


@pytest.mark.parametrize("precision", [64, 32])
def test_two_layer_transonic_dam_break(precision):
    d = _two_layer_dam(I.dam_break_1d(160, ny=6, h_left=10.0, h_right=0.5), r=0.3)
    assert_parity2(d, precision, 60)


def test_two_layer_fix_changes_the_solution():
    d = _two_layer_dam(I.dam_break_1d(160, ny=6, h_left=10.0, h_right=0.5), r=0.3)
    Wf, _, _ = gpu_run2(d, 64, 60)
    Wp, _, _ = gpu_run2(dict(d, entropy_fix=0), 64, 60)
    assert np.abs(Wf[3] - Wp[3]).max() > 0.1


@pytest.mark.parametrize("precision", [64, 32])
def test_two_layer_radial_dam_break_on_anisotropic_cells(precision):
    d = _two_layer_dam(I.circular_dam(60, 40, dx=5.0, dy=8.0, radius=70.0, h_in=10.0,
                                      h_out=0.5), r=0.5, upper=30.0)
    assert_parity2(d, precision, 40)


@pytest.mark.parametrize("precision", [64, 32])
def test_two_layer_dam_break_on_triangles(precision):
    xy, tri = I.square_tri_mesh(40, 30, jitter=0.2, seed=78)
    c = I.tri_centroids(xy, tri)
    inside = (c[:, 0] - 20.0) ** 2 + (c[:, 1] - 15.0) ** 2 < 8.0 ** 2
    h2 = np.where(inside, 10.0, 0.5)
    z = np.zeros_like(h2)
    d = dict(xy=xy, tri=tri, n_cells=tri.shape[0], n_layers=2, mesh=True, g=9.81, cfl=0.9,
             r=0.5, H=z, h1=30.0 - h2, q1x=z, q1y=z, h2=h2, q2x=z.copy(), q2y=z.copy(),
             entropy_fix=1)
    assert_parity_mesh(d, precision, 40)
