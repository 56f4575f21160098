"""The workloads' own step counts, on reduced grids the oracle finishes in
seconds: the GPU stays within the stated tolerances of the fp64 oracle over
1000 steps (2048^2 hills recipe), 200 steps (8192^2 pulses recipe), 500
steps (two-layer interface dam break) and 500 steps (two-layer triangle
mesh), every step's dt included.  Runs go through swe_run, so the two-layer
grid runs take the fused update-and-flux pass."""
import numpy as np
import pytest

from finite_volume_shallow_gb300 import inputs as I
from gpu_util import (TOL, assert_parity_mesh, gpu_run, oracle_run, rel_errors,
                      assert_parity2)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("workload,nx,ny,precision,steps", [
    ("hills2048", 160, 128, 64, 1000),
    ("hills2048", 160, 128, 32, 1000),
    ("pulses8192", 384, 256, 32, 200),
])
def test_one_layer_grid_full_step_count(workload, nx, ny, precision, steps):
    d = I.make_workload(workload, nx=nx, ny=ny)
    Wg, dtg, tg = gpu_run(d, precision, steps, use_run=True)
    Wo, dto = oracle_run(d, precision, steps)
    tol = TOL[precision]
    errs = rel_errors(Wg, Wo, I.fields_of(d))
    for k in ("h", "qx", "qy", "hC"):
        assert errs[k] <= tol[k], (k, errs)
    assert len(dtg) == steps
    assert np.abs(dtg / dto - 1.0).max() <= tol["dt"]


@pytest.mark.parametrize("precision", [64, 32])
def test_two_layer_interface_full_step_count(precision):
    d = I.make_workload("interface2048", nx=64, ny=24)
    assert_parity2(d, precision, 500)


@pytest.mark.parametrize("precision", [32, 64])
def test_two_layer_triangles_full_step_count(precision):
    d = I.tri_workload(16, sigma_scale=0.05, bump=1.0)
    assert_parity_mesh(d, precision, 500)
