"""Parity of the CUDA path (through the C ABI) with the fp64 oracle on the same
seeded inputs, element by element, on sizes that span several column bands
and row segments with ragged tails, plus the degenerate grids.

Tolerances: fp64 max relative error <= 1e-10 per field and dt <= 1e-12
relative; fp32 <= 1e-4 on h, <= 1e-3 on q and hC, dt <= 1e-6 relative.
"""
import numpy as np
import pytest

from finite_volume_shallow_gb300 import inputs as I
from gpu_util import assert_parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("precision", [64, 32])
def test_dam128_100_steps(precision):
    # the 128 x 128 circular dam break, 100 steps
    assert_parity(I.make_workload("dam128"), precision, 100)


@pytest.mark.parametrize("precision", [64, 32])
def test_dam128_through_swe_run(precision):
    assert_parity(I.make_workload("dam128"), precision, 60, use_run=True)


@pytest.mark.parametrize("precision", [64, 32])
@pytest.mark.parametrize("nx,ny", [(300, 97), (249, 130)])
def test_hills_ragged(precision, nx, ny):
    assert_parity(I.make_workload("hills2048", nx=nx, ny=ny), precision, 100)


@pytest.mark.parametrize("precision", [64, 32])
@pytest.mark.parametrize("nx,ny", [(251, 70), (130, 1000)])
def test_pulses_moving_water(precision, nx, ny):
    # random velocities; (130, 1000) cuts the rows into many segments
    assert_parity(I.make_workload("pulses8192", nx=nx, ny=ny), precision, 60)


@pytest.mark.parametrize("precision", [64, 32])
@pytest.mark.parametrize("extra", [0, 1, 2, 3])
def test_band_edges(precision, extra):
    # exactly one band (124 columns in fp32, 60 in fp64) and a few more, so
    # the last band owns 1-3 columns and the right wall sits in a halo
    own = 124 if precision == 32 else 60
    d = I.make_workload("pulses8192", nx=own + extra, ny=40)
    assert_parity(d, precision, 40)


@pytest.mark.parametrize("precision", [64, 32])
@pytest.mark.parametrize("nx,ny", [(1, 1), (1, 9), (9, 1), (2, 2), (3, 150), (150, 3), (5, 33)])
def test_degenerate_grids(precision, nx, ny):
    d = I.make_workload("pulses8192", nx=nx, ny=ny)
    assert_parity(d, precision, 30)


@pytest.mark.parametrize("precision", [64, 32])
def test_anisotropic_cells(precision):
    d = I.hills(77, 45, dx=10.0, dy=25.0, seed=77, umax=0.1)
    d.update(g=9.81, cfl=0.9)
    assert_parity(d, precision, 50)


@pytest.mark.parametrize("precision", [64, 32])
def test_dam_break_1d(precision):
    d = I.dam_break_1d(400)
    d.update(g=9.81, cfl=0.9)
    assert_parity(d, precision, 100)


def test_low_cfl():
    d = I.make_workload("pulses8192", nx=140, ny=60)
    d["cfl"] = 0.25
    assert_parity(d, 64, 40)


@pytest.mark.parametrize("precision", [64, 32])
def test_cfl_limit(precision):
    # gamma = 1, the largest value eq. (5) allows
    d = I.make_workload("pulses8192", nx=140, ny=60)
    d["cfl"] = 1.0
    assert_parity(d, precision, 60)
