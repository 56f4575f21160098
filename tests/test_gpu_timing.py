"""Per-kernel device timing through the C ABI (swe_set_timing /
swe_get_timing): every kernel of the handle's step is listed with its launch
count, the times are positive, and timing does not change any result."""
import numpy as np
import pytest

from finite_volume_shallow_gb300 import inputs as I
from finite_volume_shallow_gb300 import swe as S
from gpu_util import gpu_create, gpu_create2, gpu_create_mesh

pytestmark = pytest.mark.gpu


def run(make, steps, timed):
    s = make()
    if timed:
        S.swe_set_timing(s, True)
    S.swe_run(s, steps)
    S.swe_step(s, 0.9)
    W, t = S.swe_get_state(s)
    times = S.swe_get_timing(s)
    S.swe_destroy(s)
    return W, t, times


STEPS = 150   # more steps than the event ring holds
# launches per kernel over run(STEPS) + step(): a two-layer grid runs a
# flux pass, STEPS - 1 fused passes and an update, then flux + update for
# the lone step
EVERY = STEPS + 1


@pytest.mark.parametrize("case,kernels", [
    ("grid1", {"cart1_step_kernel": EVERY}),
    ("grid2", {"cart2_march_kernel<plain>": 2, "cart2_march_kernel<fused>": STEPS - 1,
               "cart2_update_kernel": 2}),
    ("mesh2", {"mesh_tile_kernel": EVERY, "mesh_update_kernel": EVERY}),
    ("mesh1", {"mesh_tile_kernel": EVERY, "mesh_update_kernel": EVERY}),
])
def test_kernel_times_listed_and_results_unchanged(case, kernels):
    if case == "grid1":
        d = I.make_workload("pulses8192", nx=300, ny=200)
        make = lambda: gpu_create(d, 32)
    elif case == "grid2":
        d = I.two_layer_hills(96, 64, umax=0.05, bump=0.5)
        make = lambda: gpu_create2(d, 32)
    elif case == "mesh2":
        d = I.tri_workload(48, sigma_scale=0.05, bump=1.0)
        make = lambda: gpu_create_mesh(d, 32)
    else:
        d = I.tri_workload1(40, 30)
        make = lambda: gpu_create_mesh(d, 64)
    Wa, ta, none = run(make, STEPS, False)
    Wb, tb, times = run(make, STEPS, True)
    assert none == {}
    assert list(times) == list(kernels)
    for name, (launches, ms) in times.items():
        assert launches == kernels[name], name
        assert ms > 0.0, name
    for x, y in zip(Wa, Wb):
        assert np.array_equal(x, y)
    assert ta == tb


def test_timing_restarts_from_zero_and_stops():
    d = I.tri_workload1(20, 20)
    s = gpu_create_mesh(d, 32)
    S.swe_set_timing(s, True)
    S.swe_run(s, 5)
    S.swe_set_timing(s, True)   # restart
    S.swe_run(s, 3)
    assert all(v[0] == 3 for v in S.swe_get_timing(s).values())
    S.swe_set_timing(s, False)
    S.swe_run(s, 4)
    assert all(v[0] == 3 for v in S.swe_get_timing(s).values())
    S.swe_destroy(s)
