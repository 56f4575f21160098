"""Properties the scheme guarantees at any size, checked on the CUDA path
(through the C ABI), including full-size grids in the launch configuration
the bench times, plus the API's restart, history, stream and error paths."""
import time

import numpy as np
import pytest

import oracle as O
from finite_volume_shallow_gb300 import inputs as I
from finite_volume_shallow_gb300 import swe as S
from gpu_util import TOL, gpu_create, gpu_run, np_dtype, oracle_run, rel_errors

pytestmark = pytest.mark.gpu


def test_lake_at_rest_fp64_full_hills2048():
    # well-balanced (C-property): water at rest over the 2048^2 hills
    d = I.make_workload("hills2048", lake_at_rest=True)
    W, dts, _ = gpu_run(d, 64, 100, use_run=True)
    scale = d["h"].max()
    assert np.abs(W[0] - d["h"]).max() <= 1e-13 * scale
    qs = scale * np.sqrt(9.81 * scale)
    assert np.abs(W[1]).max() <= 1e-13 * qs and np.abs(W[2]).max() <= 1e-13 * qs


def test_lake_at_rest_fp32_matches_oracle():
    # in fp32 the rounded inputs are not exactly at rest; the GPU must follow
    # the oracle started from the same rounded values, and stay near rest
    d = I.make_workload("hills2048", nx=256, ny=200, lake_at_rest=True)
    Wg, _, _ = gpu_run(d, 32, 100)
    Wo, _ = oracle_run(d, 32, 100)
    assert np.abs(Wg[0] - Wo[0]).max() <= 1e-5 * d["h"].max()
    assert np.abs(Wg[0] - d["h"]).max() <= 1e-5 * d["h"].max()


@pytest.mark.parametrize("precision,tol", [(64, 1e-12), (32, 2e-6)])
def test_conservation(precision, tol):
    d = I.make_workload("pulses8192", nx=512, ny=384)
    W, _, _ = gpu_run(d, precision, 500, use_run=True)
    dr = I.rounded(d, np_dtype(precision))
    for k, name in ((0, "h"), (3, "hC")):
        m0 = dr[name].sum()
        assert abs(W[k].sum() - m0) / m0 <= tol, name


def test_constant_concentration():
    d = I.make_workload("pulses8192", nx=300, ny=260)
    d["hC"] = 0.37 * d["h"]
    W, _, _ = gpu_run(d, 64, 200, use_run=True)
    assert np.abs(W[3] / W[0] - 0.37).max() <= 1e-14


def test_radial_dam_symmetry():
    d = I.make_workload("dam128")
    W, _, _ = gpu_run(d, 64, 100)
    h, qx, qy, hC = (w.reshape(128, 128) for w in W)
    assert np.abs(h - h.T).max() <= 1e-12 and np.abs(qx - qy.T).max() <= 1e-12
    assert np.abs(h - h[:, ::-1]).max() <= 1e-12 and np.abs(qx + qx[:, ::-1]).max() <= 1e-12
    assert np.abs(h - h[::-1, :]).max() <= 1e-12 and np.abs(qy + qy[::-1, :]).max() <= 1e-12


@pytest.mark.parametrize("precision", [64, 32])
def test_restart_is_bitwise(precision):
    d = I.make_workload("pulses8192", nx=300, ny=200)
    a = gpu_create(d, precision)
    S.swe_run(a, 100)
    Wa, ta = S.swe_get_state(a)
    b = gpu_create(d, precision)
    S.swe_run(b, 50)
    Wm, tm = S.swe_get_state(b)
    c = gpu_create(d, precision)           # a fresh handle resumed from the checkpoint
    S.swe_set_state(c, Wm, tm)
    S.swe_run(c, 50)
    Wc, tc = S.swe_get_state(c)
    for x, y in zip(Wa, Wc):
        assert np.array_equal(x, y)
    assert ta == tc
    ha = S.swe_get_dt_history(a)
    hb = np.concatenate([S.swe_get_dt_history(b), S.swe_get_dt_history(c)])
    assert np.array_equal(ha, hb)


def test_dt_history_matches_steps():
    d = I.make_workload("pulses8192", nx=200, ny=90)
    s = gpu_create(d, 64)
    dts = [S.swe_step(s, 0.9) for _ in range(25)]
    h = S.swe_get_dt_history(s)
    assert np.array_equal(h, np.array(dts))
    assert np.array_equal(S.swe_get_dt_history(s, 5), np.array(dts[-5:]))
    info = S.swe_get_info(s)
    assert info["steps"] == 25 and info["t"] == pytest.approx(sum(dts), rel=1e-14)
    assert info["bands"] >= 1 and info["segments"] >= 1


def test_step_cfl_argument():
    # swe_step's cfl scales dt of that step (eq. (5) is linear in gamma)
    d = I.make_workload("pulses8192", nx=100, ny=80)
    a, b = gpu_create(d, 64), gpu_create(d, 64)
    assert S.swe_step(a, 0.5) == pytest.approx(0.5 * S.swe_step(b, 1.0), rel=1e-15)


def test_user_stream():
    import torch
    d = I.make_workload("pulses8192", nx=260, ny=130)
    ref, _, _ = gpu_run(d, 32, 30, use_run=True)
    stream = torch.cuda.Stream()
    s = gpu_create(d, 32, stream=stream.cuda_stream)
    S.swe_run(s, 30)
    W, _ = S.swe_get_state(s)
    for x, y in zip(ref, W):
        assert np.array_equal(x, y.astype(np.float64))


@pytest.mark.parametrize("kind", ["grid2", "mesh2", "mesh1"])
def test_user_stream_two_layers_and_meshes(kind):
    """The fused two-layer passes and the mesh passes (chained by
    programmatic dependent launch) on a caller's stream give the default
    stream's results bit for bit, also with work queued on the stream ahead
    of them."""
    import torch
    from gpu_util import gpu_create2, gpu_create_mesh
    if kind == "grid2":
        d = I.two_layer_hills(70, 44, umax=0.05, bump=0.5)
        make = lambda st: gpu_create2(d, 32, stream=st)
    elif kind == "mesh2":
        d = I.tri_workload(20, sigma_scale=0.05, bump=1.0)
        make = lambda st: gpu_create_mesh(d, 32, stream=st)
    else:
        d = I.tri_workload1(24, 18, seed=3)
        make = lambda st: gpu_create_mesh(d, 64, stream=st)
    a = make(None)
    S.swe_run(a, 25)
    ref, ta = S.swe_get_state(a)
    stream = torch.cuda.Stream()
    b = make(stream.cuda_stream)
    with torch.cuda.stream(stream):
        x = torch.ones(1 << 22, device="cuda")
        for _ in range(20):   # keep the stream busy when the steps are queued
            x = x * 1.0000001
    S.swe_run(b, 25)
    W, tb = S.swe_get_state(b)
    for u, v in zip(ref, W):
        assert np.array_equal(u, v)
    assert ta == tb
    S.swe_destroy(a)
    S.swe_destroy(b)


def test_pinned_torch_buffers():
    import torch
    d = I.make_workload("pulses8192", nx=190, ny=70)
    n = d["nx"] * d["ny"]
    s = gpu_create(d, 32)
    S.swe_run(s, 10)
    out = [torch.empty(n, dtype=torch.float32).pin_memory() for _ in range(4)]
    S.swe_get_state(s, out=out)
    W, _ = S.swe_get_state(s)
    for a, b in zip(out, W):
        assert np.array_equal(a.numpy(), b)
    S.swe_set_state(s, out, 1.0)
    assert S.swe_get_info(s)["t"] == 1.0


def test_bad_initial_state_rejected():
    d = I.make_workload("pulses8192", nx=64, ny=64)
    bad = dict(d)
    bad["h"] = d["h"].copy()
    bad["h"][100] = 0.0
    with pytest.raises(S.SweError) as e:
        gpu_create(bad, 64)
    assert e.value.status == S.SWE_ERR_ARG
    bad["h"] = d["h"].copy()
    bad["qx"] = d["qx"].copy()
    bad["qx"][7] = np.nan
    with pytest.raises(S.SweError) as e:
        gpu_create(bad, 32)
    assert e.value.status == S.SWE_ERR_ARG


@pytest.mark.parametrize("precision", [64, 32])
def test_drying_is_reported_and_sticky(precision):
    # a thin sheet of water pulled apart by a strong outflow dries out
    nx, ny = 40, 20
    h = np.full(nx * ny, 0.01)
    qx = np.where(np.arange(nx * ny) % nx < nx // 2, -0.5, 0.5)
    d = dict(nx=nx, ny=ny, dx=1.0, dy=1.0, g=9.81, cfl=0.9, H=np.zeros(nx * ny), h=h,
             qx=qx, qy=np.zeros(nx * ny), hC=np.zeros(nx * ny))
    s = gpu_create(d, precision)
    with pytest.raises(S.SweError) as e:
        for _ in range(50):
            S.swe_step(s, 0.9)
    assert e.value.status in (S.SWE_ERR_DEPTH, S.SWE_ERR_NONFINITE)
    with pytest.raises(S.SweError) as e2:
        S.swe_run(s, 1)
    assert e2.value.status == e.value.status
    # a new state clears the error
    good = I.make_workload("pulses8192", nx=nx, ny=ny)
    S.swe_set_state(s, [f.astype(np_dtype(precision)) for f in I.fields_of(good)], 0.0)
    S.swe_run(s, 5)


def test_fullsize_pulses8192_first_steps():
    # the 8192^2 fp32 workload in the bench's launch configuration: the first
    # two dt and every cell after one step against the oracle, which runs on
    # the full grid (mesh-free entry points)
    d = I.make_workload("pulses8192")
    s = gpu_create(d, 32)
    dt0 = S.swe_step(s, d["cfl"])
    W1, _ = S.swe_get_state(s)
    dt1 = S.swe_step(s, d["cfl"])
    S.swe_destroy(s)
    dr = I.rounded(d, np.float32)
    Wo = I.fields_of(dr)
    del d
    odt0 = O.grid_dt1(8192, 8192, 10.0, 10.0, dr["H"], Wo, 9.81, 0.9)
    assert abs(dt0 / odt0 - 1) <= TOL[32]["dt"]
    Wo1, st = O.grid_update1(8192, 8192, 10.0, 10.0, dr["H"], Wo, 9.81, odt0)
    assert st == O.OM_OK
    errs = rel_errors([w.astype(np.float64) for w in W1], Wo1)
    for k in ("h", "qx", "qy", "hC"):
        assert errs[k] <= TOL[32][k], errs
    odt1 = O.grid_dt1(8192, 8192, 10.0, 10.0, dr["H"], Wo1, 9.81, 0.9)
    assert abs(dt1 / odt1 - 1) <= TOL[32]["dt"]


@pytest.mark.parametrize("precision", [32, 64])
def test_fullsize_hills2048_one_step(precision):
    d = I.make_workload("hills2048")
    s = gpu_create(d, precision)
    dt0 = S.swe_step(s, d["cfl"])
    W1, _ = S.swe_get_state(s)
    S.swe_destroy(s)
    dr = I.rounded(d, np_dtype(precision)) if precision == 32 else d
    odt0 = O.grid_dt1(2048, 2048, 10.0, 10.0, dr["H"], I.fields_of(dr), 9.81, 0.9)
    assert abs(dt0 / odt0 - 1) <= TOL[precision]["dt"]
    Wo1, st = O.grid_update1(2048, 2048, 10.0, 10.0, dr["H"], I.fields_of(dr), 9.81, odt0)
    errs = rel_errors([w.astype(np.float64) for w in W1], Wo1)
    for k in ("h", "qx", "qy", "hC"):
        assert errs[k] <= TOL[precision][k], errs


def test_bounded_device_wait_gives_up_and_the_context_survives():
    """Failure detection without a GPU fault: the step kernel's bounded
    mbarrier wait, run on a barrier nothing arrives on, gives up after its
    budget and reports SWE_ERR_TIMEOUT; the context then runs steps as
    before."""
    t0 = time.perf_counter()
    assert S.swe_selftest_wait(20_000_000) == S.SWE_ERR_TIMEOUT  # ~10 ms of SM clock
    assert time.perf_counter() - t0 < 10.0
    d = I.make_workload("dam128", nx=48, ny=40)
    W, dts, _ = gpu_run(d, 64, 5)
    Wo, dto = oracle_run(d, 64, 5)
    assert max(rel_errors(W, Wo).values()) <= TOL[64]["h"]
    assert np.abs(dts / dto - 1).max() <= TOL[64]["dt"]
