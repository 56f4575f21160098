"""swe_run_noalloc, the allocation-free entry point, against the handle API
and the oracle.

Some callers cannot allocate device memory once they are running (a framework
whose pool already owns the GPU's memory, a real-time loop that forbids
allocation); swe_run_noalloc runs the same step on buffers they own and keeps
its scratch in a static device array.  This test owns the buffers (torch
allocates them here, not the entry point), fills their padding with NaN to
show the padding never reaches a result, and checks two calls in a row against
swe_create_grid + swe_run + swe_get_state on the same inputs.  Both paths run
the same kernels with the same launch shape and the same order of wave-speed
slots, and a call that starts from a state computes its first dt exactly as a
running loop does, so the fields and the dt agree bit for bit.  The first call
is also checked against the oracle within the GPU parity tolerances, and a
warm call must leave the device's free memory unchanged.  It lives in the file
pytest collects last.
"""
import numpy as np
import pytest

from finite_volume_shallow_gb300 import inputs as I
from finite_volume_shallow_gb300 import swe as S
from gpu_util import TOL, gpu_create, np_dtype, oracle_run, rel_errors

pytestmark = pytest.mark.gpu


def _padded(torch, values, nx, ny, pitch, dtype):
    t = torch.full(((ny + 4) * pitch,), float("nan"), dtype=dtype, device="cuda")
    if values is not None:
        v = t.view(ny + 4, pitch)
        v[2:ny + 2, 2:nx + 2] = torch.from_numpy(values.reshape(ny, nx)).to("cuda")
    return t


def _interior(t, nx, ny, pitch):
    return t.view(ny + 4, pitch)[2:ny + 2, 2:nx + 2].cpu().numpy().reshape(-1)


@pytest.mark.parametrize("precision", [32, 64])
def test_noalloc_matches_handle_api(precision):
    import torch

    nx, ny = 190, 130
    d = I.make_workload("pulses8192", nx=nx, ny=ny)
    npdt = np_dtype(precision)
    tdt = torch.float32 if precision == 32 else torch.float64
    pitch = S.noalloc_pitch(nx)
    H = _padded(torch, d["H"].astype(npdt), nx, ny, pitch, tdt)
    Wa = [_padded(torch, f.astype(npdt), nx, ny, pitch, tdt) for f in I.fields_of(d)]
    Wb = [_padded(torch, None, nx, ny, pitch, tdt) for _ in range(4)]
    torch.cuda.synchronize()

    def call(nsteps):
        return S.swe_run_noalloc(nx, ny, d["dx"], d["dy"], H.data_ptr(),
                                 [w.data_ptr() for w in Wa], [w.data_ptr() for w in Wb], pitch,
                                 nsteps, precision=precision, g=d["g"], cfl=d["cfl"])

    ref = gpu_create(d, precision)
    start = [f.astype(np.float64) for f in I.fields_of(d)]
    for nsteps in (7, 12):  # two calls in a row: odd, then even step count
        free_before = torch.cuda.mem_get_info()[0]
        dts = call(nsteps)
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        if nsteps == 12:  # a warm call: the entry point allocated nothing
            assert free_after == free_before, (free_before, free_after)
        S.swe_run(ref, nsteps)
        W_ref, _ = S.swe_get_state(ref)
        dts_ref = S.swe_get_dt_history(ref, nsteps)
        W = [_interior(w, nx, ny, pitch) for w in Wa]
        assert len(dts) == nsteps
        assert np.array_equal(dts, dts_ref), (nsteps, dts, dts_ref)
        for k, (a, b) in enumerate(zip(W, W_ref)):
            assert np.array_equal(a, b), (nsteps, k, np.abs(a.astype(float) - b).max())
        assert all(np.isfinite(w).all() for w in W)
        if nsteps == 7:  # independent of the handle: the oracle on the same inputs
            Wo, dto = oracle_run(d, precision, nsteps)
            errs = rel_errors([w.astype(np.float64) for w in W], Wo, start)
            for k in ("h", "qx", "qy", "hC"):
                assert errs[k] <= TOL[precision][k], errs
            assert np.abs(dts / dto - 1.0).max() <= TOL[precision]["dt"]
    S.swe_destroy(ref)


def test_noalloc_rejects_more_steps_than_its_scratch_holds():
    import torch

    nx, ny = 64, 40
    pitch = S.noalloc_pitch(nx)
    bufs = [torch.zeros((ny + 4) * pitch, dtype=torch.float64, device="cuda") for _ in range(9)]
    with pytest.raises(S.SweError) as e:
        S.swe_run_noalloc(nx, ny, 1.0, 1.0, bufs[0].data_ptr(), [b.data_ptr() for b in bufs[1:5]],
                          [b.data_ptr() for b in bufs[5:9]], pitch, S.NOALLOC_MAX_STEPS + 1)
    assert e.value.status == S.SWE_ERR_ARG
