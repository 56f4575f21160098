"""libswe loads and exports every function that include/*.h declares, and
rejects bad arguments before it touches the GPU (no compute calls here)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from finite_volume_shallow_gb300 import build as B
from finite_volume_shallow_gb300 import swe as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(swe_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    B.build()
    return S.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("swe_create_grid", "swe_step", "swe_run", "swe_get_state", "swe_set_state",
                 "swe_get_dt_history", "swe_get_info", "swe_device_fields", "swe_destroy",
                 "swe_status_str", "swe_run_noalloc", "swe_probe_fma_rate"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    handle = C.CDLL(B.LIB)
    for name in declared_functions():
        assert hasattr(handle, name), name


def test_library_is_for_sm103a():
    out = open(B.LIB, "rb").read()
    assert b"sm_103a" in out or b"sm_103" in out


def test_status_strings(lib):
    for code in range(-8, 1):
        s = S.swe_status_str(code)
        assert isinstance(s, str) and s and s != "unknown status"
    assert S.swe_status_str(-99) == "unknown status"


def _grid(nx=4, ny=3, dx=1.0, dy=1.0):
    return S._Grid(nx, ny, dx, dy)


def _params(**kw):
    p = dict(n_layers=1, precision=64, pollutant=1, g=9.81, r=0.0, cfl=0.9, stream=None,
             entropy_fix=0, wet_dry=0, h_dry=0.0)
    p.update(kw)
    return S._Params(p["n_layers"], p["precision"], p["pollutant"], p["g"], p["r"], p["cfl"],
                     p["stream"], p["entropy_fix"], p["wet_dry"], p["h_dry"])


def _create(lib, grid, params, n=12, with_fields=True):
    H = np.zeros(n)
    W = [np.ones(n), np.zeros(n), np.zeros(n), np.zeros(n)]
    Wp = (C.c_void_p * 4)(*[w.ctypes.data for w in W]) if with_fields else None
    out = C.c_void_p(123)
    st = lib.swe_create_grid(C.byref(grid) if grid is not None else None,
                             C.c_void_p(H.ctypes.data), Wp,
                             C.byref(params) if params is not None else None, C.byref(out))
    return st, out.value


@pytest.mark.parametrize("grid,params,expect", [
    (None, _params(), S.SWE_ERR_ARG),
    (_grid(), None, S.SWE_ERR_ARG),
    (_grid(nx=0), _params(), S.SWE_ERR_ARG),
    (_grid(ny=-3), _params(), S.SWE_ERR_ARG),
    (_grid(dx=0.0), _params(), S.SWE_ERR_ARG),
    (_grid(dy=float("nan")), _params(), S.SWE_ERR_ARG),
    (_grid(), _params(precision=16), S.SWE_ERR_ARG),
    (_grid(), _params(g=-1.0), S.SWE_ERR_ARG),
    (_grid(), _params(cfl=0.0), S.SWE_ERR_ARG),
    (_grid(), _params(cfl=1.5), S.SWE_ERR_ARG),
    (_grid(), _params(n_layers=3), S.SWE_ERR_ARG),
    (_grid(), _params(n_layers=2), S.SWE_ERR_UNSUPPORTED),
    (_grid(), _params(pollutant=0), S.SWE_ERR_UNSUPPORTED),
    (_grid(), _params(entropy_fix=2), S.SWE_ERR_ARG),
    (_grid(), _params(entropy_fix=-1), S.SWE_ERR_ARG),
    (_grid(), _params(n_layers=2, pollutant=0, r=0.5, entropy_fix=2), S.SWE_ERR_ARG),
    (_grid(), _params(wet_dry=2, h_dry=1e-4), S.SWE_ERR_ARG),
    (_grid(), _params(wet_dry=1, h_dry=-1e-4), S.SWE_ERR_ARG),
    (_grid(), _params(wet_dry=1, h_dry=float("nan")), S.SWE_ERR_ARG),
    (_grid(), _params(wet_dry=1, h_dry=float("inf")), S.SWE_ERR_ARG),
    (_grid(), _params(n_layers=2, pollutant=0, r=0.5, wet_dry=1, h_dry=1e-4),
     S.SWE_ERR_UNSUPPORTED),
    (_grid(ny=524281), _params(wet_dry=1, h_dry=1e-4), S.SWE_ERR_ARG),
])
def test_create_rejects_bad_arguments(lib, grid, params, expect):
    st, out = _create(lib, grid, params)
    assert st == expect
    assert out is None   # *out is cleared on failure


def test_create_rejects_missing_fields(lib):
    st, out = _create(lib, _grid(), _params(), with_fields=False)
    assert st == S.SWE_ERR_ARG and out is None


def test_null_handles(lib):
    lib.swe_destroy(None)
    assert lib.swe_step(None, C.c_double(0.9), None) == S.SWE_ERR_ARG
    assert lib.swe_run(None, 1) == S.SWE_ERR_ARG
    assert lib.swe_get_state(None, None, None) == S.SWE_ERR_ARG
    assert lib.swe_set_state(None, None, C.c_double(0.0)) == S.SWE_ERR_ARG
    n = C.c_int64()
    assert lib.swe_get_dt_history(None, None, 0, C.byref(n)) == S.SWE_ERR_ARG
    assert lib.swe_get_info(None, None) == S.SWE_ERR_ARG
    assert lib.swe_device_fields(None, None) == S.SWE_ERR_ARG


def test_binding_checks_host_arrays(lib):
    with pytest.raises(ValueError):
        S._host_ptr(np.zeros(5, dtype=np.float32), np.float64, 5)
    with pytest.raises(ValueError):
        S._host_ptr(np.zeros(6), np.float64, 5)
    with pytest.raises(ValueError):
        S._host_ptr(np.zeros((4, 4))[:, 0], np.float64, 4)


def test_noalloc_rejects_bad_arguments_before_touching_the_gpu(lib):
    # arguments are checked before any CUDA call (fake, aligned addresses)
    fake = [0x10000 * (k + 1) for k in range(9)]
    ok = dict(nx=64, ny=40, dx=1.0, dy=1.0, H=fake[0], W_a=fake[1:5], W_b=fake[5:9],
              pitch=S.noalloc_pitch(64), nsteps=3)
    cases = [dict(nsteps=S.NOALLOC_MAX_STEPS + 1), dict(nsteps=-1), dict(pitch=32),
             dict(pitch=S.noalloc_pitch(64) + 8), dict(H=fake[0] + 4), dict(nx=0),
             dict(dx=0.0)]
    for bad in cases:
        a = dict(ok, **bad)
        with pytest.raises(S.SweError) as e:
            S.swe_run_noalloc(a["nx"], a["ny"], a["dx"], a["dy"], a["H"], a["W_a"], a["W_b"],
                              a["pitch"], a["nsteps"])
        assert e.value.status == S.SWE_ERR_ARG, bad
    with pytest.raises(S.SweError) as e:
        S.swe_run_noalloc(64, 40, 1.0, 1.0, fake[0], fake[1:5], fake[5:9], S.noalloc_pitch(64), 3,
                          precision=16)
    assert e.value.status == S.SWE_ERR_ARG
    with pytest.raises(S.SweError) as e:
        S.swe_run_noalloc(64, 40, 1.0, 1.0, fake[0], fake[1:5], fake[5:9], S.noalloc_pitch(64), 3,
                          entropy_fix=3)
    assert e.value.status == S.SWE_ERR_ARG
    # the layer count and the pollutant switch, straight through the C ABI:
    # two layers or no pollutant are unsupported, any other count is invalid
    import ctypes as C
    grid = S._Grid(64, 40, 1.0, 1.0)
    wa = (C.c_void_p * 4)(*fake[1:5])
    wb = (C.c_void_p * 4)(*fake[5:9])
    for layers, pollutant, want in ((2, 1, S.SWE_ERR_UNSUPPORTED), (1, 0, S.SWE_ERR_UNSUPPORTED),
                                    (0, 1, S.SWE_ERR_ARG), (3, 1, S.SWE_ERR_ARG)):
        params = S._Params(layers, 64, pollutant, 9.81, 0.0, 0.9, None, 0)
        got = lib.swe_run_noalloc(C.byref(grid), C.byref(params), C.c_void_p(fake[0]), wa, wb,
                                  S.noalloc_pitch(64), 3, None)
        assert got == want, (layers, pollutant, got)


def test_wait_selftest_rejects_bad_budgets_before_touching_the_gpu(lib):
    for budget in (0, -5, 4_000_000_001):
        assert S.swe_selftest_wait(budget) == S.SWE_ERR_ARG


def test_missing_library_fails_loudly(lib, monkeypatch):
    # the binding never falls back to anything else when libswe is absent
    monkeypatch.setattr(B, "LIB", os.path.join(ROOT, "no_such_dir", "libswe.so"))
    monkeypatch.setattr(S, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        S.load(build_if_needed=False)


def test_valid_create_without_a_gpu_is_a_cuda_error(lib):
    # no CPU path: on a machine without a GPU a valid request fails with
    # SWE_ERR_CUDA instead of computing anything
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, out = _create(lib, _grid(), _params())
    assert st == S.SWE_ERR_CUDA and out is None


def test_mesh_has_no_wet_dry_treatment(lib):
    # refused before the mesh is prepared or any CUDA call
    xy = np.array([0.0, 0.0, 1.0, 0.0, 0.0, 1.0])
    tri = np.array([0, 1, 2], dtype=np.int32)
    mesh = S._Mesh(3, xy.ctypes.data, 1, tri.ctypes.data, 1)
    W = [np.ones(1), np.zeros(1), np.zeros(1), np.zeros(1)]
    Wp = (C.c_void_p * 4)(*[w.ctypes.data for w in W])
    H = np.zeros(1)
    out = C.c_void_p(123)
    st = lib.swe_create_mesh(C.byref(mesh), C.c_void_p(H.ctypes.data), Wp,
                             C.byref(_params(wet_dry=1, h_dry=1e-4)), C.byref(out))
    assert st == S.SWE_ERR_UNSUPPORTED and out.value is None
