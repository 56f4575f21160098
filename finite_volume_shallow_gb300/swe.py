"""Python binding of the libswe C ABI (include/swe.h): argument marshalling
only, the same names as the C functions.  Every step of the scheme runs in the
library's CUDA kernels; there is no CPU fallback: if the library cannot be
built or loaded, every call raises.

Host arrays may be numpy arrays or CPU torch tensors (pinned or not) of the
state's precision (float32 for precision 32, float64 for 64), each holding
nx*ny values in row-major (x fastest) order on a grid, or one value per
triangle in the caller's numbering on a mesh.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

SWE_OK = 0
SWE_ERR_ARG = -1
SWE_ERR_CUDA = -2
SWE_ERR_OOM = -3
SWE_ERR_DEPTH = -4
SWE_ERR_NONFINITE = -5
SWE_ERR_HYPERBOLIC = -6
SWE_ERR_UNSUPPORTED = -7
SWE_ERR_TIMEOUT = -8

FIELDS = ("h", "qx", "qy", "hC")


class SweError(RuntimeError):
    def __init__(self, status, where):
        self.status = int(status)
        super().__init__(f"{where}: {swe_status_str(status)} ({status})")


class _Grid(C.Structure):
    _fields_ = [("nx", C.c_int32), ("ny", C.c_int32), ("dx", C.c_double), ("dy", C.c_double)]


class _Mesh(C.Structure):
    _fields_ = [("n_vertices", C.c_int64), ("xy", C.c_void_p), ("n_cells", C.c_int64),
                ("tri", C.c_void_p), ("reorder", C.c_int32)]


class _Params(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("precision", C.c_int32), ("pollutant", C.c_int32),
                ("g", C.c_double), ("r", C.c_double), ("cfl", C.c_double),
                ("stream", C.c_void_p), ("entropy_fix", C.c_int32), ("wet_dry", C.c_int32),
                ("h_dry", C.c_double)]


class _Info(C.Structure):
    _fields_ = [("steps", C.c_int64), ("t", C.c_double), ("nx", C.c_int32), ("ny", C.c_int32),
                ("precision", C.c_int32), ("pitch", C.c_int32), ("field_offset", C.c_int64),
                ("device_bytes", C.c_int64), ("bands", C.c_int32), ("segments", C.c_int32),
                ("warps_per_block", C.c_int32), ("n_layers", C.c_int32),
                ("n_cells", C.c_int64), ("n_edges", C.c_int64), ("mesh", C.c_int32)]


class _KernelTime(C.Structure):
    _fields_ = [("name", C.c_char * 32), ("launches", C.c_int64), ("ms", C.c_double)]


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_needed: bool = True):
    """Load libswe (building it first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_needed else _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libswe is not built ({path}); call finite_volume_shallow_gb300.build.build()")
    L = C.CDLL(path)
    vp, i32, i64, d = C.c_void_p, C.c_int32, C.c_int64, C.c_double
    L.swe_create_grid.argtypes = [C.POINTER(_Grid), vp, vp, C.POINTER(_Params), C.POINTER(vp)]
    L.swe_create_mesh.argtypes = [C.POINTER(_Mesh), vp, vp, C.POINTER(_Params), C.POINTER(vp)]
    L.swe_cell_index.argtypes = [vp, vp]
    L.swe_mesh_info.argtypes = [C.POINTER(_Mesh), vp, vp, vp, vp, vp]
    L.swe_set_timing.argtypes = [vp, i32]
    L.swe_get_timing.argtypes = [vp, vp, i32, C.POINTER(i32)]
    L.swe_step.argtypes = [vp, d, C.POINTER(d)]
    L.swe_run.argtypes = [vp, i64]
    L.swe_get_state.argtypes = [vp, vp, C.POINTER(d)]
    L.swe_set_state.argtypes = [vp, vp, d]
    L.swe_get_dt_history.argtypes = [vp, vp, i64, C.POINTER(i64)]
    L.swe_get_info.argtypes = [vp, C.POINTER(_Info)]
    L.swe_device_fields.argtypes = [vp, vp]
    L.swe_run_noalloc.argtypes = [C.POINTER(_Grid), C.POINTER(_Params), vp, vp, vp, i32, i64, vp]
    L.swe_selftest_wait.argtypes = [i64]
    L.swe_probe_fma_rate.argtypes = [i32, d, vp, C.POINTER(d), C.POINTER(d)]
    L.swe_destroy.argtypes = [vp]
    L.swe_destroy.restype = None
    L.swe_status_str.argtypes = [i32]
    L.swe_status_str.restype = C.c_char_p
    for name in ("swe_create_grid", "swe_create_mesh", "swe_cell_index", "swe_mesh_info",
                 "swe_step", "swe_run",
                 "swe_get_state", "swe_set_state", "swe_get_dt_history", "swe_get_info",
                 "swe_device_fields", "swe_run_noalloc", "swe_set_timing", "swe_get_timing",
                 "swe_selftest_wait", "swe_probe_fma_rate"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def swe_status_str(status) -> str:
    return load().swe_status_str(int(status)).decode()


def _check(st, where):
    if st != SWE_OK:
        raise SweError(st, where)


def _dtype(precision):
    if precision == 32:
        return np.float32
    if precision == 64:
        return np.float64
    raise ValueError("precision must be 32 or 64")


def _host_ptr(x, dtype, n, writable=False):
    """Address of a host buffer of n elements of dtype; numpy or CPU torch."""
    if hasattr(x, "data_ptr") and hasattr(x, "is_cuda"):
        import torch
        want = torch.float32 if dtype == np.float32 else torch.float64
        if x.is_cuda or x.dtype != want or x.numel() != n or not x.is_contiguous():
            raise ValueError(f"expected a contiguous CPU {want} tensor of {n} elements")
        return x.data_ptr()
    if not isinstance(x, np.ndarray) or x.dtype != dtype or x.size != n or not x.flags.c_contiguous:
        raise ValueError(f"expected a C-contiguous numpy {np.dtype(dtype).name} array of {n} elements")
    if writable and not x.flags.writeable:
        raise ValueError("output array is read-only")
    return x.ctypes.data


class State:
    """An open simulation handle (``swe_state*``)."""

    def __init__(self, ptr, nx, ny, precision, n_layers=1):
        self.ptr = C.c_void_p(ptr)
        self.nx, self.ny, self.precision = nx, ny, precision
        self.n_layers = n_layers
        self.nfields = 6 if n_layers == 2 else 4

    @property
    def n(self):
        return self.nx * self.ny

    def __del__(self):
        try:
            swe_destroy(self)
        except Exception:
            pass


def swe_create_grid(nx, ny, dx, dy, H, W0, precision=64, g=9.81, cfl=0.9, stream=None,
                    n_layers=1, pollutant=1, r=0.0, entropy_fix=0, wet_dry=0,
                    h_dry=0.0) -> State:
    """Create a simulation on an nx x ny grid (see swe_create_grid in swe.h).
    H and the fields of W0 (h, qx, qy, hC; or h1, q1x, q1y, h2, q2x, q2y with
    n_layers=2, pollutant=0) are host arrays of the state's precision;
    ``stream`` is a cudaStream_t as an int (e.g.
    ``torch.cuda.current_stream().cuda_stream``) or None; ``entropy_fix=1``
    switches on the Harten-Hyman entropy fix, ``wet_dry=1`` the wet/dry
    treatment with dry threshold ``h_dry`` (see swe_params in swe.h)."""
    L = load()
    dt = _dtype(precision)
    n = int(nx) * int(ny)
    grid = _Grid(int(nx), int(ny), float(dx), float(dy))
    params = _Params(int(n_layers), int(precision), int(pollutant), float(g), float(r),
                     float(cfl), C.c_void_p(stream) if stream else None, int(entropy_fix),
                     int(wet_dry), float(h_dry))
    Hp = _host_ptr(H, dt, n)
    W = (C.c_void_p * len(W0))(*[_host_ptr(w, dt, n) for w in W0])
    out = C.c_void_p()
    _check(L.swe_create_grid(C.byref(grid), C.c_void_p(Hp), W, C.byref(params), C.byref(out)),
           "swe_create_grid")
    return State(out.value, int(nx), int(ny), int(precision), int(n_layers))


def swe_create_mesh(xy, tri, H, W0, precision=64, g=9.81, cfl=0.9, stream=None, n_layers=1,
                    pollutant=1, r=0.0, reorder=1, entropy_fix=0, wet_dry=0,
                    h_dry=0.0) -> State:
    """Create a simulation on a triangle mesh (see swe_create_mesh in swe.h):
    ``xy`` is an (n_vertices, 2) float64 array, ``tri`` an (n_cells, 3) int32
    array of counter-clockwise vertex indices; H and the fields of W0 hold
    n_cells values in the same numbering as ``tri``."""
    L = load()
    dt = _dtype(precision)
    mesh, xy, tri = _mesh_struct(xy, tri, reorder)
    n = int(tri.shape[0])
    params = _Params(int(n_layers), int(precision), int(pollutant), float(g), float(r),
                     float(cfl), C.c_void_p(stream) if stream else None, int(entropy_fix),
                     int(wet_dry), float(h_dry))
    Hp = _host_ptr(H, dt, n)
    W = (C.c_void_p * len(W0))(*[_host_ptr(w, dt, n) for w in W0])
    out = C.c_void_p()
    _check(L.swe_create_mesh(C.byref(mesh), C.c_void_p(Hp), W, C.byref(params), C.byref(out)),
           "swe_create_mesh")
    return State(out.value, n, 1, int(precision), int(n_layers))


def _mesh_struct(xy, tri, reorder):
    xy = np.asarray(xy)
    tri = np.asarray(tri)
    if xy.dtype != np.float64 or xy.ndim != 2 or xy.shape[1] != 2 or not xy.flags.c_contiguous:
        raise ValueError("xy must be a C-contiguous (n_vertices, 2) float64 array")
    if tri.dtype != np.int32 or tri.ndim != 2 or tri.shape[1] != 3 or not tri.flags.c_contiguous:
        raise ValueError("tri must be a C-contiguous (n_cells, 3) int32 array")
    return _Mesh(int(xy.shape[0]), xy.ctypes.data, int(tri.shape[0]), tri.ctypes.data,
                 int(reorder)), xy, tri


def swe_mesh_info(xy, tri, reorder=1):
    """Host-only preview of the mesh preparation: (new_of_old, n_edges,
    n_tiles, n_edge_evals, n_halo); see swe_mesh_info in swe.h."""
    mesh, xy, tri = _mesh_struct(xy, tri, reorder)
    order = np.empty(tri.shape[0], dtype=np.int32)
    out = [C.c_int64() for _ in range(4)]
    _check(load().swe_mesh_info(C.byref(mesh), order.ctypes.data, *[C.byref(v) for v in out]),
           "swe_mesh_info")
    return (order, *[v.value for v in out])


def swe_cell_index(s: State):
    """Element index of every cell (caller numbering) within the device fields."""
    idx = np.empty(s.n, dtype=np.int64)
    _check(load().swe_cell_index(s.ptr, idx.ctypes.data), "swe_cell_index")
    return idx


def swe_set_timing(s: State, on=True):
    """Start (from zero) or stop per-kernel device timing of later steps."""
    _check(load().swe_set_timing(s.ptr, 1 if on else 0), "swe_set_timing")


def swe_get_timing(s: State) -> dict:
    """{kernel name: (launches, summed milliseconds)} of the timed steps."""
    buf = (_KernelTime * 8)()
    n = C.c_int32()
    _check(load().swe_get_timing(s.ptr, buf, 8, C.byref(n)), "swe_get_timing")
    return {buf[k].name.decode(): (int(buf[k].launches), float(buf[k].ms)) for k in range(n.value)}


def swe_step(s: State, cfl) -> float:
    dt = C.c_double()
    _check(load().swe_step(s.ptr, float(cfl), C.byref(dt)), "swe_step")
    return dt.value


def swe_run(s: State, nsteps):
    _check(load().swe_run(s.ptr, int(nsteps)), "swe_run")


def swe_get_state(s: State, out=None):
    """Returns (fields, t); ``out`` may supply the four host output arrays."""
    dt = _dtype(s.precision)
    if out is None:
        out = [np.empty(s.n, dtype=dt) for _ in range(s.nfields)]
    ptrs = (C.c_void_p * len(out))(*[_host_ptr(o, dt, s.n, writable=True) for o in out])
    t = C.c_double()
    _check(load().swe_get_state(s.ptr, ptrs, C.byref(t)), "swe_get_state")
    return out, t.value


def swe_set_state(s: State, fields, t=0.0):
    dt = _dtype(s.precision)
    ptrs = (C.c_void_p * len(fields))(*[_host_ptr(f, dt, s.n) for f in fields])
    _check(load().swe_set_state(s.ptr, ptrs, float(t)), "swe_set_state")


def swe_get_dt_history(s: State, max_n=1 << 16):
    buf = np.empty(int(max_n), dtype=np.float64)
    n = C.c_int64()
    _check(load().swe_get_dt_history(s.ptr, buf.ctypes.data, int(max_n), C.byref(n)),
           "swe_get_dt_history")
    return buf[: n.value].copy()


def swe_get_info(s: State) -> dict:
    info = _Info()
    _check(load().swe_get_info(s.ptr, C.byref(info)), "swe_get_info")
    return {k: getattr(info, k) for k, _ in _Info._fields_}


def swe_device_fields(s: State):
    """Device addresses of the current state's fields followed by H."""
    ptrs = (C.c_void_p * (s.nfields + 1))()
    _check(load().swe_device_fields(s.ptr, ptrs), "swe_device_fields")
    return [p or 0 for p in ptrs]


NOALLOC_MAX_STEPS = 1024


def noalloc_pitch(nx) -> int:
    """Smallest row pitch (elements) swe_run_noalloc accepts for nx columns."""
    need = 60 * ((int(nx) + 59) // 60) + 4
    return (need + 31) // 32 * 32


def swe_run_noalloc(nx, ny, dx, dy, H, W_a, W_b, pitch, nsteps, precision=64, g=9.81,
                    cfl=0.9, stream=None, entropy_fix=0):
    """Allocation-free run on caller-owned device buffers (see swe.h): H, W_a
    (4) and W_b (4) are device addresses (ints) in the padded layout.
    Returns the dt of each step."""
    grid = _Grid(int(nx), int(ny), float(dx), float(dy))
    params = _Params(1, int(precision), 1, float(g), 0.0, float(cfl),
                     C.c_void_p(stream) if stream else None, int(entropy_fix))
    wa = (C.c_void_p * 4)(*[int(p) for p in W_a])
    wb = (C.c_void_p * 4)(*[int(p) for p in W_b])
    dts = np.zeros(max(int(nsteps), 1), dtype=np.float64)
    _check(load().swe_run_noalloc(C.byref(grid), C.byref(params), C.c_void_p(int(H)), wa, wb,
                                  int(pitch), int(nsteps), dts.ctypes.data), "swe_run_noalloc")
    return dts[: int(nsteps)]


def swe_selftest_wait(budget_cycles) -> int:
    """Run the step kernel's bounded device wait on a barrier nothing arrives
    on (see swe.h); returns the status, SWE_ERR_TIMEOUT when the wait gave up
    as designed."""
    return int(load().swe_selftest_wait(int(budget_cycles)))


PROBE_FFMA, PROBE_FFMA2, PROBE_DFMA = 0, 1, 2


def swe_probe_fma_rate(kind, target_ms=50.0, stream=None):
    """Measured FMA throughput of the current device (see swe_probe.h):
    (flops per second, duration of the timed launch in ms)."""
    rate, ms = C.c_double(0.0), C.c_double(0.0)
    _check(load().swe_probe_fma_rate(int(kind), float(target_ms),
                                      C.c_void_p(stream) if stream else None, C.byref(rate),
                                      C.byref(ms)), "swe_probe_fma_rate")
    return rate.value, ms.value


def swe_destroy(s: State):
    if s is not None and s.ptr:
        load().swe_destroy(s.ptr)
        s.ptr = C.c_void_p()
