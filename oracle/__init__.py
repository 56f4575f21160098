"""ctypes wrapper of the plain fp64 CPU oracle (``swe_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the bench's
CPU-baseline leg are the only callers.  The product path never imports it.

The oracle restates An MPI-CUDA implementation of an improved Roe method for
two-layer shallow water systems, Sec. 2.2 (eq. (4), flux steps 1-4, CFL
eq. (5)) for one layer plus a passive pollutant (A multi-GPU shallow-water
simulation with transport of contaminants, abstract) on a generic polygon
mesh, in fp64 on one CPU thread.  ``build()`` compiles it with the host C
compiler; nothing here depends on the CUDA extension.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")
SOURCES = [os.path.join(HERE, "swe_oracle.c")]
HEADERS = [os.path.join(HERE, "swe_oracle.h")]

OM_OK = 0
OM_ERR_ARG = -1
OM_ERR_DEPTH = -4
OM_ERR_NONFINITE = -5
OM_ERR_HYPERBOLIC = -6

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` if it is missing
    or older than its sources.  Strict IEEE fp64: no fast-math and no FMA
    contraction, so x86-64 and aarch64 hosts give the same bits."""
    newest = max(os.path.getmtime(p) for p in SOURCES + HEADERS)
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Werror", "-o", tmp] + SOURCES + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


class _Mesh(C.Structure):
    _fields_ = [("n_cells", C.c_int64), ("area", C.c_void_p),
                ("edge_start", C.c_void_p), ("nbr", C.c_void_p),
                ("eta_x", C.c_void_p), ("eta_y", C.c_void_p),
                ("len", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        # SWE_ORACLE_LIB points the wrapper at another build of the same
        # source (the mutation tests load deliberately broken copies).
        _lib = C.CDLL(os.environ.get("SWE_ORACLE_LIB") or build())
        d, i64, vp = C.c_double, C.c_int64, C.c_void_p
        _lib.om_grid_edges.restype = i64
        _lib.om_grid_edges.argtypes = [i64, i64]
        _lib.om_grid_mesh.restype = None
        _lib.om_grid_mesh.argtypes = [i64, i64, d, d, vp, vp, vp, vp, vp, vp]
        _lib.om_flux1.restype = None
        _lib.om_flux1.argtypes = [vp, vp, d, d, d, d, d, vp, vp]
        _lib.om_set_entropy_fix.restype = None
        _lib.om_set_entropy_fix.argtypes = [C.c_int]
        _lib.om_set_wet_dry.restype = None
        _lib.om_set_wet_dry.argtypes = [C.c_int, C.c_double]
        _lib.om_wall_ghost1.restype = None
        _lib.om_wall_ghost1.argtypes = [vp, d, d, vp]
        _lib.om_dt1.restype = d
        _lib.om_dt1.argtypes = [C.POINTER(_Mesh), vp, vp, d, d]
        _lib.om_update1.restype = C.c_int
        _lib.om_update1.argtypes = [C.POINTER(_Mesh), vp, vp, d, d, vp]
        _lib.om_update1_at.restype = None
        _lib.om_update1_at.argtypes = [C.POINTER(_Mesh), vp, vp, d, d, vp, i64, vp]
        _lib.om_run1.restype = C.c_int
        _lib.om_run1.argtypes = [C.POINTER(_Mesh), vp, vp, d, d, i64, vp, vp,
                                 C.POINTER(C.c_int64)]
        _lib.om_wall_ghost2.restype = None
        _lib.om_wall_ghost2.argtypes = [vp, d, d, vp]
        _lib.om_roots2.restype = C.c_int
        _lib.om_roots2.argtypes = [d, d, d, d, d, vp]
        _lib.om_flux2.restype = C.c_int
        _lib.om_flux2.argtypes = [vp, vp, d, d, d, d, d, d, vp, vp]
        _lib.om_dt2.restype = d
        _lib.om_dt2.argtypes = [C.POINTER(_Mesh), vp, vp, d, d, d, C.POINTER(C.c_int)]
        _lib.om_update2.restype = C.c_int
        _lib.om_update2.argtypes = [C.POINTER(_Mesh), vp, vp, d, d, d, vp]
        _lib.om_update2_at.argtypes = [C.POINTER(_Mesh), vp, vp, d, d, d, vp, i64, vp]
        _lib.om_run2.restype = C.c_int
        _lib.om_run2.argtypes = [C.POINTER(_Mesh), vp, vp, d, d, d, i64, vp, vp,
                                 C.POINTER(C.c_int64)]
        _lib.om_grid_dt2.restype = d
        _lib.om_grid_dt2.argtypes = [i64, i64, d, d, vp, vp, d, d, d, C.POINTER(C.c_int)]
        _lib.om_grid_update2.restype = C.c_int
        _lib.om_grid_update2.argtypes = [i64, i64, d, d, vp, vp, d, d, d, vp]
        _lib.om_grid_run2.restype = C.c_int
        _lib.om_grid_run2.argtypes = [i64, i64, d, d, vp, vp, d, d, d, i64, vp, vp,
                                      C.POINTER(C.c_int64)]
        _lib.om_tri_mesh.restype = C.c_int
        _lib.om_tri_mesh.argtypes = [i64, vp, i64, vp, vp, vp, vp, vp, vp, vp]
        _lib.om_grid_dt1.restype = d
        _lib.om_grid_dt1.argtypes = [i64, i64, d, d, vp, vp, d, d]
        _lib.om_grid_update1.restype = C.c_int
        _lib.om_grid_update1.argtypes = [i64, i64, d, d, vp, vp, d, d, vp]
        _lib.om_grid_run1.restype = C.c_int
        _lib.om_grid_run1.argtypes = [i64, i64, d, d, vp, vp, d, d, i64, vp, vp,
                                      C.POINTER(C.c_int64)]
    return _lib


class entropy_fix:
    """Context manager: the flux of the oracle (one layer or two) with the
    Harten-Hyman entropy fix switched on (see om_set_entropy_fix)."""

    def __init__(self, on=True):
        self.on = bool(on)

    def __enter__(self):
        lib().om_set_entropy_fix(1 if self.on else 0)
        return self

    def __exit__(self, *exc):
        lib().om_set_entropy_fix(0)
        return False


class wet_dry:
    """Context manager: the one-layer oracle with the wet/dry treatment on
    (depth threshold h_dry; see om_set_wet_dry)."""

    def __init__(self, h_dry=1e-6, on=True):
        self.on = bool(on)
        self.h_dry = float(h_dry)

    def __enter__(self):
        lib().om_set_wet_dry(1 if self.on else 0, self.h_dry)
        return self

    def __exit__(self, *exc):
        lib().om_set_wet_dry(0, 0.0)
        return False


def _ptr(a):
    return a.ctypes.data_as(C.c_void_p)


class Mesh:
    """Polygon mesh in per-cell edge lists (see ``om_mesh`` in the header)."""

    def __init__(self, area, edge_start, nbr, eta_x, eta_y, length):
        self.area = np.ascontiguousarray(area, dtype=np.float64)
        self.edge_start = np.ascontiguousarray(edge_start, dtype=np.int64)
        self.nbr = np.ascontiguousarray(nbr, dtype=np.int64)
        self.eta_x = np.ascontiguousarray(eta_x, dtype=np.float64)
        self.eta_y = np.ascontiguousarray(eta_y, dtype=np.float64)
        self.len = np.ascontiguousarray(length, dtype=np.float64)
        self.n_cells = self.area.size
        counts = np.diff(self.edge_start)
        if self.edge_start.size != self.n_cells + 1 or counts.min(initial=1) < 1:
            raise ValueError("bad edge_start")
        if counts.max(initial=0) > 16:
            raise ValueError("the oracle handles at most 16 edges per cell")
        if self.nbr.max(initial=-1) >= self.n_cells:
            raise ValueError("neighbour index out of range")
        self._c = _Mesh(self.n_cells, _ptr(self.area).value, _ptr(self.edge_start).value,
                        _ptr(self.nbr).value, _ptr(self.eta_x).value,
                        _ptr(self.eta_y).value, _ptr(self.len).value)

    @property
    def c(self):
        return C.byref(self._c)


def grid_mesh(nx, ny, dx, dy=None) -> Mesh:
    """The nx x ny Cartesian grid as a polygon mesh; cell (i, j) is index
    j*nx + i, its edges listed East, North, West, South."""
    dy = dx if dy is None else dy
    L = lib()
    ne = L.om_grid_edges(nx, ny)
    area = np.empty(nx * ny)
    es = np.empty(nx * ny + 1, dtype=np.int64)
    nbr = np.empty(ne, dtype=np.int64)
    ex = np.empty(ne)
    ey = np.empty(ne)
    ln = np.empty(ne)
    L.om_grid_mesh(nx, ny, float(dx), float(dy), _ptr(area), _ptr(es), _ptr(nbr),
                   _ptr(ex), _ptr(ey), _ptr(ln))
    return Mesh(area, es, nbr, ex, ey, ln)


def tri_mesh(xy, tri) -> Mesh:
    """Polygon-mesh arrays of a counter-clockwise triangle mesh (edges of cell
    c: (v0 v1), (v1 v2), (v2 v0))."""
    xy = np.ascontiguousarray(xy, dtype=np.float64).reshape(-1)
    tri = np.ascontiguousarray(tri, dtype=np.int32).reshape(-1)
    nv, nc = xy.size // 2, tri.size // 3
    area = np.empty(nc)
    es = np.empty(nc + 1, dtype=np.int64)
    nbr = np.empty(3 * nc, dtype=np.int64)
    ex = np.empty(3 * nc)
    ey = np.empty(3 * nc)
    ln = np.empty(3 * nc)
    st = lib().om_tri_mesh(nv, _ptr(xy), nc, _ptr(tri), _ptr(area), _ptr(es), _ptr(nbr),
                           _ptr(ex), _ptr(ey), _ptr(ln))
    if st != OM_OK:
        raise ValueError("invalid triangle mesh (index, orientation or non-manifold edge)")
    return Mesh(area, es, nbr, ex, ey, ln)


def _field_ptrs(W):
    arr = (C.c_void_p * len(W))(*[_ptr(w).value for w in W])
    return arr


def _fields(W, n, k=4):
    out = [np.array(w, dtype=np.float64, copy=True).reshape(-1) for w in W]
    if len(out) != k or any(w.size != n for w in out):
        raise ValueError(f"expected {k} fields of n_cells values")
    return out


def flux1(Wi, Wj, Hi, Hj, eta, g):
    """F_ij^- (Cartesian h, qx, qy, hC components) and ||D_ij||_inf."""
    wi = np.ascontiguousarray(Wi, dtype=np.float64)
    wj = np.ascontiguousarray(Wj, dtype=np.float64)
    F = np.empty(4)
    D = np.empty(1)
    lib().om_flux1(_ptr(wi), _ptr(wj), float(Hi), float(Hj), float(eta[0]),
                   float(eta[1]), float(g), _ptr(F), _ptr(D))
    return F, float(D[0])


def wall_ghost1(Wi, eta):
    wi = np.ascontiguousarray(Wi, dtype=np.float64)
    out = np.empty(4)
    lib().om_wall_ghost1(_ptr(wi), float(eta[0]), float(eta[1]), _ptr(out))
    return out


def dt1(mesh: Mesh, H, W, g, cfl) -> float:
    """Time step of eq. (5) for the state W = (h, qx, qy, hC)."""
    Wf = _fields(W, mesh.n_cells)
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    return float(lib().om_dt1(mesh.c, _field_ptrs(Wf), _ptr(Hf), float(g), float(cfl)))


def update1(mesh: Mesh, H, W, g, dt):
    """One step of eq. (4) with a given dt; returns (fields, status)."""
    Wf = _fields(W, mesh.n_cells)
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    work = np.empty(4 * mesh.n_cells)
    st = lib().om_update1(mesh.c, _field_ptrs(Wf), _ptr(Hf), float(g), float(dt), _ptr(work))
    return Wf, int(st)


def update1_at(mesh: Mesh, H, W, g, dt, cells):
    """The fields after one step of size dt, at the given cells only:
    array of shape (4, len(cells))."""
    Wf = [np.ascontiguousarray(w, dtype=np.float64).reshape(-1) for w in W]
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    cells = np.ascontiguousarray(cells, dtype=np.int64)
    out = np.empty(4 * cells.size)
    lib().om_update1_at(mesh.c, _field_ptrs(Wf), _ptr(Hf), float(g), float(dt),
                        _ptr(cells), cells.size, _ptr(out))
    return out.reshape(4, cells.size)


def run1(mesh: Mesh, H, W, g, cfl, nsteps):
    """``nsteps`` steps from W; returns (fields, dts, status, steps_done)."""
    Wf = _fields(W, mesh.n_cells)
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    work = np.empty(4 * mesh.n_cells)
    dts = np.zeros(max(int(nsteps), 1))
    done = C.c_int64(0)
    st = lib().om_run1(mesh.c, _field_ptrs(Wf), _ptr(Hf), float(g), float(cfl),
                       int(nsteps), _ptr(dts), _ptr(work), C.byref(done))
    return Wf, dts[: done.value], int(st), int(done.value)


def grid_dt1(nx, ny, dx, dy, H, W, g, cfl) -> float:
    """eq. (5) on the implicit nx x ny grid (no mesh arrays)."""
    Wf = [np.ascontiguousarray(w, dtype=np.float64).reshape(-1) for w in W]
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    return float(lib().om_grid_dt1(int(nx), int(ny), float(dx), float(dy), _field_ptrs(Wf),
                                   _ptr(Hf), float(g), float(cfl)))


def grid_update1(nx, ny, dx, dy, H, W, g, dt):
    """eq. (4) with a given dt on the implicit grid; returns (fields, status)."""
    Wf = _fields(W, int(nx) * int(ny))
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    work = np.empty(4 * int(nx) * int(ny))
    st = lib().om_grid_update1(int(nx), int(ny), float(dx), float(dy), _field_ptrs(Wf),
                               _ptr(Hf), float(g), float(dt), _ptr(work))
    return Wf, int(st)


def grid_run1(nx, ny, dx, dy, H, W, g, cfl, nsteps):
    """``nsteps`` steps on the implicit grid; returns (fields, dts, status)."""
    n = int(nx) * int(ny)
    Wf = _fields(W, n)
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    work = np.empty(4 * n)
    dts = np.zeros(max(int(nsteps), 1))
    done = C.c_int64(0)
    st = lib().om_grid_run1(int(nx), int(ny), float(dx), float(dy), _field_ptrs(Wf), _ptr(Hf),
                            float(g), float(cfl), int(nsteps), _ptr(dts), _ptr(work),
                            C.byref(done))
    return Wf, dts[: done.value], int(st)


def run_grid(d, nsteps=None, cfl=None):
    """Run a workload dict (see ``finite_volume_shallow_gb300.inputs``) on its
    Cartesian grid; returns (fields, dts, status)."""
    mesh = grid_mesh(d["nx"], d["ny"], d["dx"], d["dy"])
    n = d["steps"] if nsteps is None else nsteps
    W = [d["h"], d["qx"], d["qy"], d["hC"]]
    Wf, dts, st, _ = run1(mesh, d["H"], W, d["g"], d["cfl"] if cfl is None else cfl, n)
    return Wf, dts, st


# ---- two layers: W = (h1, q1x, q1y, h2, q2x, q2y) --------------------------

def wall_ghost2(Wi, eta):
    wi = np.ascontiguousarray(Wi, dtype=np.float64)
    out = np.empty(6)
    lib().om_wall_ghost2(_ptr(wi), float(eta[0]), float(eta[1]), _ptr(out))
    return out


def roots2(u1, u2, c1s, c2s, r):
    """(status, eigenvalues ascending) of the 2-layer Roe matrix."""
    lam = np.zeros(4)
    st = lib().om_roots2(float(u1), float(u2), float(c1s), float(c2s), float(r), _ptr(lam))
    return int(st), lam


def flux2(Wi, Wj, Hi, Hj, eta, g, r):
    """(status, F_ij^- (6 Cartesian components), ||D_ij||_inf)."""
    wi = np.ascontiguousarray(Wi, dtype=np.float64)
    wj = np.ascontiguousarray(Wj, dtype=np.float64)
    F = np.zeros(6)
    D = np.zeros(1)
    st = lib().om_flux2(_ptr(wi), _ptr(wj), float(Hi), float(Hj), float(eta[0]), float(eta[1]),
                        float(g), float(r), _ptr(F), _ptr(D))
    return int(st), F, float(D[0])


def dt2(mesh: Mesh, H, W, g, r, cfl):
    Wf = _fields(W, mesh.n_cells, 6)
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    st = C.c_int(0)
    dt = lib().om_dt2(mesh.c, _field_ptrs(Wf), _ptr(Hf), float(g), float(r), float(cfl),
                      C.byref(st))
    return float(dt), int(st.value)


def update2(mesh: Mesh, H, W, g, r, dt):
    Wf = _fields(W, mesh.n_cells, 6)
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    work = np.empty(6 * mesh.n_cells)
    st = lib().om_update2(mesh.c, _field_ptrs(Wf), _ptr(Hf), float(g), float(r), float(dt),
                          _ptr(work))
    return Wf, int(st)


def update2_at(mesh: Mesh, H, W, g, r, dt, cells):
    """The six fields after one step of size dt, at the given cells only:
    (array of shape (6, len(cells)), status)."""
    Wf = [np.ascontiguousarray(w, dtype=np.float64).reshape(-1) for w in W]
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    cells = np.ascontiguousarray(cells, dtype=np.int64)
    out = np.empty(6 * cells.size)
    st = lib().om_update2_at(mesh.c, _field_ptrs(Wf), _ptr(Hf), float(g), float(r), float(dt),
                             _ptr(cells), cells.size, _ptr(out))
    return out.reshape(6, cells.size), int(st)


def run2(mesh: Mesh, H, W, g, r, cfl, nsteps):
    Wf = _fields(W, mesh.n_cells, 6)
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    work = np.empty(6 * mesh.n_cells)
    dts = np.zeros(max(int(nsteps), 1))
    done = C.c_int64(0)
    st = lib().om_run2(mesh.c, _field_ptrs(Wf), _ptr(Hf), float(g), float(r), float(cfl),
                       int(nsteps), _ptr(dts), _ptr(work), C.byref(done))
    return Wf, dts[: done.value], int(st)


def grid_dt2(nx, ny, dx, dy, H, W, g, r, cfl):
    Wf = [np.ascontiguousarray(w, dtype=np.float64).reshape(-1) for w in W]
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    st = C.c_int(0)
    dt = lib().om_grid_dt2(int(nx), int(ny), float(dx), float(dy), _field_ptrs(Wf), _ptr(Hf),
                           float(g), float(r), float(cfl), C.byref(st))
    return float(dt), int(st.value)


def grid_update2(nx, ny, dx, dy, H, W, g, r, dt):
    n = int(nx) * int(ny)
    Wf = _fields(W, n, 6)
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    work = np.empty(6 * n)
    st = lib().om_grid_update2(int(nx), int(ny), float(dx), float(dy), _field_ptrs(Wf),
                               _ptr(Hf), float(g), float(r), float(dt), _ptr(work))
    return Wf, int(st)


def grid_run2(nx, ny, dx, dy, H, W, g, r, cfl, nsteps):
    n = int(nx) * int(ny)
    Wf = _fields(W, n, 6)
    Hf = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    work = np.empty(6 * n)
    dts = np.zeros(max(int(nsteps), 1))
    done = C.c_int64(0)
    st = lib().om_grid_run2(int(nx), int(ny), float(dx), float(dy), _field_ptrs(Wf), _ptr(Hf),
                            float(g), float(r), float(cfl), int(nsteps), _ptr(dts), _ptr(work),
                            C.byref(done))
    return Wf, dts[: done.value], int(st)
