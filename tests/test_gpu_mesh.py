"""Triangle meshes on the GPU (through the C ABI) against the oracle on its
own, independently built mesh (An MPI-CUDA implementation of an improved Roe
method for two-layer shallow water systems, Sec. 2.2: triangle volumes,
eq. (4), CFL eq. (5)), same seeded inputs, element by element in the
caller's numbering; plus invariants and the full 1024 x 1024-square,
2.1M-triangle two-layer workload (sampled cells against the oracle's update
of the same state).

Tolerances: fp64 <= 1e-10 per field and dt <= 1e-12; fp32 <= 1e-4 on depths,
<= 1e-3 on discharges and pollutant, dt <= 1e-6 (relative to each field's
scale).
"""
import ctypes as C
import os

import numpy as np
import pytest

import oracle as O
from finite_volume_shallow_gb300 import inputs as I
from finite_volume_shallow_gb300 import swe as S
from gpu_util import (TOL2, assert_parity_mesh, gpu_create_mesh, gpu_run_mesh, mesh_fields,
                      np_dtype, oracle_run_mesh)

pytestmark = pytest.mark.gpu
G = 9.81


@pytest.mark.parametrize("precision", [64, 32])
def test_two_layer_triangles(precision):
    # features resolved on this small mesh (widths 2.5-15 squares), interface
    # bump of 1 m so that the layers move well above fp32 rounding
    d = I.tri_workload(40, sigma_scale=0.05, bump=1.0)
    assert_parity_mesh(d, precision, 40)


@pytest.mark.parametrize("precision", [64, 32])
def test_small_density_ratio_on_triangles(precision):
    # layers of nearly equal depth at r = 0.01 (interface near mid-depth,
    # tilted so that it moves): nearly coinciding outer roots
    d = I.tri_workload(16, r=0.01, bump=0.0, sigma_scale=0.05)
    x = I.tri_centroids(d["xy"], d["tri"])[:, 0]
    d["h1"] = d["H"] * (0.5 + 0.02 * (x - x.mean()) / np.ptp(x))
    d["h2"] = d["H"] - d["h1"]
    rel = np.abs(np.sqrt(d["h1"]) - np.sqrt(d["h2"])) / np.sqrt(d["h1"])
    assert rel.min() < 1e-3
    assert_parity_mesh(d, precision, 20)


@pytest.mark.parametrize("precision", [64, 32])
def test_one_layer_triangles_with_pollutant(precision):
    d = I.tri_workload1(36, 22)
    assert_parity_mesh(d, precision, 60)


@pytest.mark.parametrize("precision", [64, 32])
def test_caller_order_kept(precision):
    # reorder = 0 runs the same scheme in the caller's (shuffled) order
    d = I.tri_workload1(20, 16, seed=31)
    assert_parity_mesh(d, precision, 30, reorder=0)


def small_meshes():
    out = {}
    xy = np.array([[0.0, 0.0], [2.0, 0.1], [0.7, 1.5]])
    out["one_triangle"] = (xy, np.array([[0, 1, 2]], dtype=np.int32))
    out["one_square"] = I.square_tri_mesh(1, jitter=0.0, shuffle=False)
    out["strip_1x9"] = I.square_tri_mesh(9, 1, jitter=0.0, shuffle=True, seed=4)
    out["strip_9x1"] = I.square_tri_mesh(1, 9, jitter=0.0, shuffle=True, seed=5)
    xy1, tri1 = I.square_tri_mesh(4, 3, jitter=0.2, seed=6)
    xy2 = xy1 + np.array([50.0, 0.0])
    out["two_components"] = (np.ascontiguousarray(np.concatenate([xy1, xy2])),
                             np.ascontiguousarray(np.concatenate([tri1, tri1 + len(xy1)])))
    out["ragged_13x7"] = I.square_tri_mesh(13, 7, jitter=0.25, seed=7)
    return out


def mesh_state(xy, tri, n_layers, seed):
    rng = np.random.default_rng(seed)
    n = tri.shape[0]
    cxy = I.tri_centroids(xy, tri)
    H = 2.0 - 0.3 * np.sin(cxy[:, 0]) * np.cos(cxy[:, 1])
    d = dict(xy=xy, tri=tri, n_cells=n, n_layers=n_layers, g=G, cfl=0.9, H=H)
    if n_layers == 1:
        h = H + 1.0 + 0.3 * rng.uniform(0, 1, n)
        d.update(h=h, qx=h * rng.uniform(-0.1, 0.1, n), qy=h * rng.uniform(-0.1, 0.1, n),
                 hC=h * rng.uniform(0, 1, n))
    else:
        H = H + 8.0
        h1 = 3.0 + 0.4 * rng.uniform(0, 1, n)
        h2 = H + 1.0 - h1
        d.update(H=H, r=0.98, h1=h1, q1x=h1 * rng.uniform(-0.05, 0.05, n),
                 q1y=h1 * rng.uniform(-0.05, 0.05, n), h2=h2,
                 q2x=h2 * rng.uniform(-0.05, 0.05, n), q2y=h2 * rng.uniform(-0.05, 0.05, n))
    return d


@pytest.mark.parametrize("precision", [64, 32])
@pytest.mark.parametrize("n_layers", [1, 2])
@pytest.mark.parametrize("name", sorted(small_meshes()))
def test_small_and_degenerate_meshes(name, n_layers, precision):
    xy, tri = small_meshes()[name]
    d = mesh_state(xy, tri, n_layers, seed=len(name))
    assert_parity_mesh(d, precision, 15)


@pytest.mark.parametrize("precision", [64, 32])
@pytest.mark.parametrize("n_layers", [1, 2])
def test_lake_at_rest_on_triangles(n_layers, precision):
    xy, tri = I.square_tri_mesh(30, 20, jitter=0.25, seed=12)
    d = mesh_state(xy, tri, n_layers, seed=12)
    if n_layers == 1:
        d["h"] = d["H"] + 1.0
        h = d["h"]
        for k in ("qx", "qy"):
            d[k] = np.zeros_like(h)
        W, _, _ = gpu_run_mesh(d, precision, 100)
        pairs = [(0, "h")]
        qs = [1, 2]
    else:
        d["h1"] = np.full_like(d["H"], 3.0)
        d["h2"] = d["H"] + 1.0 - d["h1"]
        for k in ("q1x", "q1y", "q2x", "q2y"):
            d[k] = np.zeros_like(d["H"])
        W, _, _ = gpu_run_mesh(d, precision, 100)
        pairs = [(0, "h1"), (3, "h2")]
        qs = [1, 2, 4, 5]
    tol = 1e-13 if precision == 64 else 2e-6
    ref = {k: d[k].astype(np_dtype(precision)).astype(np.float64) for _, k in pairs}
    hmax = max(ref[k].max() for _, k in pairs)
    for i, k in pairs:
        assert np.abs(W[i] - ref[k]).max() <= tol * ref[k].max(), k
    qs_scale = hmax * np.sqrt(G * hmax)
    for i in qs:
        assert np.abs(W[i]).max() <= tol * qs_scale


@pytest.mark.parametrize("n_layers", [1, 2])
def test_conservation_on_triangles(n_layers):
    d = I.tri_workload1(40, 30, seed=13) if n_layers == 1 else I.tri_workload(48)
    W, _, _ = gpu_run_mesh(d, 64, 150)
    area = O.tri_mesh(d["xy"], d["tri"]).area
    idx = (0, 3)
    for i, w0 in zip(idx, [mesh_fields(d)[k] for k in idx]):
        assert abs(W[i].dot(area) - w0.dot(area)) / w0.dot(area) <= 1e-12


def test_mesh_restart_is_bitwise_and_history_kept():
    d = I.tri_workload1(24, 18, seed=14)
    a = gpu_create_mesh(d, 32)
    S.swe_run(a, 30)
    Wa, ta = S.swe_get_state(a)
    b = gpu_create_mesh(d, 32)
    S.swe_run(b, 12)
    Wm, tm = S.swe_get_state(b)
    S.swe_set_state(b, Wm, tm)
    S.swe_run(b, 18)
    Wb, tb = S.swe_get_state(b)
    for x, y in zip(Wa, Wb):
        assert np.array_equal(x, y)
    assert ta == pytest.approx(tb, rel=1e-15)
    info = S.swe_get_info(a)
    assert info["mesh"] == 1 and info["n_cells"] == d["n_cells"] and info["steps"] == 30
    assert info["n_edges"] == S.swe_mesh_info(d["xy"], d["tri"])[1]
    assert len(S.swe_get_dt_history(a)) == 30
    # a rejected state leaves the handle usable
    bad = [w.copy() for w in Wa]
    bad[0][3] = -1.0
    with pytest.raises(S.SweError) as e:
        S.swe_set_state(a, bad, 0.0)
    assert e.value.status == S.SWE_ERR_ARG
    S.swe_set_state(a, Wa, ta)
    S.swe_run(a, 2)


def _cudart():
    for name in ("libcudart.so.13", "libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            return C.CDLL(name)
        except OSError:
            continue
    pytest.skip("libcudart not found for the zero-copy check")


def test_cell_index_addresses_the_device_fields():
    d = I.tri_workload1(16, 12, seed=15)
    s = gpu_create_mesh(d, 64)
    S.swe_run(s, 3)
    W, _ = S.swe_get_state(s)
    idx = S.swe_cell_index(s)
    ptrs = S.swe_device_fields(s)
    rt = _cudart()
    rt.cudaMemcpy.argtypes = [C.c_void_p, C.c_void_p, C.c_size_t, C.c_int]
    n = d["n_cells"]
    for k in range(4):
        buf = np.empty(n, dtype=np.float64)
        assert rt.cudaMemcpy(buf.ctypes.data, ptrs[k], n * 8, 2) == 0   # device to host
        assert np.array_equal(buf[idx], W[k])
    Hd = np.empty(n, dtype=np.float64)
    assert rt.cudaMemcpy(Hd.ctypes.data, ptrs[4], n * 8, 2) == 0
    assert np.array_equal(Hd[idx], d["H"])


def test_hyperbolicity_loss_on_triangles():
    xy, tri = I.square_tri_mesh(8, 6, jitter=0.1, seed=16)
    d = mesh_state(xy, tri, 2, seed=16)
    n = d["n_cells"]
    d.update(h1=np.full(n, 3.0), h2=np.full(n, 7.0), H=np.full(n, 10.0),
             q1x=np.full(n, 6.0), q1y=np.zeros(n), q2x=np.full(n, -14.0), q2y=np.zeros(n))
    s = gpu_create_mesh(d, 64)
    with pytest.raises(S.SweError) as e:
        S.swe_step(s, 0.9)
    assert e.value.status == S.SWE_ERR_HYPERBOLIC


@pytest.mark.parametrize("precision", [32])
def test_full_size_triangle_workload(precision):
    # the 1024 x 1024-square, 2.1M-triangle two-layer workload in the launch
    # configuration of the benchmark: after K steps on the GPU, one more GPU
    # step must equal the oracle's update of the GPU's own state at sampled
    # cells, with the oracle's dt of that state; layer masses are conserved
    d = I.make_workload("tri1024")
    n = d["n_cells"]
    s = gpu_create_mesh(d, precision)
    K = 20
    S.swe_run(s, K)
    Wk, _ = S.swe_get_state(s)
    dt_gpu = S.swe_step(s, d["cfl"])
    Wk1, _ = S.swe_get_state(s)
    S.swe_destroy(s)
    m = O.tri_mesh(d["xy"], d["tri"])
    W64 = [w.astype(np.float64) for w in Wk]
    dt_o, st = O.dt2(m, d["H"].astype(np_dtype(precision)).astype(np.float64), W64, G, d["r"],
                     d["cfl"])
    assert st == O.OM_OK
    assert abs(dt_gpu / dt_o - 1) <= TOL2[precision]["dt"]
    rng = np.random.default_rng(17)
    boundary = np.nonzero((m.nbr < 0).reshape(-1, 3).any(axis=1))[0]
    cells = np.unique(np.concatenate([rng.integers(0, n, 3000), boundary[::7]]))
    Hr = d["H"].astype(np_dtype(precision)).astype(np.float64)
    ref, st = O.update2_at(m, Hr, W64, G, d["r"], dt_o, cells)
    assert st == O.OM_OK
    for k, name in enumerate(I.TWO_LAYER_FIELDS):
        scale = max(np.abs(W64[k]).max(), 1e-30)
        # one step from the same state: the error is one step's rounding
        err = np.abs(Wk1[k][cells].astype(np.float64) - ref[k]).max() / scale
        assert err <= 0.1 * TOL2[precision][name], (name, err)
    area = m.area
    for k in (0, 3):
        w0 = d[I.TWO_LAYER_FIELDS[k]].astype(np_dtype(precision)).astype(np.float64)
        assert abs(Wk1[k].astype(np.float64).dot(area) - w0.dot(area)) / w0.dot(area) <= 2e-6


@pytest.mark.parametrize("precision", [64, 32])
def test_cfl_limit_on_triangles(precision):
    d = I.tri_workload1(30, 20, seed=41)
    d["cfl"] = 1.0
    assert_parity_mesh(d, precision, 40)
