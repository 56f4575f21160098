"""Pins of the oracle on triangle meshes (the finite volumes of An MPI-CUDA
implementation of an improved Roe method for two-layer shallow water systems,
Sec. 2.2, are triangles there).

* geometry: the cells tile the domain, every cell closes (sum of |Gamma| eta
  is zero), every interior edge is seen from both sides with opposite normals;
* lake at rest over a bumpy bottom, one and two layers;
* mass, pollutant and layer-mass conservation with walls;
* a constant concentration stays constant;
* Stoker's dam break on triangulated strips, error decreasing under
  refinement;
* symmetry under the half-turn that maps the triangulation onto itself;
* independence of the cell and vertex numbering.
"""
import math

import numpy as np
import pytest

import oracle as O
from finite_volume_shallow_gb300 import inputs as I
import stoker

G = 9.81


def bump_bottom(cxy, L, amp=1.5, sigma_frac=0.15):
    return amp * np.exp(-((cxy[:, 0] - 0.4 * L) ** 2 + (cxy[:, 1] - 0.55 * L) ** 2)
                        / (2 * (sigma_frac * L) ** 2))


def test_geometry_closes_and_pairs():
    n = 14
    xy, tri = I.square_tri_mesh(n, jitter=0.2, seed=3)
    m = O.tri_mesh(xy, tri)
    assert m.area.sum() == pytest.approx(n * n, rel=1e-14)
    assert (m.nbr < 0).sum() == 4 * n
    for c in range(m.n_cells):
        e = slice(m.edge_start[c], m.edge_start[c + 1])
        assert abs((m.len[e] * m.eta_x[e]).sum()) <= 1e-14 and abs((m.len[e] * m.eta_y[e]).sum()) <= 1e-14
    # each interior edge from both sides: opposite normals, equal length
    for c in range(m.n_cells):
        for e in range(m.edge_start[c], m.edge_start[c + 1]):
            j = m.nbr[e]
            if j < 0:
                continue
            back = [f for f in range(m.edge_start[j], m.edge_start[j + 1]) if m.nbr[f] == c]
            assert len(back) == 1
            f = back[0]
            assert m.eta_x[f] == -m.eta_x[e] and m.eta_y[f] == -m.eta_y[e]
            assert m.len[f] == m.len[e]
    # unit normals
    assert np.abs(np.hypot(m.eta_x, m.eta_y) - 1).max() <= 1e-15


def test_rejects_bad_meshes():
    xy, tri = I.square_tri_mesh(3, jitter=0.0, shuffle=False)
    bad = tri.copy()
    bad[0] = bad[0][::-1]            # clockwise
    with pytest.raises(ValueError):
        O.tri_mesh(xy, bad)
    bad = np.concatenate([tri, tri[:1]])   # an edge shared by three triangles
    with pytest.raises(ValueError):
        O.tri_mesh(xy, bad)


def test_lake_at_rest_one_layer_on_triangles():
    n = 16
    xy, tri = I.square_tri_mesh(n, jitter=0.2, seed=4)
    m = O.tri_mesh(xy, tri)
    cxy = I.tri_centroids(xy, tri)
    H = 3.0 - bump_bottom(cxy, n)
    h = H + 1.0                       # surface at +1 m
    z = np.zeros_like(h)
    W, dts, st, _ = O.run1(m, H, [h, z, z, 0.5 * h], G, 0.9, 60)
    assert st == O.OM_OK
    assert np.abs(W[0] - h).max() <= 1e-12 * h.max()
    qs = h.max() * math.sqrt(G * h.max())
    assert np.abs(W[1]).max() <= 1e-12 * qs and np.abs(W[2]).max() <= 1e-12 * qs


def test_lake_at_rest_two_layers_on_triangles():
    n = 14
    xy, tri = I.square_tri_mesh(n, jitter=0.2, seed=5)
    m = O.tri_mesh(xy, tri)
    cxy = I.tri_centroids(xy, tri)
    H = 10.0 - bump_bottom(cxy, n, amp=3.0)
    h1 = np.full_like(H, 3.0)
    h2 = H + 1.0 - h1
    z = np.zeros_like(H)
    W, dts, st = O.run2(m, H, [h1, z, z, h2, z, z], G, 0.98, 0.9, 40)
    assert st == O.OM_OK
    assert np.abs(W[0] - h1).max() <= 1e-12 * 3.0
    assert np.abs(W[3] - h2).max() <= 1e-12 * h2.max()


def test_conservation_and_constant_concentration_on_triangles():
    n = 16
    xy, tri = I.square_tri_mesh(n, jitter=0.2, seed=6)
    m = O.tri_mesh(xy, tri)
    cxy = I.tri_centroids(xy, tri)
    rng = np.random.default_rng(6)
    H = 3.0 - bump_bottom(cxy, n)
    h = H + 1.0 + 0.3 * np.exp(-((cxy[:, 0] - 4) ** 2 + (cxy[:, 1] - 9) ** 2) / 4.0)
    qx, qy = h * rng.uniform(-0.1, 0.1, (2, h.size))
    W, dts, st, _ = O.run1(m, H, [h, qx, qy, 0.37 * h], G, 0.9, 80)
    assert st == O.OM_OK
    assert abs(W[0].dot(m.area) - h.dot(m.area)) / h.dot(m.area) <= 1e-12
    assert abs(W[3].dot(m.area) - 0.37 * h.dot(m.area)) / h.dot(m.area) <= 1e-12
    assert np.abs(W[3] / W[0] - 0.37).max() <= 1e-14
    # two layers
    h1 = 3.0 + 0.5 * np.exp(-((cxy[:, 0] - 8) ** 2 + (cxy[:, 1] - 8) ** 2) / 6.0)
    H2 = 10.0 - bump_bottom(cxy, n, amp=3.0)
    W2, _, st = O.run2(m, H2, [h1, 0 * h1, 0 * h1, H2 + 1.0 - h1, 0 * h1, 0 * h1], G, 0.98,
                       0.9, 40)
    assert st == O.OM_OK
    for k, ref in ((0, h1), (3, H2 + 1.0 - h1)):
        assert abs(W2[k].dot(m.area) - ref.dot(m.area)) / ref.dot(m.area) <= 1e-12


def strip_dam(nsq, length=2000.0, ny=4):
    side = length / nsq
    xy, tri = I.square_tri_mesh(nsq, ny, side=side, jitter=0.0, shuffle=False)
    cxy = I.tri_centroids(xy, tri)
    h = np.where(cxy[:, 0] < 1000.0, 2.0, 1.0)
    return xy, tri, cxy, h


def test_stoker_on_triangulated_strips():
    # depth and discharge against the exact solution: the discharge pins the
    # orientation of the normals (reversing all of them leaves h unchanged and
    # flips q, the equations being invariant under q -> -q, t -> -t)
    errs, errq = [], []
    for nsq in (100, 200, 400):
        xy, tri, cxy, h = strip_dam(nsq)
        m = O.tri_mesh(xy, tri)
        z = np.zeros_like(h)
        W = [h, z, z, z]
        t = 0.0
        while t < 40.0:
            W, dts, st, _ = O.run1(m, z, W, G, 0.9, 1)
            assert st == O.OM_OK
            t += dts[0]
        ha, ua = stoker.solution(cxy[:, 0], t, 1000.0, 2.0, 1.0, G)
        width = 4 * 2000.0 / nsq
        errs.append(np.abs(W[0] - ha).dot(m.area) / width)
        errq.append(np.abs(W[1] - ha * ua).dot(m.area) / width)
    for e in (errs, errq):
        ratios = [e[k] / e[k + 1] for k in range(2)]
        assert all(r >= 1.3 for r in ratios), (e, ratios)
    assert errs[-1] / (2000.0 * 1.5) < 3e-3
    assert errq[-1] / (2000.0 * 1.5 * stoker.middle_state(2.0, 1.0, G)[1]) < 1e-2


def test_half_turn_symmetry():
    # (x, y) -> (L - x, L - y) maps the diagonal-split triangulation onto itself
    n = 20
    xy, tri = I.square_tri_mesh(n, jitter=0.0, shuffle=False)
    m = O.tri_mesh(xy, tri)
    cxy = I.tri_centroids(xy, tri)
    rr = np.hypot(cxy[:, 0] - 10.0, cxy[:, 1] - 10.0)
    h = np.where(rr < 4.0, 2.0, 1.0)
    z = np.zeros_like(h)
    W, _, st, _ = O.run1(m, z, [h, z, z, h], G, 0.9, 40)
    assert st == O.OM_OK
    # partner cell under the half turn: centroid at (L - x, L - y)
    key = {(round(x, 9), round(y, 9)): c for c, (x, y) in enumerate(cxy)}
    partner = np.array([key[(round(n - x, 9), round(n - y, 9))] for x, y in cxy])
    assert np.abs(W[0] - W[0][partner]).max() <= 1e-12
    assert np.abs(W[1] + W[1][partner]).max() <= 1e-12
    assert np.abs(W[2] + W[2][partner]).max() <= 1e-12


def test_numbering_independence_on_triangles():
    n = 10
    xy, tri = I.square_tri_mesh(n, jitter=0.2, seed=8, shuffle=False)
    rng = np.random.default_rng(8)
    cxy = I.tri_centroids(xy, tri)
    h = 2.0 + 0.4 * np.exp(-((cxy[:, 0] - 3) ** 2 + (cxy[:, 1] - 6) ** 2) / 3.0)
    H = 1.0 - 0.3 * bump_bottom(cxy, n)
    z = np.zeros_like(h)
    m = O.tri_mesh(xy, tri)
    Wa, da, sa, _ = O.run1(m, H, [h, z, z, h], G, 0.9, 25)
    # renumber the vertices and the cells, and rotate each triangle's vertex
    # list (same orientation)
    vp = rng.permutation(xy.shape[0])
    xy2 = np.empty_like(xy)
    xy2[vp] = xy
    cp = rng.permutation(tri.shape[0])
    tri2 = vp[tri][cp]
    tri2 = np.roll(tri2, 1, axis=1)
    m2 = O.tri_mesh(xy2, tri2)
    Wb, db, sb, _ = O.run1(m2, H[cp], [h[cp], z, z, h[cp]], G, 0.9, 25)
    assert sa == sb == O.OM_OK
    assert np.allclose(da, db, rtol=1e-13, atol=0)
    for a, b in zip(Wa, Wb):
        assert np.abs(a[cp] - b).max() <= 1e-12 * np.abs(a).max()


def test_update2_at_is_the_update_restricted_to_the_cells():
    d = I.tri_workload(12)
    m = O.tri_mesh(d["xy"], d["tri"])
    W = I.fields2_of(d)
    full, st = O.update2(m, d["H"], W, G, d["r"], 0.05)
    assert st == O.OM_OK
    cells = np.array([0, 5, 77, d["n_cells"] - 1])
    part, st = O.update2_at(m, d["H"], W, G, d["r"], 0.05, cells)
    assert st == O.OM_OK
    for k in range(6):
        assert np.array_equal(part[k], full[k][cells])
