"""Host side of the triangle-mesh path (no GPU): mesh validation, the cell
order and the tiles, through swe_mesh_info and swe_create_mesh's argument
checks, which run entirely on the host before any device call.  Every
preparation also runs libswe's own consistency check of the tiles (each
cell's three slot references against the edges), so every call here that
succeeds has passed it."""
import ctypes as C

import numpy as np
import pytest

from finite_volume_shallow_gb300 import build as B
from finite_volume_shallow_gb300 import inputs as I
from finite_volume_shallow_gb300 import swe as S
import oracle as O


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build()
    return S.load()


def n_edges_of(tri):
    # every undirected vertex pair once
    e = np.sort(np.concatenate([tri[:, [0, 1]], tri[:, [1, 2]], tri[:, [2, 0]]]), axis=1)
    return len(np.unique(e, axis=0))


@pytest.mark.parametrize("n,m,shuffle", [(1, 1, False), (3, 2, True), (17, 5, True),
                                         (40, 40, True)])
def test_order_is_a_permutation_and_edges_are_counted(n, m, shuffle):
    xy, tri = I.square_tri_mesh(n, m, jitter=0.2, seed=n, shuffle=shuffle)
    for reorder in (0, 1):
        order, ne, nt, nev, nh = S.swe_mesh_info(xy, tri, reorder=reorder)
        assert np.array_equal(np.sort(order), np.arange(tri.shape[0]))
        assert ne == n_edges_of(tri)
        assert 1 <= nt <= tri.shape[0]
        # every edge evaluated at least once, at most once per tile it touches
        assert ne <= nev <= 2 * ne
        if nt == 1:
            assert nev == ne and nh == 0
        if reorder == 0:
            assert np.array_equal(order, np.arange(tri.shape[0]))
    # the oracle's independent edge pairing sees the same edges
    mo = O.tri_mesh(xy, tri)
    assert ne == (len(mo.nbr) + int((mo.nbr < 0).sum())) // 2


def test_hilbert_order_makes_compact_tiles():
    # a shuffled 64 x 64 square (8192 triangles): in the caller's numbering a
    # run of consecutive cells is scattered over the mesh, so nearly every
    # edge of a tile is shared with another tile; in the internal order the
    # tiles are compact patches
    xy, tri = I.square_tri_mesh(64, jitter=0.2, seed=9, shuffle=True)
    n = tri.shape[0]
    _, ne, nt0, nev0, nh0 = S.swe_mesh_info(xy, tri, reorder=0)
    order, ne1, nt, nev, nh = S.swe_mesh_info(xy, tri, reorder=1)
    assert ne1 == ne
    assert nev0 > 1.8 * ne and nh0 > 2 * n
    assert nev < 1.10 * ne and nh < 0.2 * n
    # tiles hold about 300 cells: at most 511 edges each, 1.5 per cell
    assert 250 <= n / nt <= 400
    # consecutive cells of the internal order are close in the plane: the
    # step between them is about one cell, never more than a few on average
    c = I.tri_centroids(xy, tri)
    inv = np.empty(n, dtype=np.int64)
    inv[order] = np.arange(n)
    step = np.hypot(*(c[inv[1:]] - c[inv[:-1]]).T)
    assert np.median(step) < 1.0 and step.mean() < 2.0


def test_tiles_of_a_graded_mesh():
    # cells of very different sizes: tiles are cut by counts, not by area
    xy, tri = I.square_tri_mesh(48, jitter=0.2, seed=4, shuffle=True)
    xy = np.ascontiguousarray(np.stack([xy[:, 0] ** 3 / 48.0 ** 2, xy[:, 1]], axis=1))
    order, ne, nt, nev, nh = S.swe_mesh_info(xy, tri)
    assert np.array_equal(np.sort(order), np.arange(tri.shape[0]))
    assert nev < 1.15 * ne


def test_disconnected_components_are_all_ordered():
    xy1, tri1 = I.square_tri_mesh(5, jitter=0.0, shuffle=False)
    xy2 = xy1 + np.array([100.0, 0.0])
    xy = np.ascontiguousarray(np.concatenate([xy1, xy2]))
    tri = np.ascontiguousarray(np.concatenate([tri1, tri1 + xy1.shape[0]]).astype(np.int32))
    order, ne, nt, nev, nh = S.swe_mesh_info(xy, tri)
    assert np.array_equal(np.sort(order), np.arange(tri.shape[0]))
    assert ne == 2 * n_edges_of(tri1)
    assert nt == 1 and nev == ne and nh == 0


def bad_meshes():
    xy, tri = I.square_tri_mesh(3, jitter=0.0, shuffle=False)
    out = {}
    t = tri.copy()
    t[0] = t[0][::-1]
    out["clockwise"] = (xy, t)
    t = tri.copy()
    t[1, 2] = t[1, 0]
    out["degenerate"] = (xy, t)
    t = tri.copy()
    t[2, 1] = xy.shape[0]
    out["index_high"] = (xy, t)
    t = tri.copy()
    t[2, 1] = -1
    out["index_negative"] = (xy, t)
    out["edge_of_three"] = (xy, np.ascontiguousarray(np.concatenate([tri, tri[:1]])))
    x = xy.copy()
    x[4, 0] = np.nan
    out["nan_vertex"] = (x, tri)
    # collinear vertices (zero area)
    x = np.array([[0.0, 0.0], [1.0, 0.0], [2.0, 0.0]])
    out["zero_area"] = (x, np.array([[0, 1, 2]], dtype=np.int32))
    return out


@pytest.mark.parametrize("name", sorted(bad_meshes()))
def test_invalid_meshes_are_rejected_on_the_host(name):
    xy, tri = bad_meshes()[name]
    tri = np.ascontiguousarray(tri, dtype=np.int32)
    with pytest.raises(S.SweError) as e:
        S.swe_mesh_info(xy, tri)
    assert e.value.status == S.SWE_ERR_ARG
    n = tri.shape[0]
    W = [np.ones(n), np.zeros(n), np.zeros(n), np.zeros(n)]
    with pytest.raises(S.SweError) as e:
        S.swe_create_mesh(xy, tri, np.zeros(n), W, precision=64)
    assert e.value.status == S.SWE_ERR_ARG


def test_create_mesh_rejects_bad_parameters_on_the_host():
    xy, tri = I.square_tri_mesh(2, jitter=0.0, shuffle=False)
    n = tri.shape[0]
    W1 = [np.ones(n), np.zeros(n), np.zeros(n), np.zeros(n)]
    W2 = [np.ones(n), np.zeros(n), np.zeros(n), np.ones(n), np.zeros(n), np.zeros(n)]
    cases = [
        (dict(precision=64, cfl=0.0), W1, S.SWE_ERR_ARG),
        (dict(precision=64, n_layers=2, pollutant=0, r=1.0), W2, S.SWE_ERR_ARG),
        (dict(precision=64, n_layers=2, pollutant=1, r=0.5), W2, S.SWE_ERR_UNSUPPORTED),
        (dict(precision=64, pollutant=0), W1, S.SWE_ERR_UNSUPPORTED),
        (dict(precision=64, reorder=2), W1, S.SWE_ERR_ARG),
    ]
    for kw, W, expect in cases:
        with pytest.raises(S.SweError) as e:
            S.swe_create_mesh(xy, tri, np.zeros(n), W, **kw)
        assert e.value.status == expect, kw
    with pytest.raises(ValueError):
        S.swe_create_mesh(xy, tri.astype(np.int64), np.zeros(n), W1)
    with pytest.raises(ValueError):
        S.swe_create_mesh(xy, tri, np.zeros(n), W1, precision=16)
    L = S.load()
    out = C.c_void_p(7)
    assert L.swe_create_mesh(None, None, None, None, C.byref(out)) == S.SWE_ERR_ARG
    assert out.value is None
    assert L.swe_mesh_info(None, None, None, None, None, None) == S.SWE_ERR_ARG
    assert L.swe_cell_index(None, None) == S.SWE_ERR_ARG
