"""Pins of the two-layer oracle (An MPI-CUDA implementation of an improved Roe
method for two-layer shallow water systems, Sec. 2.1 eq. (1) and Sec. 2.2,
the IR-Roe flux with four components in the normal frame).

* eigenvalues against a library eigen-solver, and the r = 0 closed form;
* loss of hyperbolicity reported exactly when the library finds complex
  eigenvalues;
* the flux of equal states is the physical flux of eq. (1);
* path conservation: F_ij^- + F_ji^- equals minus the coupling and
  bathymetry terms integrated over the edge;
* r = 0 decouples the lower layer, which then follows the one-layer scheme;
* two-layer lake at rest over hills (flat surface and flat interface);
* mass of each layer conserved with walls; y-invariance of a 1D problem;
* bitwise transpose symmetry of a radial interface bump; numbering
  independence on a permuted mesh.
"""
import math

import numpy as np
import pytest

import oracle as O
from finite_volume_shallow_gb300 import inputs as I

G = 9.81


def roe_matrix(u1, u2, c1s, c2s, r):
    return np.array([[0, 1, 0, 0], [c1s - u1 * u1, 2 * u1, c1s, 0], [0, 0, 0, 1],
                     [r * c2s, 0, c2s - u2 * u2, 2 * u2]], dtype=np.float64)


def test_roots_against_library_eigensolver():
    rng = np.random.default_rng(10)
    nh = 0
    for _ in range(3000):
        u1, u2 = rng.uniform(-3, 3, 2)
        c1s, c2s = rng.uniform(0.5, 80, 2)
        r = rng.uniform(0, 0.999)
        ev = np.linalg.eigvals(roe_matrix(u1, u2, c1s, c2s, r))
        st, lam = O.roots2(u1, u2, c1s, c2s, r)
        scale = np.abs(ev).max()
        if np.abs(ev.imag).max() > 1e-7 * scale:
            assert st == O.OM_ERR_HYPERBOLIC
            nh += 1
        elif st == O.OM_OK:
            assert np.abs(np.sort(ev.real) - lam).max() <= 1e-12 * scale
    assert nh > 50   # the sample does contain non-hyperbolic states


def test_roots_decouple_at_r0():
    rng = np.random.default_rng(11)
    for _ in range(200):
        u1, u2 = rng.uniform(-2, 2, 2)
        c1s, c2s = rng.uniform(1, 60, 2)
        st, lam = O.roots2(u1, u2, c1s, c2s, 0.0)
        want = np.sort([u1 - math.sqrt(c1s), u1 + math.sqrt(c1s),
                        u2 - math.sqrt(c2s), u2 + math.sqrt(c2s)])
        assert st == O.OM_OK
        assert np.abs(lam - want).max() <= 1e-14 * np.abs(want).max()


def test_roots_of_equal_layers():
    # c1 = c2 = c and u1 = u2 = u: p = Q^2 - r c^4, so the roots are
    # u -+ c sqrt(1 +- sqrt(r)) in closed form; the roots of Q1 and Q2
    # coincide here (the inner pair must still be found), also after
    # perturbations at the rounding level
    rng = np.random.default_rng(18)
    for _ in range(300):
        u = rng.uniform(-1, 1) * 10.0 ** rng.integers(-14, 1)
        cs = rng.uniform(1, 80)
        r = rng.uniform(0, 0.999)
        eps = rng.uniform(-1, 1, 3) * 1e-14 * np.array([1.0, cs, cs])
        st, lam = O.roots2(u, u + eps[0], cs + eps[1], cs + eps[2], r)
        c = math.sqrt(cs)
        want = np.sort([u - c * math.sqrt(1 + math.sqrt(r)), u - c * math.sqrt(1 - math.sqrt(r)),
                        u + c * math.sqrt(1 - math.sqrt(r)), u + c * math.sqrt(1 + math.sqrt(r))])
        assert st == O.OM_OK, (u, cs, r)
        assert np.abs(lam - want).max() <= 1e-9 * c


def phys_flux2(W, eta, g=G):
    out = np.zeros(6)
    for k in range(2):
        h, qx, qy = W[3 * k: 3 * k + 3]
        F1 = np.array([qx, qx * qx / h + 0.5 * g * h * h, qx * qy / h])
        F2 = np.array([qy, qx * qy / h, qy * qy / h + 0.5 * g * h * h])
        out[3 * k: 3 * k + 3] = F1 * eta[0] + F2 * eta[1]
    return out


def random_state2(rng, umax=0.5):
    h1, h2 = rng.uniform(1.0, 6.0, 2)
    u = rng.uniform(-umax, umax, 4)
    return np.array([h1, h1 * u[0], h1 * u[1], h2, h2 * u[2], h2 * u[3]])


def test_consistency_equal_states():
    rng = np.random.default_rng(12)
    for _ in range(200):
        W = random_state2(rng, umax=0.1)   # shear small enough to stay hyperbolic
        th = rng.uniform(0, 2 * np.pi)
        eta = (math.cos(th), math.sin(th))
        st, F, D = O.flux2(W, W, 0.4, 0.4, eta, G, 0.98)
        assert st == O.OM_OK
        Fp = phys_flux2(W, eta)
        assert np.allclose(F, Fp, rtol=1e-11, atol=1e-11 * np.abs(Fp).max())


def test_path_conservation_identity():
    rng = np.random.default_rng(13)
    done = 0
    while done < 200:
        Wi, Wj = random_state2(rng, 0.1), random_state2(rng, 0.1)
        th = rng.uniform(0, 2 * np.pi)
        eta = np.array([math.cos(th), math.sin(th)])
        Hi, Hj = rng.uniform(-1, 1, 2) + 10
        r = rng.uniform(0.5, 0.99)
        s1, Fij, _ = O.flux2(Wi, Wj, Hi, Hj, eta, G, r)
        s2, Fji, _ = O.flux2(Wj, Wi, Hj, Hi, -eta, G, r)
        if s1 != O.OM_OK or s2 != O.OM_OK:
            continue
        hb1 = 0.5 * (Wi[0] + Wj[0])
        hb2 = 0.5 * (Wi[3] + Wj[3])
        dH = Hj - Hi
        s_up = G * hb1 * (dH - (Wj[3] - Wi[3]))
        s_lo = G * hb2 * (dH - r * (Wj[0] - Wi[0]))
        expect = -np.array([0, s_up * eta[0], s_up * eta[1], 0, s_lo * eta[0], s_lo * eta[1]])
        scale = np.abs(Fij).max() + abs(s_up) + abs(s_lo)
        assert np.allclose(Fij + Fji, expect, rtol=0, atol=1e-11 * scale)
        done += 1


def test_hyperbolicity_loss_reported():
    # strong shear between the layers makes the inner eigenvalues complex
    Wi = np.array([3.0, 3.0 * 2.0, 0.0, 3.0, -3.0 * 2.0, 0.0])
    st, F, D = O.flux2(Wi, Wi, 0.0, 0.0, (1.0, 0.0), G, 0.98)
    assert st == O.OM_ERR_HYPERBOLIC


def test_lower_layer_decouples_at_r0():
    nx, ny = 24, 14
    d = I.make_workload("pulses8192", nx=nx, ny=ny)
    rng = np.random.default_rng(14)
    h1 = rng.uniform(1.0, 2.0, nx * ny)
    q1x, q1y = rng.uniform(-0.2, 0.2, (2, nx * ny))
    W2 = [h1, q1x, q1y, d["h"], d["qx"], d["qy"]]
    m = O.grid_mesh(nx, ny, d["dx"], d["dy"])
    dt = 0.4
    Wa, sa = O.update2(m, d["H"], W2, G, 0.0, dt)
    Wb, sb = O.update1(m, d["H"], [d["h"], d["qx"], d["qy"], d["hC"]], G, dt)
    assert sa == sb == O.OM_OK
    for a, b in zip(Wa[3:], Wb[:3]):
        assert np.abs(a - b).max() <= 1e-13 * np.abs(b).max()


def lake2(nx, ny, seed=15):
    d = I.make_workload("hills2048", nx=nx, ny=ny, lake_at_rest=True)
    H = d["H"] + 10.0                      # bottom 10 m further down
    h1 = np.full(nx * ny, 3.0)             # flat interface 3 m below the surface
    h2 = H + 5.0 - h1                      # surface at +5 m
    z = np.zeros(nx * ny)
    return H, [h1, z, z, h2, z.copy(), z.copy()]


def test_two_layer_lake_at_rest():
    nx, ny = 40, 32
    H, W = lake2(nx, ny)
    Wf, dts, st = O.grid_run2(nx, ny, 10.0, 10.0, H, W, G, 0.98, 0.9, 60)
    assert st == O.OM_OK
    for k in (0, 3):
        assert np.abs(Wf[k] - W[k]).max() <= 1e-13 * W[k].max()
    qs = W[3].max() * math.sqrt(G * W[3].max())
    for k in (1, 2, 4, 5):
        assert np.abs(Wf[k]).max() <= 1e-13 * qs


def interface_dam(nx, ny, dx=10.0, x_split=None):
    L = nx * dx
    x = (np.arange(nx) + 0.5) * dx
    xs = L / 2 if x_split is None else x_split
    h1 = np.tile(np.where(x < xs, 6.0, 4.0), (ny, 1)).reshape(-1)
    H = np.full(nx * ny, 10.0)
    z = np.zeros(nx * ny)
    return H, [h1, z, z, H - h1, z.copy(), z.copy()]


def test_layer_mass_conservation_and_y_invariance():
    nx, ny = 64, 6
    H, W = interface_dam(nx, ny)
    Wf, dts, st = O.grid_run2(nx, ny, 10.0, 10.0, H, W, G, 0.98, 0.9, 120)
    assert st == O.OM_OK
    for k in (0, 3):
        assert abs(Wf[k].sum() - W[k].sum()) / W[k].sum() <= 1e-12
    for k in range(6):
        rows = Wf[k].reshape(ny, nx)
        assert np.array_equal(rows, np.tile(rows[0], (ny, 1)))
    assert np.all(Wf[2] == 0) and np.all(Wf[5] == 0)
    assert np.abs(Wf[1]).max() > 1e-3        # the interface moved


def test_moving_layers_conserve_mass():
    nx, ny = 30, 22
    rng = np.random.default_rng(16)
    H, W = lake2(nx, ny)
    W = [w.copy() for w in W]
    W[0] = W[0] + 0.3 * rng.uniform(0, 1, nx * ny)
    for k in (1, 2):
        W[k] = W[0] * rng.uniform(-0.05, 0.05, nx * ny)
    for k in (4, 5):
        W[k] = W[3] * rng.uniform(-0.05, 0.05, nx * ny)
    Wf, dts, st = O.grid_run2(nx, ny, 10.0, 10.0, H, W, G, 0.95, 0.9, 40)
    assert st == O.OM_OK
    for k in (0, 3):
        assert abs(Wf[k].sum() - W[k].sum()) / W[k].sum() <= 1e-12


def test_radial_interface_bump_symmetry():
    n = 32
    x = (np.arange(n) + 0.5) * 10.0
    X, Y = np.meshgrid(x, x)
    rr = np.hypot(X - 160.0, Y - 160.0)
    h1 = (3.0 + 1.0 * np.exp(-(rr / 60.0) ** 2)).reshape(-1)
    H = np.full(n * n, 10.0)
    z = np.zeros(n * n)
    Wf, _, st = O.grid_run2(n, n, 10.0, 10.0, H, [h1, z, z, H - h1, z.copy(), z.copy()],
                            G, 0.98, 0.9, 40)
    assert st == O.OM_OK
    a = [w.reshape(n, n) for w in Wf]
    assert np.array_equal(a[0], a[0].T) and np.array_equal(a[3], a[3].T)
    assert np.array_equal(a[1], a[2].T) and np.array_equal(a[4], a[5].T)
    assert np.abs(a[0] - a[0][:, ::-1]).max() <= 1e-12
    assert np.abs(a[1] + a[1][:, ::-1]).max() <= 1e-12


def test_two_layer_numbering_independence():
    nx, ny = 14, 11
    H, W = lake2(nx, ny)
    rng = np.random.default_rng(17)
    W = [w.copy() for w in W]
    W[0] = W[0] + 0.5 * rng.uniform(0, 1, nx * ny)
    m = O.grid_mesh(nx, ny, 10.0, 10.0)
    perm = rng.permutation(nx * ny)
    inv = np.argsort(perm)
    counts = np.diff(m.edge_start)
    es = np.concatenate([[0], np.cumsum(counts[inv])])
    idx = np.concatenate([np.arange(m.edge_start[o], m.edge_start[o + 1]) for o in inv])
    nbr = np.where(m.nbr[idx] >= 0, perm[np.maximum(m.nbr[idx], 0)], -1)
    mp = O.Mesh(m.area[inv], es, nbr, m.eta_x[idx], m.eta_y[idx], m.len[idx])
    Wa, da, sa = O.run2(m, H, W, G, 0.98, 0.9, 20)
    Wb, db, sb = O.run2(mp, H[inv], [w[inv] for w in W], G, 0.98, 0.9, 20)
    assert sa == sb == O.OM_OK and np.array_equal(da, db)
    for a, b in zip(Wa, Wb):
        assert np.abs(a[inv] - b).max() <= 1e-13 * np.abs(a).max()


# ---- the Harten-Hyman entropy fix with two layers ---------------------------
def test_entropy_fix_lower_layer_decouples_at_r0():
    # With r = 0 the lower layer is the one-layer system over H, and the
    # eigenvectors of its two waves have no upper-layer part in K^-1, so the
    # two-layer fix must give the lower layer exactly the one-layer fix (whose
    # own pins tie it to Stoker's solution).  The lower layer is the
    # transonic dam break h 10 m / 0.5 m; the upper layer is 50-59.5 m thick
    # with a flat surface, so its speeds (+-23 m/s) stay clear of the lower
    # layer's and the eigenvector basis is well conditioned.
    nx = 200
    d = I.dam_break_1d(nx, h_left=10.0, h_right=0.5)
    h2 = d["h"]
    z = np.zeros(h2.size)
    m = O.grid_mesh(nx, 4, d["dx"], d["dy"])
    dt = 0.15   # below the CFL limit of the initial state (0.186 s)
    lower = {}
    for fix in (0, 1):
        W2 = [60.0 - h2, z, z, h2, z, z]
        W1 = [h2, z, z, d["hC"]]
        with O.entropy_fix(fix):
            for _ in range(40):
                W2, s2 = O.update2(m, d["H"], W2, G, 0.0, dt)
                W1, s1 = O.update1(m, d["H"], W1, G, dt)
                assert s1 == s2 == O.OM_OK
        for a, b in zip(W2[3:], W1[:3]):
            assert np.abs(a - b).max() <= 1e-13 * np.abs(b).max()
        lower[fix] = W2[3]
    assert np.abs(lower[0] - lower[1]).max() > 0.1   # the fix acts here


def test_entropy_fix_two_layers_at_rest_and_conservative():
    nx, ny = 40, 32
    H, W = lake2(nx, ny)
    with O.entropy_fix():
        Wf, _, st = O.grid_run2(nx, ny, 10.0, 10.0, H, W, G, 0.98, 0.9, 60)
    assert st == O.OM_OK
    for k in (0, 3):
        assert np.abs(Wf[k] - W[k]).max() <= 1e-13 * W[k].max()
    qs = W[3].max() * math.sqrt(G * W[3].max())
    for k in (1, 2, 4, 5):
        assert np.abs(Wf[k]).max() <= 1e-13 * qs
    # a radial transonic dam break in the lower layer at r = 0.5: each
    # layer's mass is conserved with the fix on
    d = I.circular_dam(48, 40, dx=5.0, radius=60.0, h_in=10.0, h_out=0.5)
    h2 = d["h"]
    z = np.zeros(h2.size)
    W = [30.0 - h2, z, z, h2, z, z]
    with O.entropy_fix():
        Wf, _, st = O.grid_run2(48, 40, 5.0, 5.0, d["H"], W, G, 0.5, 0.9, 60)
    assert st == O.OM_OK
    for k in (0, 3):
        assert abs(Wf[k].sum() - W[k].sum()) <= 1e-12 * W[k].sum()
