"""Pins of the fp64 CPU oracle against what the mathematics fixes.

The oracle restates An MPI-CUDA implementation of an improved Roe method for
two-layer shallow water systems, Sec. 2.2 (update eq. (4), flux steps 1-4,
CFL eq. (5)) for one layer plus a passive pollutant.  The pages print no worked
numerical example, so each test below checks a property that an error in the
oracle (dropped term, wrong sign or index, transposed operand) would break:

* consistency: the flux of two equal states is the physical flux F_eta(W) of
  eq. (1), written out from the model;
* the linear acoustic Riemann problem at rest, solved by hand;
* supercritical upwinding (P^- = 0 or I);
* path conservation: F_ij^- + F_ji^- equals the bathymetry source term;
* lake at rest over variable bathymetry (the well-balanced / C-property claim
  of Sec. 2.2);
* mass and pollutant conservation with reflective walls;
* a constant concentration stays constant;
* Stoker's analytic dam-break solution, with the L1 error decreasing under
  refinement;
* bitwise x/y transpose symmetry and mirror symmetry of the radial dam break;
* independence of the cell numbering on the polygon-mesh path;
* a two-cell dam break whose single step is derived by hand.
"""
import math

import numpy as np
import pytest

import oracle as O
from finite_volume_shallow_gb300 import inputs as I
import stoker

G = 9.81


def phys_flux(W, eta, g=G):
    """F_eta(W) = F_1(W) eta_x + F_2(W) eta_y of eq. (1), one layer, plus the
    pollutant flux (q . eta) C of the transport equation."""
    h, qx, qy, hC = W
    F1 = np.array([qx, qx * qx / h + 0.5 * g * h * h, qx * qy / h, qx * hC / h])
    F2 = np.array([qy, qx * qy / h, qy * qy / h + 0.5 * g * h * h, qy * hC / h])
    return F1 * eta[0] + F2 * eta[1]


def random_states(rng, n, umax=1.0):
    h = rng.uniform(0.5, 5.0, n)
    u = rng.uniform(-umax, umax, (2, n))
    C = rng.uniform(0.0, 1.0, n)
    return np.stack([h, h * u[0], h * u[1], h * C], axis=1)


def random_normals(rng, n):
    th = rng.uniform(0, 2 * np.pi, n)
    return np.stack([np.cos(th), np.sin(th)], axis=1)


def test_consistency_equal_states():
    rng = np.random.default_rng(1)
    for W, eta in zip(random_states(rng, 200, umax=8.0), random_normals(rng, 200)):
        F, D = O.flux1(W, W, 0.3, 0.3, eta, G)
        Fp = phys_flux(W, eta)
        assert np.allclose(F, Fp, rtol=1e-12, atol=1e-12 * np.abs(Fp).max())
        un = (W[1] * eta[0] + W[2] * eta[1]) / W[0]
        assert D == pytest.approx(abs(un) + math.sqrt(G * W[0]), rel=1e-13)


@pytest.mark.parametrize("eta", [(1.0, 0.0), (0.0, 1.0), (-1.0, 0.0), (0.6, -0.8)])
def test_acoustic_riemann_at_rest(eta):
    # Flat bottom, both states at rest: u_bar = 0, lambda = -+ c_bar,
    # d = (0, g (hR^2 - hL^2) / 2), P^- d = alpha_1 (1, -c) with
    # alpha_1 = -d_1 / (2 c).  Hence mass flux c (hL - hR) / 2 and normal
    # momentum flux g (hL^2 + hR^2) / 4, no tangential momentum.
    hL, hR, CL, CR = 2.5, 0.75, 0.3, 0.9
    F, D = O.flux1([hL, 0, 0, hL * CL], [hR, 0, 0, hR * CR], 0.0, 0.0, eta, G)
    c = math.sqrt(G * 0.5 * (hL + hR))
    mass = c * (hL - hR) / 2
    mom = G * (hL * hL + hR * hR) / 4
    assert F[0] == pytest.approx(mass, rel=1e-14)
    assert F[1] == pytest.approx(mom * eta[0], rel=1e-14, abs=1e-14)
    assert F[2] == pytest.approx(mom * eta[1], rel=1e-14, abs=1e-14)
    assert F[3] == pytest.approx(mass * CL, rel=1e-14)   # upwind from the left
    assert D == pytest.approx(c, rel=1e-15)
    # reversed jump: mass flows from j into i and carries j's concentration
    F2, _ = O.flux1([hR, 0, 0, hR * CR], [hL, 0, 0, hL * CL], 0.0, 0.0, eta, G)
    assert F2[0] == pytest.approx(-mass, rel=1e-14)
    assert F2[3] == pytest.approx(-mass * CL, rel=1e-14)


def test_supercritical_upwind():
    rng = np.random.default_rng(2)
    for _ in range(100):
        eta = random_normals(rng, 1)[0]
        h = rng.uniform(0.5, 2.0, 2)
        c = np.sqrt(G * h.max())
        un = rng.uniform(3.0, 5.0, 2) * c          # both states supercritical
        ut = rng.uniform(-1, 1, 2)
        perp = np.array([-eta[1], eta[0]])
        W = [np.array([h[k], *(h[k] * (un[k] * eta + ut[k] * perp)), h[k] * 0.5]) for k in range(2)]
        F, _ = O.flux1(W[0], W[1], 0.0, 0.0, eta, G)
        Fp = phys_flux(W[0], eta)
        assert np.allclose(F, Fp, rtol=1e-12, atol=1e-12 * np.abs(Fp).max())
        # flow against the normal: both eigenvalues negative, P^- = I, the
        # flux is the downstream state's (flat bottom)
        Wn = [np.array([w[0], -w[1], -w[2], w[3]]) for w in W]
        F, _ = O.flux1(Wn[0], Wn[1], 0.0, 0.0, eta, G)
        Fp = phys_flux(Wn[1], eta)
        assert np.allclose(F, Fp, rtol=1e-12, atol=1e-12 * np.abs(Fp).max())


def shock_pair(hL, hR, uL, family, g=G):
    """States joined by a single shock (Rankine-Hugoniot): in the shock
    frame the mass flux m = h v is continuous and
    m^2 = g hL hR (hL + hR) / 2.  family -1 / +1 picks the 1- or 2-shock."""
    vL = -family * math.sqrt(0.5 * g * hR * (hL + hR) / hL)
    vR = hL * vL / hR
    s = uL - vL
    return s, s + vR


@pytest.mark.parametrize("family", [-1, 1])
def test_isolated_shock_is_resolved_exactly(family):
    # Roe's linearisation has the jump of a single shock as an eigenvector
    # with the shock speed as eigenvalue, so the flux is the upwind physical
    # flux: F(W_L) if the shock moves towards j, F(W_R) otherwise.  A wrong
    # average (e.g. the arithmetic mean of velocities) breaks this.
    rng = np.random.default_rng(6 + family)
    for _ in range(100):
        hL, hR = rng.uniform(0.5, 4.0, 2)
        if (hR > hL) != (family == 1):
            hL, hR = hR, hL          # admissible (compressive) shocks only
        uL = rng.uniform(-6, 6)
        s, uR = shock_pair(hL, hR, uL, family)
        eta = random_normals(rng, 1)[0]
        WL = np.array([hL, hL * uL * eta[0], hL * uL * eta[1], hL * 0.2])
        WR = np.array([hR, hR * uR * eta[0], hR * uR * eta[1], hR * 0.7])
        F, _ = O.flux1(WL, WR, 0.0, 0.0, eta, G)
        up = WL if s > 0 else WR
        Fp = phys_flux(up, eta)
        scale = np.abs(Fp[:3]).max()
        assert np.allclose(F[:3], Fp[:3], rtol=0, atol=1e-12 * scale), (s, F, Fp)


def test_path_conservation_identity():
    # F_ij^- + F_ji^- = -(0, g hbar (H_j - H_i) eta, 0): the two one-sided
    # fluxes differ only by the bathymetry source integrated over the edge.
    rng = np.random.default_rng(3)
    S = random_states(rng, 400, umax=3.0)
    etas = random_normals(rng, 200)
    Hs = rng.uniform(-2, 2, (200, 2))
    for k in range(200):
        Wi, Wj, eta = S[2 * k], S[2 * k + 1], etas[k]
        Fij, Dij = O.flux1(Wi, Wj, Hs[k, 0], Hs[k, 1], eta, G)
        Fji, Dji = O.flux1(Wj, Wi, Hs[k, 1], Hs[k, 0], -eta, G)
        hbar = 0.5 * (Wi[0] + Wj[0])
        src = G * hbar * (Hs[k, 1] - Hs[k, 0])
        expect = np.array([0.0, -src * eta[0], -src * eta[1], 0.0])
        scale = np.abs(Fij).max() + abs(src)
        assert np.allclose(Fij + Fji, expect, rtol=0, atol=1e-13 * scale)
        assert Dij == pytest.approx(Dji, rel=1e-14)


def test_wall_ghost_is_mirror():
    rng = np.random.default_rng(4)
    for W, eta in zip(random_states(rng, 50), random_normals(rng, 50)):
        Wg = O.wall_ghost1(W, eta)
        qn = W[1] * eta[0] + W[2] * eta[1]
        qt = -W[1] * eta[1] + W[2] * eta[0]
        qng = Wg[1] * eta[0] + Wg[2] * eta[1]
        qtg = -Wg[1] * eta[1] + Wg[2] * eta[0]
        assert Wg[0] == W[0] and Wg[3] == W[3]
        assert qng == pytest.approx(-qn, abs=1e-14) and qtg == pytest.approx(qt, abs=1e-14)
        # no mass or pollutant crosses the wall; the normal momentum flux is
        # the pressure plus the reflected-shock term q_n^2/h + g h^2/2 + c q_n
        F, D = O.flux1(W, Wg, 0.0, 0.0, eta, G)
        c = math.sqrt(G * W[0])
        assert abs(F[0]) <= 1e-14 * (abs(qn) + 1) and abs(F[3]) <= 1e-14 * (abs(qn) + 1)
        pn = qn * qn / W[0] + 0.5 * G * W[0] ** 2 + c * qn
        assert F[1] * eta[0] + F[2] * eta[1] == pytest.approx(pn, rel=1e-13)
        assert D == pytest.approx(c, rel=1e-15)


def test_lake_at_rest_c_property():
    d = I.make_workload("hills2048", nx=64, ny=48, lake_at_rest=True)
    h0 = d["h"].copy()
    W, dts, st = O.run_grid(d, nsteps=100)
    assert st == O.OM_OK and len(dts) == 100
    scale = np.abs(h0).max()
    assert np.abs(W[0] - h0).max() <= 1e-13 * scale
    qscale = scale * math.sqrt(G * scale)
    assert np.abs(W[1]).max() <= 1e-13 * qscale
    assert np.abs(W[2]).max() <= 1e-13 * qscale


def test_conservation_with_walls():
    d = I.make_workload("pulses8192", nx=96, ny=80)     # moving water, hills
    W, dts, st = O.run_grid(d, nsteps=200)
    assert st == O.OM_OK
    for k, name in ((0, "h"), (3, "hC")):
        m0, m1 = d[name].sum(), W[k].sum()
        assert abs(m1 - m0) / m0 <= 1e-12, name
    # momentum is not conserved (walls and bottom push), so it must change
    assert np.abs(W[1] - d["qx"]).max() > 1e-3


def test_constant_concentration_stays_constant():
    d = I.make_workload("pulses8192", nx=64, ny=64)
    d["hC"] = 0.37 * d["h"]
    W, _, st = O.run_grid(d, nsteps=100)
    assert st == O.OM_OK
    assert np.abs(W[3] / W[0] - 0.37).max() <= 1e-14


def test_stoker_dam_break_convergence():
    errs = []
    for nx in (200, 400, 800, 1600):
        d = I.dam_break_1d(nx)
        mesh = O.grid_mesh(nx, 4, d["dx"], d["dy"])
        W = [d["h"], d["qx"], d["qy"], d["hC"]]
        t = 0.0
        while t < 40.0:
            W, dts, st, _ = O.run1(mesh, d["H"], W, G, 0.9, 1)
            assert st == O.OM_OK
            t += dts[0]
        x = (np.arange(nx) + 0.5) * d["dx"]
        ha, ua = stoker.solution(x, t, 1000.0, 2.0, 1.0, G)
        h = W[0].reshape(4, nx)
        assert np.array_equal(h, np.tile(h[0], (4, 1)))    # rows identical
        assert np.all(W[2] == 0.0)                          # no transverse flow
        errs.append(np.sum(np.abs(h[0] - ha)) * d["dx"])
    ratios = [errs[k] / errs[k + 1] for k in range(3)]
    assert all(r >= 1.3 for r in ratios), (errs, ratios)
    # a first-order scheme is within a few per cent of the exact profile
    assert errs[-1] / (2000.0 * 1.5) < 2e-3


def test_stoker_anisotropic_cells():
    # a y-invariant problem sees the cell aspect ratio only through dt: with
    # dy = 2.5 dx the transverse edges weigh less in eq. (5), dt grows and the
    # scheme is a little less diffusive, but the waves must still sit where
    # Stoker puts them (an edge length applied to the wrong direction would
    # move them by a factor 2.5)
    nx = 800
    errs = []
    for aspect in (1.0, 2.5):
        d = I.dam_break_1d(nx)
        mesh = O.grid_mesh(nx, 4, d["dx"], aspect * d["dx"])
        W = [d["h"], d["qx"], d["qy"], d["hC"]]
        t = 0.0
        while t < 40.0:
            W, dts, st, _ = O.run1(mesh, d["H"], W, G, 0.9, 1)
            t += dts[0]
        x = (np.arange(nx) + 0.5) * d["dx"]
        ha, _ = stoker.solution(x, t, 1000.0, 2.0, 1.0, G)
        errs.append(np.sum(np.abs(W[0].reshape(4, nx)[0] - ha)) * d["dx"])
    assert 0.6 * errs[0] <= errs[1] <= 1.02 * errs[0], errs


def test_stoker_reference_itself():
    # the analytic middle state satisfies both Rankine-Hugoniot conditions
    # of the shock and the rarefaction's Riemann invariant
    hm, um, s = stoker.middle_state(2.0, 1.0, G)
    assert 1.0 < hm < 2.0
    assert s * (hm - 1.0) == pytest.approx(hm * um, rel=1e-12)
    assert s * hm * um == pytest.approx(hm * um * um + 0.5 * G * (hm * hm - 1.0), rel=1e-12)
    assert um + 2 * math.sqrt(G * hm) == pytest.approx(2 * math.sqrt(G * 2.0), rel=1e-12)


def test_radial_dam_symmetry():
    d = I.make_workload("dam128")
    W, dts, st = O.run_grid(d, nsteps=100)
    assert st == O.OM_OK
    h, qx, qy, hC = (w.reshape(128, 128) for w in W)
    # transpose: bitwise (the pairwise (E+N)+(W+S) sum maps to itself)
    assert np.array_equal(h, h.T) and np.array_equal(hC, hC.T)
    assert np.array_equal(qx, qy.T)
    # mirror x -> L - x and y -> L - y: to round-off
    assert np.abs(h - h[:, ::-1]).max() <= 1e-12
    assert np.abs(qx + qx[:, ::-1]).max() <= 1e-12
    assert np.abs(qy - qy[:, ::-1]).max() <= 1e-12
    assert np.abs(h - h[::-1, :]).max() <= 1e-12


def test_cell_numbering_independence():
    nx, ny = 20, 15
    d = I.make_workload("pulses8192", nx=nx, ny=ny)
    m = O.grid_mesh(nx, ny, d["dx"], d["dy"])
    rng = np.random.default_rng(5)
    perm = rng.permutation(nx * ny)          # new index of old cell i: perm[i]
    inv = np.argsort(perm)                   # old index of new cell k
    counts = np.diff(m.edge_start)
    es = np.concatenate([[0], np.cumsum(counts[inv])])
    idx = np.concatenate([np.arange(m.edge_start[o], m.edge_start[o + 1]) for o in inv])
    nbr = np.where(m.nbr[idx] >= 0, perm[np.maximum(m.nbr[idx], 0)], -1)
    mp = O.Mesh(m.area[inv], es, nbr, m.eta_x[idx], m.eta_y[idx], m.len[idx])
    W0 = [d[k] for k in ("h", "qx", "qy", "hC")]
    Wa, dta, sa, _ = O.run1(m, d["H"], W0, G, 0.9, 50)
    Wb, dtb, sb, _ = O.run1(mp, d["H"][inv], [w[inv] for w in W0], G, 0.9, 50)
    assert sa == sb == O.OM_OK
    assert np.array_equal(dta, dtb)
    for a, b in zip(Wa, Wb):
        assert np.abs(a[inv] - b).max() <= 1e-13 * np.abs(a).max()


def test_two_cell_dam_break_by_hand():
    # Two unit cells side by side, flat bottom, at rest: h = (2, 1),
    # C = (1, 0).  Wall edges of a resting state carry only the pressure
    # g h^2 / 2; the middle edge is the acoustic problem above.
    m = O.grid_mesh(2, 1, 1.0, 1.0)
    hL, hR = 2.0, 1.0
    W0 = [np.array([hL, hR]), np.zeros(2), np.zeros(2), np.array([hL, 0.0])]
    H = np.zeros(2)
    c = math.sqrt(G * 1.5)
    # eq. (5): sum of |Gamma| ||D|| per cell; the left cell has the largest
    dt = min(2 * 0.9 / (c + 3 * math.sqrt(G * hL)), 2 * 0.9 / (c + 3 * math.sqrt(G * hR)))
    assert O.dt1(m, H, W0, G, 0.9) == pytest.approx(dt, rel=1e-15)
    W1, st = O.update1(m, H, W0, G, dt)
    assert st == O.OM_OK
    mass = c * (hL - hR) / 2
    mom = G * (hL * hL + hR * hR) / 4
    expect_h = [hL - dt * mass, hR + dt * mass]
    # left cell: middle edge pushes +mom, its west wall pushes -g hL^2/2
    expect_qx = [-dt * (mom - 0.5 * G * hL * hL), -dt * (-mom + 0.5 * G * hR * hR)]
    assert np.allclose(W1[0], expect_h, rtol=1e-14)
    assert np.allclose(W1[1], expect_qx, rtol=1e-13)
    assert np.abs(W1[2]).max() <= 1e-14
    assert np.allclose(W1[3], [hL - dt * mass, dt * mass], rtol=1e-13)


def test_depth_error_reported():
    m = O.grid_mesh(2, 1, 1.0, 1.0)
    W0 = [np.array([1.0, 1e-3]), np.array([0.0, -5.0]), np.zeros(2), np.zeros(2)]
    _, _, st, done = O.run1(m, np.zeros(2), W0, G, 0.9, 5)
    assert st in (O.OM_ERR_DEPTH, O.OM_ERR_NONFINITE)


def test_implicit_grid_equals_explicit_mesh():
    # the mesh-free Cartesian entry points list the same edges in the same
    # order as the explicit mesh, so they agree bit for bit
    d = I.make_workload("pulses8192", nx=37, ny=29)
    m = O.grid_mesh(37, 29, d["dx"], d["dy"])
    W0 = [d[k] for k in ("h", "qx", "qy", "hC")]
    Wa, dta, sa, _ = O.run1(m, d["H"], W0, G, 0.9, 20)
    Wb, dtb, sb = O.grid_run1(37, 29, d["dx"], d["dy"], d["H"], W0, G, 0.9, 20)
    assert sa == sb == O.OM_OK and np.array_equal(dta, dtb)
    for a, b in zip(Wa, Wb):
        assert np.array_equal(a, b)
    assert O.grid_dt1(37, 29, d["dx"], d["dy"], d["H"], W0, G, 0.9) == dta[0]


def test_update_at_selected_cells_equals_full_update():
    d = I.make_workload("pulses8192", nx=31, ny=17)
    m = O.grid_mesh(31, 17, d["dx"], d["dy"])
    W0 = [d[k] for k in ("h", "qx", "qy", "hC")]
    dt = O.dt1(m, d["H"], W0, G, 0.9)
    Wf, st = O.update1(m, d["H"], W0, G, dt)
    cells = np.array([0, 5, 30, 31, 263, 31 * 17 - 1])
    sel = O.update1_at(m, d["H"], W0, G, dt, cells)
    for k in range(4):
        assert np.array_equal(sel[k], Wf[k][cells])


# ---- the Harten-Hyman entropy fix (switched on with O.entropy_fix) ----------
def _transonic_dam(nx, fix, T=20.0, hl=10.0, hr=0.5):
    d = I.dam_break_1d(nx, h_left=hl, h_right=hr)
    mesh = O.grid_mesh(nx, 4, d["dx"], d["dy"])
    W = [d["h"], d["qx"], d["qy"], d["hC"]]
    t = 0.0
    with O.entropy_fix(fix):
        while t < T:
            W, dts, st, _ = O.run1(mesh, d["H"], W, G, 0.9, 1)
            assert st == O.OM_OK
            t += dts[0]
    x = (np.arange(nx) + 0.5) * d["dx"]
    ha, _ = stoker.solution(x, t, 1000.0, hl, hr, G)
    err = np.abs(W[0].reshape(4, nx)[0] - ha)
    return np.sum(err) * d["dx"], float(err[np.abs(x - 1000.0) < 60.0].max())


def test_entropy_fix_removes_the_transonic_glitch():
    # h_r / h_l = 0.05: the middle state is supercritical (u_m > c_m), so the
    # rarefaction fan contains the sonic point at the dam.  Roe's scheme alone
    # keeps an entropy-violating jump there that does not shrink under
    # refinement; with the fix the solution converges to Stoker's at first
    # order, near the dam too.
    hm, um, _ = stoker.middle_state(10.0, 0.5, G)
    assert um > math.sqrt(G * hm)
    plain = [_transonic_dam(nx, False) for nx in (200, 400, 800, 1600)]
    fixed = [_transonic_dam(nx, True) for nx in (200, 400, 800, 1600)]
    assert all(near >= 0.6 for _, near in plain), plain
    l1 = [e for e, _ in fixed]
    near = [n for _, n in fixed]
    assert all(l1[k] / l1[k + 1] >= 1.5 for k in range(3)), fixed
    assert all(near[k] / near[k + 1] >= 1.4 for k in range(3)), fixed
    assert l1[-1] < 0.6 * plain[-1][0]


def test_entropy_fix_leaves_subcritical_flow_and_rest_alone():
    # the fix acts only where |lambda_k| < delta_k, i.e. at sonic points: the
    # subcritical Stoker problem is unchanged to the last bit and water at rest
    # over hills stays at rest
    d = I.dam_break_1d(400)
    mesh = O.grid_mesh(400, 4, d["dx"], d["dy"])
    W0 = [d["h"], d["qx"], d["qy"], d["hC"]]
    Wa, dta, _, _ = O.run1(mesh, d["H"], W0, G, 0.9, 300)
    with O.entropy_fix():
        Wb, dtb, _, _ = O.run1(mesh, d["H"], W0, G, 0.9, 300)
    assert all(np.array_equal(a, b) for a, b in zip(Wa, Wb))
    assert np.array_equal(dta, dtb)
    dl = I.make_workload("hills2048", nx=48, ny=40, lake_at_rest=True)
    W0 = I.fields_of(dl)
    with O.entropy_fix():
        W, _, st = O.grid_run1(dl["nx"], dl["ny"], dl["dx"], dl["dy"], dl["H"], W0, G, 0.9, 100)
    assert st == O.OM_OK
    for a, b in zip(W, W0):
        assert np.abs(a - b).max() <= 1e-13 * max(np.abs(b).max(), 1.0)


def test_entropy_fix_conserves_mass_and_pollutant():
    # a strong radial dam break (sonic points all round the dam) with the fix
    d = I.circular_dam(64, 64, radius=12.0, h_in=10.0, h_out=0.5)
    mesh = O.grid_mesh(64, 64, 1.0, 1.0)
    W0 = I.fields_of(d)
    with O.entropy_fix():
        W, _, st, _ = O.run1(mesh, d["H"], W0, G, 0.9, 60)
    assert st == O.OM_OK
    for k in (0, 3):
        assert abs(W[k].sum() - W0[k].sum()) <= 1e-12 * W0[k].sum()
    # and it changed the flow (sonic points were crossed)
    Wp, _, _, _ = O.run1(mesh, d["H"], W0, G, 0.9, 60)
    assert np.abs(W[0] - Wp[0]).max() > 1e-3


# ---- the CFL limit ----------------------------------------------------------
@pytest.mark.parametrize("hl,hr,fix", [(2.0, 1.0, False), (10.0, 0.5, True)])
def test_stable_at_the_cfl_limit(hl, hr, fix):
    # eq. (5) allows gamma up to 1: at gamma = 1 the dam breaks stay within
    # the range of their initial depths (no over- or undershoot) and conserve
    # mass over 300 steps, before any wave reaches a wall
    d = I.dam_break_1d(400, h_left=hl, h_right=hr)
    with O.entropy_fix(fix):
        W, dts, st = O.grid_run1(400, 4, d["dx"], d["dy"], d["H"], I.fields_of(d), G, 1.0, 300)
    assert st == O.OM_OK
    h = W[0]
    assert h.min() >= hr * (1 - 1e-12) and h.max() <= hl * (1 + 1e-12)
    assert abs(h.sum() - d["h"].sum()) <= 1e-12 * d["h"].sum()
    assert dts.sum() * math.sqrt(G * hl) < 1000.0   # the fan has not reached the wall
