"""Seeded synthetic inputs for the shallow-water workloads.

This module only draws and lays out initial data (bathymetry ``H``, depth
``h``, discharge ``qx, qy`` and pollutant mass ``hC``); it holds none of the
numerical scheme's arithmetic, so the CUDA path and the CPU oracle can both be
fed from it without sharing any code of the method.

Conventions (An MPI-CUDA implementation of an improved Roe method for
two-layer shallow water systems, Sec. 2.1, eq. (1)): ``H`` is the depth of the
bottom measured downward from a fixed reference level, so the bottom elevation
is ``z_b = -H`` and the free surface is ``h - H``.  Cell ``(i, j)`` of an
``nx x ny`` grid is stored at flat index ``j * nx + i`` with its centre at
``((i + 1/2) dx, (j + 1/2) dy)``.

Workloads (the pages give no datasets; these stand in for their "internal dam
break" and "realistic pollutant problem"):

* ``dam128``   128 x 128, dx = 1 m, flat bottom, circular dam break of radius
  20 m about (64, 64): h = 2 inside, 1 outside, q = 0, C = 1 inside, 0 outside.
* ``hills2048`` 2048 x 2048, dx = 10 m, 8 Gaussian hills under a 5 m surface,
  3 surface bumps of 0.5 m, q = 0, C uniform per 16 x 16 block.
* ``pulses8192`` 8192 x 8192, dx = 10 m, 128 hills (8 per 2048^2 of area),
  16 surface pulses of 0.5 m, random velocities |u| <= 0.1 m/s, C per block.

Every random draw comes from ``numpy.random.Generator(PCG64(seed))`` in the
order documented in each function, so a workload is a pure function of its
name, size and seed.
"""
from __future__ import annotations

import numpy as np

G_DEFAULT = 9.81
CFL_DEFAULT = 0.9

# workload name -> (nx, ny, dx, default steps, seed, default precision)
WORKLOADS = {
    "dam128": dict(nx=128, ny=128, dx=1.0, steps=100, seed=1001, precision=64),
    "hills2048": dict(nx=2048, ny=2048, dx=10.0, steps=1000, seed=1002, precision=32),
    "pulses8192": dict(nx=8192, ny=8192, dx=10.0, steps=200, seed=1003, precision=32),
    "interface2048": dict(nx=2048, ny=2048, dx=10.0, steps=500, seed=1004, precision=64),
    "tri1024": dict(nx=1024, ny=1024, dx=1.0, steps=500, seed=1005, precision=32),
    "tri1024_1l": dict(nx=1024, ny=1024, dx=1.0, steps=500, seed=1006, precision=32),
    "flood2048": dict(nx=2048, ny=2048, dx=10.0, steps=500, seed=1007, precision=32),
}
TWO_LAYER = ("interface2048", "tri1024")


def _gaussian_sum(nx, ny, dx, dy, amp, sigma, cx, cy, cutoff=8.0):
    """Sum of isotropic Gaussians ``amp * exp(-r^2 / (2 sigma^2))`` sampled at
    cell centres.  Each Gaussian is evaluated on the window within
    ``cutoff * sigma`` of its centre (exp(-32) ~ 1e-14 relative is dropped)
    as an outer product of its separable x and y factors."""
    out = np.zeros((ny, nx), dtype=np.float64)
    xc = (np.arange(nx) + 0.5) * dx
    yc = (np.arange(ny) + 0.5) * dy
    for a, s, x0, y0 in zip(amp, sigma, cx, cy):
        i0 = max(int(np.floor((x0 - cutoff * s) / dx)), 0)
        i1 = min(int(np.ceil((x0 + cutoff * s) / dx)) + 1, nx)
        j0 = max(int(np.floor((y0 - cutoff * s) / dy)), 0)
        j1 = min(int(np.ceil((y0 + cutoff * s) / dy)) + 1, ny)
        if i0 >= i1 or j0 >= j1:
            continue
        gx = np.exp(-((xc[i0:i1] - x0) ** 2) / (2.0 * s * s))
        gy = np.exp(-((yc[j0:j1] - y0) ** 2) / (2.0 * s * s))
        out[j0:j1, i0:i1] += a * np.outer(gy, gx)
    return out


def _hills(rng, n, lx, ly, amp_lo, amp_hi):
    """Draw ``n`` Gaussian features: amplitudes U[amp_lo, amp_hi], widths
    sigma U[50, 300] m, centres U[0, lx] x U[0, ly]; drawn in that order."""
    amp = rng.uniform(amp_lo, amp_hi, n)
    sigma = rng.uniform(50.0, 300.0, n)
    cx = rng.uniform(0.0, lx, n)
    cy = rng.uniform(0.0, ly, n)
    return amp, sigma, cx, cy


def _block_concentration(rng, nx, ny, block=16):
    """C ~ U[0, 1], constant on each ``block x block`` tile of cells."""
    bx = (nx + block - 1) // block
    by = (ny + block - 1) // block
    cb = rng.uniform(0.0, 1.0, (by, bx))
    return np.repeat(np.repeat(cb, block, axis=0), block, axis=1)[:ny, :nx]


def _as_fields(H, h, qx, qy, hC, **meta):
    d = dict(meta)
    d["H"] = np.ascontiguousarray(H, dtype=np.float64).reshape(-1)
    d["h"] = np.ascontiguousarray(h, dtype=np.float64).reshape(-1)
    d["qx"] = np.ascontiguousarray(qx, dtype=np.float64).reshape(-1)
    d["qy"] = np.ascontiguousarray(qy, dtype=np.float64).reshape(-1)
    d["hC"] = np.ascontiguousarray(hC, dtype=np.float64).reshape(-1)
    return d


def circular_dam(nx=128, ny=128, dx=1.0, dy=None, radius=20.0, centre=None,
                 h_in=2.0, h_out=1.0, c_in=1.0, c_out=0.0):
    """Circular dam break on a flat bottom (H = 0), water at rest."""
    dy = dx if dy is None else dy
    if centre is None:
        centre = (0.5 * nx * dx, 0.5 * ny * dy)
    x = (np.arange(nx) + 0.5) * dx
    y = (np.arange(ny) + 0.5) * dy
    X, Y = np.meshgrid(x, y)
    inside = (X - centre[0]) ** 2 + (Y - centre[1]) ** 2 < radius * radius
    h = np.where(inside, h_in, h_out)
    C = np.where(inside, c_in, c_out)
    z = np.zeros_like(h)
    return _as_fields(z, h, z, z, h * C, nx=nx, ny=ny, dx=dx, dy=dy)


def hills(nx, ny, dx=10.0, dy=None, seed=1002, n_hills=8, n_bumps=3,
          eta0=5.0, bump_amp=0.5, umax=0.0, lake_at_rest=False):
    """Gaussian-hill bathymetry under a flat surface ``eta0`` plus Gaussian
    surface bumps; pollutant concentration uniform per 16 x 16 block.

    Draw order: hills (amp U[0.2, 0.8], sigma, cx, cy), bumps (amp fixed at
    ``bump_amp``; sigma, cx, cy drawn with amplitudes drawn and discarded so the
    stream layout matches the hills), block concentrations, then (only when
    ``umax > 0``) per-cell speed U[0, umax] and direction U[0, 2 pi) as two
    full arrays.  ``lake_at_rest`` drops the bumps and velocities (surface
    exactly ``eta0``) while keeping the same draws.
    """
    dy = dx if dy is None else dy
    rng = np.random.Generator(np.random.PCG64(seed))
    lx, ly = nx * dx, ny * dy
    a, s, cx, cy = _hills(rng, n_hills, lx, ly, 0.2, 0.8)
    zb = _gaussian_sum(nx, ny, dx, dy, a, s, cx, cy)
    _, bs, bx, by = _hills(rng, n_bumps, lx, ly, 0.0, 1.0)
    bumps = _gaussian_sum(nx, ny, dx, dy, np.full(n_bumps, bump_amp), bs, bx, by)
    C = _block_concentration(rng, nx, ny)
    if umax > 0.0:
        speed = rng.uniform(0.0, umax, (ny, nx))
        theta = rng.uniform(0.0, 2.0 * np.pi, (ny, nx))
    H = -zb
    if lake_at_rest:
        h = eta0 + H
        qx = np.zeros_like(h)
        qy = np.zeros_like(h)
    else:
        h = eta0 + bumps + H
        if umax > 0.0:
            qx = h * speed * np.cos(theta)
            qy = h * speed * np.sin(theta)
        else:
            qx = np.zeros_like(h)
            qy = np.zeros_like(h)
    if np.min(h) < 0.5:
        raise ValueError("generator produced a depth below 0.5 m")
    return _as_fields(H, h, qx, qy, h * C, nx=nx, ny=ny, dx=dx, dy=dy)


def dam_break_1d(nx, ny=4, length=2000.0, x_dam=1000.0, h_left=2.0, h_right=1.0):
    """Wet-bed dam break along x on a flat bottom: h = h_left for x < x_dam,
    h_right beyond, water at rest, C = 1 on the left and 0 on the right;
    square cells (dy = dx)."""
    dx = length / nx
    x = (np.arange(nx) + 0.5) * dx
    h1 = np.where(x < x_dam, h_left, h_right)
    h = np.tile(h1, (ny, 1))
    C = np.tile(np.where(x < x_dam, 1.0, 0.0), (ny, 1))
    z = np.zeros_like(h)
    return _as_fields(z, h, z, z, h * C, nx=nx, ny=ny, dx=dx, dy=dx)


def dry_dam_1d(nx, ny=4, length=2000.0, x_dam=1000.0, h0=2.0):
    """Dam break over a dry, flat bed along x (Ritter's problem): h = h0 for
    x < x_dam and 0 beyond, water at rest, C = 1 in the water; square cells.
    For runs with the wet/dry treatment."""
    dx = length / nx
    x = (np.arange(nx) + 0.5) * dx
    h1 = np.where(x < x_dam, h0, 0.0)
    h = np.tile(h1, (ny, 1))
    z = np.zeros_like(h)
    return _as_fields(z, h, z, z, h.copy(), nx=nx, ny=ny, dx=dx, dy=dx)


def emerged_hills(nx, ny, dx=10.0, seed=1007, n_hills=8, eta=None, column=None, slope=0.0):
    """Gaussian hills (amplitude U[0.5, 2.5] m, sigma U[50, 300] m, centres
    U[0, L]^2) that pierce a lake at rest, for runs with the wet/dry
    treatment.  The surface ``eta`` (default: 0.3 m below the highest bed
    point) leaves the hill tops dry: h = max(0, eta - z_b) exactly, q = 0,
    C per 16 x 16 block.  ``slope`` tilts the bed, z_b += slope (x - L/2),
    so that one side of the domain is dry land.  ``column = (cx, cy,
    radius, rise)`` raises the surface by ``rise`` inside the disc (a dam
    break that floods dry land).  Draw order: hills (amp, sigma, cx, cy),
    then block concentrations."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lx, ly = nx * dx, ny * dx
    a, s, cx, cy = _hills(rng, n_hills, lx, ly, 0.5, 2.5)
    zb = _gaussian_sum(nx, ny, dx, dx, a, s, cx, cy)
    if slope:
        zb = zb + slope * ((np.arange(nx) + 0.5) * dx - 0.5 * lx)[None, :]
    C = _block_concentration(rng, nx, ny)
    level = zb.max() - 0.3 if eta is None else float(eta)
    surf = np.full_like(zb, level)
    if column is not None:
        x0, y0, rad, rise = column
        xc = (np.arange(nx) + 0.5) * dx
        yc = (np.arange(ny) + 0.5) * dx
        X, Y = np.meshgrid(xc, yc)
        surf = np.where(np.hypot(X - x0, Y - y0) < rad, level + rise, level)
    h = np.maximum(0.0, surf - zb)
    z = np.zeros_like(h)
    return _as_fields(-zb, h, z, z, h * C, nx=nx, ny=ny, dx=dx, dy=dx)


def interface_dam(nx, ny, dx=10.0, depth=10.0, h_left=6.0, h_right=4.0, r=0.98):
    """Two-layer interface dam break on a flat bottom ``depth`` deep: upper
    layer h1 = h_left for x < L/2 and h_right beyond, lower layer
    h2 = depth - h1, both at rest."""
    x = (np.arange(nx) + 0.5) * dx
    h1 = np.tile(np.where(x < 0.5 * nx * dx, h_left, h_right), (ny, 1))
    H = np.full((ny, nx), float(depth))
    z = np.zeros((ny, nx))
    d = dict(nx=nx, ny=ny, dx=dx, dy=dx, r=r, n_layers=2)
    for k, v in (("H", H), ("h1", h1), ("q1x", z), ("q1y", z), ("h2", H - h1), ("q2x", z),
                 ("q2y", z)):
        d[k] = np.ascontiguousarray(v, dtype=np.float64).reshape(-1)
    return d


def two_layer_hills(nx, ny, dx=10.0, seed=1005, interface_depth=3.0, umax=0.0,
                    bump=0.0, r=0.95):
    """Two layers over the Gaussian-hill bottom (pushed 10 m down): surface at
    +5 m, flat interface ``interface_depth`` below it, an optional Gaussian
    bump of the interface at the domain centre (amplitude ``bump``) and random
    velocities |u| <= umax in both layers (drawn speed then direction, upper
    layer first, after the hills)."""
    rng = np.random.default_rng(seed)
    lx, ly = nx * dx, ny * dx
    a, sg, cx, cy = _hills(rng, 8, lx, ly, 0.2, 0.8)
    H = 10.0 - _gaussian_sum(nx, ny, dx, dx, a, sg, cx, cy)
    x = (np.arange(nx) + 0.5) * dx
    y = (np.arange(ny) + 0.5) * dx
    X, Y = np.meshgrid(x, y)
    h1 = interface_depth + bump * np.exp(-((X - lx / 2) ** 2 + (Y - ly / 2) ** 2) / (0.1 * lx) ** 2)
    h2 = H + 5.0 - h1
    d = dict(nx=nx, ny=ny, dx=dx, dy=dx, r=r, n_layers=2)
    q = []
    for hk in (h1, h2):
        if umax > 0.0:
            sp = rng.uniform(0.0, umax, (ny, nx))
            th = rng.uniform(0.0, 2.0 * np.pi, (ny, nx))
            q.append((hk * sp * np.cos(th), hk * sp * np.sin(th)))
        else:
            q.append((np.zeros_like(hk), np.zeros_like(hk)))
    for k, v in (("H", H), ("h1", h1), ("q1x", q[0][0]), ("q1y", q[0][1]), ("h2", h2),
                 ("q2x", q[1][0]), ("q2y", q[1][1])):
        d[k] = np.ascontiguousarray(v, dtype=np.float64).reshape(-1)
    return d


TWO_LAYER_FIELDS = ("h1", "q1x", "q1y", "h2", "q2x", "q2y")


def square_tri_mesh(n, m=None, side=1.0, jitter=0.2, seed=1005, shuffle=True):
    """Triangle mesh of n x m squares of size ``side``: (n+1)(m+1) vertices,
    vertex (i, j) at index j*(n+1) + i; square (i, j) split along its lower-left
    to upper-right diagonal into the counter-clockwise triangles (a, b, c) and
    (a, c, d) with a = (i, j), b = (i+1, j), c = (i+1, j+1), d = (i, j+1).
    Interior vertices move by U[-jitter, jitter] * side in x then in y (one
    array of draws each); with ``shuffle`` the cells are then reordered by a
    seeded permutation (drawn after the jitter).  Returns (xy, tri) with xy of
    shape (nv, 2) and tri of shape (nc, 3)."""
    m = n if m is None else m
    rng = np.random.default_rng(seed)
    i, j = np.meshgrid(np.arange(n + 1), np.arange(m + 1))
    x = i.astype(np.float64) * side
    y = j.astype(np.float64) * side
    inner = (i > 0) & (i < n) & (j > 0) & (j < m)
    jx = rng.uniform(-jitter, jitter, x.shape) * side
    jy = rng.uniform(-jitter, jitter, y.shape) * side
    x = np.where(inner, x + jx, x)
    y = np.where(inner, y + jy, y)
    xy = np.stack([x.reshape(-1), y.reshape(-1)], axis=1)
    si, sj = np.meshgrid(np.arange(n), np.arange(m))
    a = (sj * (n + 1) + si).reshape(-1)
    b, c, d = a + 1, a + n + 2, a + n + 1
    tri = np.empty((2 * n * m, 3), dtype=np.int32)
    tri[0::2] = np.stack([a, b, c], axis=1)
    tri[1::2] = np.stack([a, c, d], axis=1)
    if shuffle:
        tri = tri[rng.permutation(tri.shape[0])]
    return xy, np.ascontiguousarray(tri)


def tri_centroids(xy, tri):
    """Vertex mean of each triangle (where the initial state is sampled)."""
    return xy[tri].mean(axis=1)


def tri_workload(n, seed=1005, jitter=0.2, r=0.98, n_hills=8, bump=0.5, sigma_scale=None):
    """The two-layer triangle-mesh workload on n x n unit squares (see the
    module docstring); the state is sampled at cell centroids.  Draw order:
    the mesh (jitter, permutation), then the hills (amplitude, width, centre)
    and the interface bump (width, centre).  Widths are U[50, 300] times
    ``sigma_scale``, by default n / 20480 (the 2048 x 10 m domain of the hills
    workload mapped onto the n x n square: 2.5 to 15 squares at n = 1024);
    small test meshes pass a larger scale to keep their features resolved."""
    xy, tri = square_tri_mesh(n, side=1.0, jitter=jitter, seed=seed)
    rng = np.random.default_rng(seed + 7919)
    L = float(n)
    scale = n / 20480.0 if sigma_scale is None else float(sigma_scale)
    amp = rng.uniform(0.2, 0.8, n_hills)
    sig = rng.uniform(50.0, 300.0, n_hills) * scale
    cx = rng.uniform(0.0, L, n_hills)
    cy = rng.uniform(0.0, L, n_hills)
    bs = rng.uniform(50.0, 300.0) * scale
    bx, by = rng.uniform(0.0, L, 2)
    cxy = tri_centroids(xy, tri)
    zb = np.zeros(tri.shape[0])
    for a_, s_, x0, y0 in zip(amp, sig, cx, cy):
        zb += a_ * np.exp(-((cxy[:, 0] - x0) ** 2 + (cxy[:, 1] - y0) ** 2) / (2 * s_ * s_))
    H = 10.0 - zb
    h1 = 5.0 + bump * np.exp(-((cxy[:, 0] - bx) ** 2 + (cxy[:, 1] - by) ** 2) / (2 * bs * bs))
    z = np.zeros_like(H)
    d = dict(xy=xy, tri=tri, n_cells=tri.shape[0], r=r, n_layers=2, mesh=True)
    for k, v in (("H", H), ("h1", h1), ("q1x", z), ("q1y", z), ("h2", H - h1), ("q2x", z),
                 ("q2y", z)):
        d[k] = np.ascontiguousarray(v, dtype=np.float64)
    return d


def tri_workload1(n, m=None, seed=1006, jitter=0.2, umax=0.1, n_hills=6, n_pulses=4):
    """A one-layer triangle-mesh workload with a pollutant on n x m unit
    squares: Gaussian hills under a 2 m deep surface (H = 3 - z_b, surface at
    h - H = 2), Gaussian surface pulses of 0.5 m, velocities U[-umax, umax]
    per component, C uniform in [0, 1] per block of 4 x 4 squares.  Draw
    order: the mesh (jitter, permutation), hills (amplitude, width, centre x,
    centre y), pulses (width, centre x, centre y), velocities (x, then y),
    block concentrations."""
    m = n if m is None else m
    xy, tri = square_tri_mesh(n, m, side=1.0, jitter=jitter, seed=seed)
    rng = np.random.default_rng(seed + 7919)
    cxy = tri_centroids(xy, tri)
    size = float(min(n, m))
    zb = np.zeros(tri.shape[0])
    amp = rng.uniform(0.2, 0.8, n_hills)
    sig = rng.uniform(0.05, 0.2, n_hills) * size
    hx = rng.uniform(0.0, n, n_hills)
    hy = rng.uniform(0.0, m, n_hills)
    for a_, s_, x0, y0 in zip(amp, sig, hx, hy):
        zb += a_ * np.exp(-((cxy[:, 0] - x0) ** 2 + (cxy[:, 1] - y0) ** 2) / (2 * s_ * s_))
    eta = np.full(tri.shape[0], 2.0)
    ps = rng.uniform(0.05, 0.15, n_pulses) * size
    px = rng.uniform(0.0, n, n_pulses)
    py = rng.uniform(0.0, m, n_pulses)
    for s_, x0, y0 in zip(ps, px, py):
        eta += 0.5 * np.exp(-((cxy[:, 0] - x0) ** 2 + (cxy[:, 1] - y0) ** 2) / (2 * s_ * s_))
    H = 3.0 - zb
    h = H + eta
    ux = rng.uniform(-umax, umax, h.size)
    uy = rng.uniform(-umax, umax, h.size)
    nbx, nby = (n + 3) // 4, (m + 3) // 4
    table = rng.uniform(0.0, 1.0, (nby, nbx))
    bx = np.minimum((cxy[:, 0] // 4).astype(np.int64), nbx - 1)
    by = np.minimum((cxy[:, 1] // 4).astype(np.int64), nby - 1)
    C = table[by, bx]
    d = dict(xy=xy, tri=tri, n_cells=tri.shape[0], n_layers=1, mesh=True, g=G_DEFAULT,
             cfl=CFL_DEFAULT)
    for k, v in (("H", H), ("h", h), ("qx", h * ux), ("qy", h * uy), ("hC", h * C)):
        d[k] = np.ascontiguousarray(v, dtype=np.float64)
    return d


def fields2_of(d, dtype=np.float64):
    """The six fields of a two-layer workload dict, cast."""
    return [np.ascontiguousarray(d[k], dtype=dtype) for k in TWO_LAYER_FIELDS]


def make_workload(name, nx=None, ny=None, lake_at_rest=False):
    """Initial data of a named workload, optionally at a reduced size.

    Returns a dict with ``nx, ny, dx, dy, g, cfl, steps, precision`` and the
    fp64 flat arrays ``H, h, qx, qy, hC`` (length ``nx * ny``).  Reduced sizes
    keep the recipe and the grid spacing; the hill count of ``pulses8192``
    scales with the domain area (8 per 2048 x 2048 cells, at least 8).
    """
    if name not in WORKLOADS:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}")
    w = WORKLOADS[name]
    nx = w["nx"] if nx is None else int(nx)
    ny = w["ny"] if ny is None else int(ny)
    dx = w["dx"]
    if name == "tri1024":
        d = tri_workload(nx)
        d.update(g=G_DEFAULT, cfl=CFL_DEFAULT, steps=w["steps"], precision=w["precision"],
                 name=name)
        return d
    if name == "flood2048":
        # wet/dry fronts: a bed rising 4 m across the domain with 64 hills
        # (16 per 1024^2 cells), a lake at rest at level 0 (about half the
        # domain dry), a disc of radius L/10 raised by 2 m at the centre;
        # cells below 1 cm are dry (thinner films run up the slope at
        # unphysical speeds)
        lx = nx * dx
        n_h = max(8, int(round(64 * nx * ny / (2048 * 2048))))
        d = emerged_hills(nx, ny, dx, seed=w["seed"], n_hills=n_h, eta=0.0,
                          column=(0.5 * lx, 0.5 * ny * dx, 0.1 * lx, 2.0), slope=4.0 / lx)
        d.update(g=G_DEFAULT, cfl=CFL_DEFAULT, steps=w["steps"], precision=w["precision"],
                 name=name, wet_dry=1, h_dry=1e-2, entropy_fix=1)
        return d
    if name == "tri1024_1l":
        d = tri_workload1(nx, ny, seed=w["seed"])
        d.update(steps=w["steps"], precision=w["precision"], name=name)
        return d
    if name == "interface2048":
        d = interface_dam(nx, ny, dx)
        d.update(g=G_DEFAULT, cfl=CFL_DEFAULT, steps=w["steps"], precision=w["precision"],
                 name=name)
        return d
    if name == "dam128":
        d = circular_dam(nx, ny, dx, radius=20.0 * min(nx, ny) / 128.0)
    elif name == "hills2048":
        d = hills(nx, ny, dx, seed=w["seed"], n_hills=8, n_bumps=3,
                  lake_at_rest=lake_at_rest)
    else:
        n_h = max(8, int(round(8 * nx * ny / (2048 * 2048))))
        d = hills(nx, ny, dx, seed=w["seed"], n_hills=n_h, n_bumps=16,
                  umax=0.1, lake_at_rest=lake_at_rest)
    d.update(g=G_DEFAULT, cfl=CFL_DEFAULT, steps=w["steps"],
             precision=w["precision"], name=name)
    return d


def fields_of(d, dtype=np.float64):
    """The four conserved fields (h, qx, qy, hC) of a workload dict, cast."""
    return [np.ascontiguousarray(d[k], dtype=dtype) for k in ("h", "qx", "qy", "hC")]


def rounded(d, dtype):
    """A copy of a workload whose fields and bathymetry are rounded to
    ``dtype`` and widened back to fp64, so a reduced-precision run and an fp64
    run start from the same values."""
    out = dict(d)
    for k in ("H", "h", "qx", "qy", "hC") + TWO_LAYER_FIELDS:
        if k in d:
            out[k] = d[k].astype(dtype).astype(np.float64)
    return out
