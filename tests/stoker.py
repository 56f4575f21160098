"""Analytic wet-bed dam-break solution of the 1D shallow-water equations
(Stoker's solution): a left rarefaction, a constant middle state and a right
shock, for water initially at rest with depth ``h_left`` for x < x0 and
``h_right`` beyond.  Used as an independent pin of the oracle.

Middle state: the rarefaction gives u_m = 2 (sqrt(g h_l) - sqrt(g h_m))
(Riemann invariant u + 2c constant across it) and the shock's
Rankine-Hugoniot conditions against the resting right state give
u_m = (h_m - h_r) sqrt(g (h_m + h_r) / (2 h_m h_r)); h_m solves the equality
of the two, by bisection on (h_r, h_l).  Shock speed s = h_m u_m / (h_m - h_r).
Inside the fan, c = (2 c_l - x/t) / 3 and u = 2 (c_l + x/t) / 3.
"""
import math

import numpy as np


def middle_state(h_left, h_right, g):
    cl = math.sqrt(g * h_left)

    def f(hm):
        u_raref = 2.0 * (cl - math.sqrt(g * hm))
        u_shock = (hm - h_right) * math.sqrt(g * (hm + h_right) / (2.0 * hm * h_right))
        return u_raref - u_shock

    lo, hi = h_right, h_left
    flo = f(lo)
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        fm = f(mid)
        if (fm > 0.0) == (flo > 0.0):
            lo, flo = mid, fm
        else:
            hi = mid
    hm = 0.5 * (lo + hi)
    um = 2.0 * (cl - math.sqrt(g * hm))
    s = hm * um / (hm - h_right)
    return hm, um, s


def solution(x, t, x0, h_left, h_right, g):
    """Depth h(x, t) and velocity u(x, t) of the dam break at x0."""
    x = np.asarray(x, dtype=np.float64)
    hm, um, s = middle_state(h_left, h_right, g)
    cl = math.sqrt(g * h_left)
    cm = math.sqrt(g * hm)
    xi = (x - x0) / t
    h = np.empty_like(x)
    u = np.empty_like(x)
    left = xi <= -cl
    fan = (xi > -cl) & (xi <= um - cm)
    mid = (xi > um - cm) & (xi <= s)
    right = xi > s
    h[left], u[left] = h_left, 0.0
    c = (2.0 * cl - xi[fan]) / 3.0
    h[fan] = c * c / g
    u[fan] = 2.0 * (cl + xi[fan]) / 3.0
    h[mid], u[mid] = hm, um
    h[right], u[right] = h_right, 0.0
    return h, u
