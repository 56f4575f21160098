"""Analytic dam break over a dry, flat, frictionless bed (Ritter's solution):
water at rest with depth h0 for x < x0 and no water beyond.  A single
rarefaction joins the still water to the dry bed; with c0 = sqrt(g h0) and
xi = (x - x0) / t the Riemann invariant u + 2c = 2 c0 carried from the still
water and the fan's characteristics dx/dt = u - c = xi give
    xi <= -c0:          h = h0, u = 0
    -c0 < xi < 2 c0:    h = (2 c0 - xi)^2 / (9 g), u = 2 (c0 + xi) / 3
    xi >= 2 c0:         h = 0, u = 0 (the front moves at 2 c0).
The fan is transonic: u = c at xi = 0, where the dam stood.  Used as an
independent pin of the oracle's wet/dry treatment.
"""
import math

import numpy as np


def solution(x, t, x0, h0, g):
    """Depth h(x, t) and velocity u(x, t)."""
    c0 = math.sqrt(g * h0)
    xi = (np.asarray(x, dtype=np.float64) - x0) / t
    fan = (xi > -c0) & (xi < 2.0 * c0)
    h = np.where(xi <= -c0, h0, 0.0)
    u = np.zeros_like(h)
    h[fan] = (2.0 * c0 - xi[fan]) ** 2 / (9.0 * g)
    u[fan] = 2.0 * (c0 + xi[fan]) / 3.0
    return h, u
