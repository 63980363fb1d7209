#!/usr/bin/env python
"""Coefficients of the normal-tail approximation in device_common.cuh (run once; prints them).

The kernels need Phi(-|h|) = erfc(z) / 2, z = |h| / sqrt 2, with a small RELATIVE error for
every h (the GeLU of a large negative pre-activation is h * Phi(h), a tiny number whose
relative accuracy is what a tail-only comparison sees). They use the form of Abramowitz &
Stegun, Handbook of Mathematical Functions, 7.1.26 --

    erfc(z) = t * Q(t) * exp(-z^2),   t = 1 / (1 + p z),

one reciprocal and one exponential (shared with the normal density of GeLU') -- but with Q a
polynomial fitted here, instead of 7.1.26's degree-4 coefficients, which are
fitted for absolute error and are 38 % off in relative terms as z grows (t Q(t) must tend to
p t / sqrt(pi), the asymptote of the scaled function erfcx(z) = exp(z^2) erfc(z) =
1 / (sqrt(pi) z) + ...). Q(t) = erfcx(z(t)) / t is smooth on t in (0, 1], so a polynomial in t
fits it in relative terms on all of z >= 0.

Fit: weighted least squares on Chebyshev nodes in t (z in [0, 40]), reweighted by the
residual (Lawson's iteration) towards the minimax relative error. Reference: scipy's erfcx
in fp64.
"""
import numpy as np
from scipy.special import erfcx

P = 0.5
# degree 8 for the fp32 paths (relative error ~2e-7 of erfcx, below fp32's tolerance of 1e-5
# with room for the exponential's rounding); degree 5 for the bf16 epilogues, whose outputs
# are rounded to bf16 (2^-9 relative): ~5e-5 there.
DEGREES = (8, 5)
DEGREE = 8
Z_MAX = 40.0


def fit(p=P, deg=DEGREE, zmax=Z_MAX, nodes=4000, iters=30):
    tmin = 1.0 / (1.0 + p * zmax)
    k = np.arange(nodes)
    t = (tmin + 1) / 2 + (1 - tmin) / 2 * np.cos(np.pi * (k + 0.5) / nodes)
    z = (1 / t - 1) / p
    y = erfcx(z) / t
    V = np.vander(t, deg + 1, increasing=True)
    w = np.ones_like(t)
    c = None
    for _ in range(iters):
        W = w / np.abs(y)
        c, *_ = np.linalg.lstsq(V * W[:, None], y * W, rcond=None)
        r = np.abs(V @ c - y) / np.abs(y)
        w = w * r
        w = np.sqrt(w / w.sum() * len(w))
    return c


def max_rel_error(c, p=P):
    z = np.linspace(0.0, 30.0, 300001)
    t = 1 / (1 + p * z)
    return float(np.max(np.abs(t * np.polyval(c[::-1], t) - erfcx(z)) / erfcx(z)))


if __name__ == "__main__":
    for deg in DEGREES:
        c = fit(deg=deg)
        print(f"p = {P}, degree {deg}: max relative error of t Q(t) vs erfcx on [0, 30]: "
              f"{max_rel_error(c):.2e}")
        for i, v in enumerate(c):
            print(f"  q{i} = {v:.9e}")
