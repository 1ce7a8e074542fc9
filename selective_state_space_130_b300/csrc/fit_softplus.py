"""Coefficients of the polynomial behind softplus_fast (ss_device.cuh).

softplus(x) = max(x, 0) + log1p(v), v = e^-|x| in (0, 1], and log1p(v) = v q(v)
with q(v) = log1p(v) / v, a smooth function on [0, 1] (q(0) = 1, q(1) = ln 2).
q is fitted by a polynomial of degree 7 in the relative-error sense: weighted
least squares on Chebyshev nodes, with the weights raised where the error is
largest (a few passes of a Lawson-style reweighting). The coefficients are then
rounded to fp32 and the polynomial is evaluated by Horner in fp32 on a fine
grid to give the bound quoted beside the constants.

    python fit_softplus.py          # prints the coefficients and the bound
"""

import numpy as np
from numpy.polynomial import polynomial as P

DEGREE = 7


def q(v):
    v = np.asarray(v, dtype=np.float64)
    safe = np.where(v == 0, 1.0, v)
    return np.where(v == 0, 1.0, np.log1p(safe) / safe)


def fit(degree=DEGREE, n=4000, passes=30):
    x = 0.5 + 0.5 * np.cos(np.pi * (np.arange(n) + 0.5) / n)
    y = q(x)
    w = 1.0 / np.abs(y)
    for _ in range(passes):
        c = P.polyfit(x, y, degree, w=w)
        err = (P.polyval(x, c) - y) / y
        w = w * (1.0 + 5.0 * np.abs(err) / np.abs(err).max())
    return c.astype(np.float32)


def horner_f32(c, v):
    v = v.astype(np.float32)
    acc = np.full_like(v, c[-1])
    for k in range(len(c) - 2, -1, -1):
        acc = (acc * v + c[k]).astype(np.float32)
    return acc


def max_rel_error(c, npts=200001):
    v = np.linspace(0.0, 1.0, npts)
    return float(np.max(np.abs((horner_f32(c, v).astype(np.float64) - q(v)) / q(v))))


if __name__ == "__main__":
    c = fit()
    for k, ck in enumerate(c):
        print(f"c{k} = {float(ck)!r}")
    print(f"max relative error of q in fp32 Horner: {max_rel_error(c):.3e}")
