"""Coefficients of the cubic used for 2^f, f in [-1/2, 1/2], in da_common.cuh.

Method: Lawson's iteratively reweighted least squares (the L-infinity limit of
weighted least squares, C. L. Lawson 1961) on Chebyshev-distributed points,
minimising the maximum *relative* error of c0 + c1 f + c2 f^2 + c3 f^3
against 2^f.  The kernels combine it with the classic range reduction
x = n + f, n = rint(x) (Cody and Waite, "Software Manual for the Elementary
Functions", 1980) and scale by 2^n through the exponent field.

Run:  python gen_exp2_poly.py      (prints the coefficients and the error bound)
"""
import numpy as np


def fit(degree: int = 3, iters: int = 200):
    f = np.cos(np.linspace(0.0, np.pi, 4001)) * 0.5
    y = 2.0 ** f
    V = np.vander(f, degree + 1, increasing=True)
    w = np.ones_like(f)
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(V / y[:, None] * sw[:, None], sw, rcond=None)
        e = np.abs(V @ c / y - 1.0)
        w = w * (e + 1e-30)
        w /= w.sum()
    return c


def max_rel_error(c) -> float:
    g = np.linspace(-0.5, 0.5, 400001)
    return float(np.abs(np.polyval(c[::-1], g) / 2.0 ** g - 1.0).max())


if __name__ == "__main__":
    c = fit()
    for i, v in enumerate(c):
        print(f"c{i} = {np.float32(v)!r}")
    print(f"max relative error on [-1/2, 1/2]: {max_rel_error(c):.3e}")
