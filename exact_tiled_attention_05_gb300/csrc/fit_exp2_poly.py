"""Fits the cubic used by the forward kernel's software exp2.

2^x is split as 2^x = 2^j * 2^f with j = round(x) and f = x - j in [-1/2, 1/2]
(Cody-Waite style range reduction); 2^j is built by adding j to the float's
exponent bits, and 2^f comes from a degree-3 polynomial.  This script fits that
polynomial by weighted least squares on Chebyshev nodes of [-1/2, 1/2], weights
1/2^f so the fit minimises relative error, with the constant term pinned to 1
(so 2^0 is exact).  It prints the coefficients and the worst relative error in
fp64 and after float32 Horner evaluation.

    python fit_exp2_poly.py
"""
import numpy as np


def fit(degree=3, nodes=4001):
    k = np.arange(nodes)
    f = 0.5 * np.cos(np.pi * (k + 0.5) / nodes)  # Chebyshev nodes on [-1/2, 1/2]
    y = np.exp2(f)
    w = 1.0 / y
    # p(f) = 1 + c1 f + c2 f^2 + c3 f^3  ->  least squares for c1..c3 on (y - 1)
    A = np.stack([f ** i for i in range(1, degree + 1)], axis=1) * w[:, None]
    b = (y - 1.0) * w
    c, *_ = np.linalg.lstsq(A, b, rcond=None)
    return np.concatenate([[1.0], c])


def horner32(coef, f):
    f = np.float32(f)
    p = np.float32(coef[-1])
    for c in coef[-2::-1]:
        p = np.float32(p * f + np.float32(c))
    return p


def max_rel_error(coef):
    f = np.linspace(-0.5, 0.5, 200001)
    p64 = sum(c * f ** i for i, c in enumerate(coef))
    e64 = np.max(np.abs(p64 / np.exp2(f) - 1.0))
    c32 = [np.float32(c) for c in coef]
    p32 = np.array([horner32(c32, x) for x in f[::50]], dtype=np.float64)
    e32 = np.max(np.abs(p32 / np.exp2(f[::50]) - 1.0))
    return e64, e32


if __name__ == "__main__":
    coef = fit()
    e64, e32 = max_rel_error(coef)
    for i, c in enumerate(coef):
        print(f"c{i} = {np.float32(c)!r}  ({c:.17g})")
    print(f"max relative error: {e64:.3e} (fp64), {e32:.3e} (float32 Horner)")
