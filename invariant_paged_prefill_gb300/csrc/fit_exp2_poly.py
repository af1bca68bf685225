"""Coefficients of the polynomial that approximates 2^f on [-1/2, 1/2].

Used by the FMA-pipe exp2 in bip_numerics.cuh (range reduction x = n + f with
n the nearest integer, 2^x = 2^n * p(f)).  Fit: relative-error weighted least
squares in float64 at 2000 Chebyshev nodes, then rounded to float32.  Prints
the coefficients (constant term first) and the worst relative error of the
float32 Horner evaluation on a dense grid.

    python fit_exp2_poly.py [degree]
"""

import sys

import numpy as np


def fit(degree: int):
    k = np.arange(2000)
    f = 0.5 * np.cos(np.pi * (k + 0.5) / 2000)           # Chebyshev nodes on [-1/2, 1/2]
    y = np.exp2(f)
    A = np.vander(f, degree + 1, increasing=True) / y[:, None]   # relative error weighting
    c, *_ = np.linalg.lstsq(A, np.ones_like(f), rcond=None)
    c32 = c.astype(np.float32)
    g = np.linspace(-0.5, 0.5, 200001).astype(np.float32)
    p = np.full_like(g, c32[-1])
    for ci in c32[-2::-1]:
        p = (p * g + ci).astype(np.float32)               # Horner in float32
    err = np.max(np.abs(p.astype(np.float64) / np.exp2(g.astype(np.float64)) - 1))
    return c32, err


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 4
    c, err = fit(deg)
    print("coefficients:", ", ".join(f"{float(x)!r}f" for x in c))
    print(f"max relative error of the float32 evaluation: {err:.3e}")
