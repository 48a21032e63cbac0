"""Derives the coefficients of the polynomial exp2 used by the kernels.

2^x is split as 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2];
2^f is replaced by the degree-3 polynomial p(f) that minimises the maximum
relative error on that interval (Remez exchange on the weighted error
(p(f) - 2^f) / 2^f). Run as a script to print the coefficients and the error
bound; the kernels' constants are these values rounded to float32.

    python -m exact_attention_97_gb300.exp2_poly_fit
"""
from __future__ import annotations

import numpy as np


def remez_exp2(degree: int = 3, lo: float = -0.5, hi: float = 0.5, iters: int = 30):
    n = degree + 2
    k = np.arange(n)
    x = (lo + hi) / 2 + (hi - lo) / 2 * np.cos(np.pi * k / (n - 1))[::-1]  # Chebyshev start
    grid = np.linspace(lo, hi, 200001)
    coeffs = None
    for _ in range(iters):
        # p(x_i) - 2^x_i = (-1)^i E 2^x_i for the coefficients and the level E
        A = np.zeros((n, n))
        for i, xi in enumerate(x):
            A[i, :degree + 1] = xi ** np.arange(degree + 1)
            A[i, degree + 1] = -((-1) ** i) * 2.0 ** xi
        sol = np.linalg.solve(A, 2.0 ** x)
        coeffs = sol[:degree + 1]
        err = (np.polyval(coeffs[::-1], grid) - 2.0 ** grid) / 2.0 ** grid
        # new reference: the extreme error of each run of equal sign
        sign = np.sign(err)
        idx, start = [], 0
        for j in range(1, len(grid) + 1):
            if j == len(grid) or sign[j] != sign[start]:
                idx.append(start + int(np.argmax(np.abs(err[start:j]))))
                start = j
        if len(idx) >= n:
            while len(idx) > n:
                idx.pop(0 if abs(err[idx[0]]) < abs(err[idx[-1]]) else -1)
            x = grid[idx]
    max_rel = float(np.max(np.abs((np.polyval(coeffs[::-1], grid) - 2.0 ** grid) / 2.0 ** grid)))
    return coeffs, max_rel


if __name__ == "__main__":
    c, e = remez_exp2()
    c32 = c.astype(np.float32)
    grid = np.linspace(-0.5, 0.5, 200001)
    e32 = float(np.max(np.abs((np.polyval(c32.astype(np.float64)[::-1], grid) - 2.0 ** grid) / 2.0 ** grid)))
    for i, v in enumerate(c32):
        print(f"c{i} = {float(v):.9g}f  ({v.view(np.uint32):#010x})")
    print(f"max relative error {e:.3e} (float32 coefficients: {e32:.3e})")
