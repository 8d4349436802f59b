"""Minimax polynomial for 2^f on [-1/2, 1/2] (relative error), by the Remez
exchange algorithm; the coefficients of the FMA-pipe exp2 in csrc/common.cuh
come from here.

exp2 on the FMA pipe (Cody and Waite's range reduction, 1980): write
x = n + f with n = round(x) an integer and f in [-1/2, 1/2]; then
2^x = 2^n * 2^f, where 2^f is this polynomial and 2^n is applied by adding n
to the float's exponent field.  The fit minimises max |p(f) / 2^f - 1| over
the interval; the coefficients are rounded to float32 and the error of the
rounded polynomial is reported.

    python -m kv_cache_compression_flash_b300.exp2_fit [degree]
"""
from __future__ import annotations

import sys

import numpy as np


def remez_exp2(degree: int, iters: int = 40, grid: int = 200001):
    """Coefficients c[0..degree] (c[0] = constant term) of the relative-error
    minimax approximation to 2^f on [-1/2, 1/2], in float64."""
    a, b = -0.5, 0.5
    n = degree + 2                                      # reference points
    k = np.arange(n)
    xs = 0.5 * (a + b) + 0.5 * (b - a) * np.cos(np.pi * (n - 1 - k) / (n - 1))   # Chebyshev extrema
    fine = np.linspace(a, b, grid)
    c = None
    for _ in range(iters):
        # p(x_i) - 2^{x_i} = (-1)^i E 2^{x_i}  (relative error equioscillates)
        A = np.zeros((n, n))
        for j in range(degree + 1):
            A[:, j] = xs ** j
        A[:, degree + 1] = -((-1.0) ** k) * np.exp2(xs)
        sol = np.linalg.solve(A, np.exp2(xs))
        c = sol[:degree + 1]
        err = np.polyval(c[::-1], fine) / np.exp2(fine) - 1.0
        # new reference: the extremum of each sign run of the error
        sgn = np.sign(err)
        sgn[sgn == 0] = 1
        cuts = np.nonzero(np.diff(sgn))[0] + 1
        runs = np.split(np.arange(grid), cuts)
        ext = [r[np.argmax(np.abs(err[r]))] for r in runs]
        if len(ext) < n:
            break
        # keep n alternating extrema with the largest errors (contiguous window)
        best, pick = -1.0, None
        for s in range(len(ext) - n + 1):
            w = ext[s:s + n]
            m = np.min(np.abs(err[w]))
            if m > best:
                best, pick = m, w
        new = fine[pick]
        if np.allclose(new, xs, atol=1e-12):
            break
        xs = new
    return c


def rounded(c):
    """The coefficients as float32 values, and the max relative error of the
    float32-coefficient polynomial on [-1/2, 1/2] (evaluated in float64)."""
    c32 = np.asarray(c, dtype=np.float32)
    f = np.linspace(-0.5, 0.5, 400001)
    err = np.abs(np.polyval(c32.astype(np.float64)[::-1], f) / np.exp2(f) - 1.0).max()
    return c32, float(err)


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c32, err = rounded(remez_exp2(deg))
    for i, v in enumerate(c32):
        print(f"c{i} = {float(v).hex()}  ({float(v)!r})")
    print(f"max relative error {err:.3e}")
