"""Coefficients of the software 2^x used for part of the softmax exponentials.

Method (Cody-Waite range reduction + minimax polynomial): write
x = n + f with n = rint(x) and f in [-1/2, 1/2]; then 2^x = 2^n * 2^f, where
2^n is applied by adding n to the binary exponent of the float and 2^f is a
degree-3 polynomial c0 + c1 f + c2 f^2 + c3 f^3 whose coefficients minimise
the maximum relative error on [-1/2, 1/2] (Remez exchange, computed below in
float64).  The result only feeds a bf16 (8-bit mantissa) or e4m3 P operand,
so a relative error near 1e-4 is far below the operand's own rounding
(2^-9 for bf16).

Run as a script to print the coefficients that attn.cu uses; the CPU tests
recompute them and check both the constants in attn.cu and the error bound.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def remez(degree: int = DEGREE, iters: int = 30):
    """Minimax relative-error fit of 2^f on [LO, HI]; returns (coeffs
    lowest degree first, max relative error)."""
    n = degree + 2
    # Chebyshev extrema as the starting reference
    k = np.arange(n)
    x = (LO + HI) / 2 + (HI - LO) / 2 * np.cos(np.pi * k[::-1] / (n - 1))
    grid = np.linspace(LO, HI, 200001)
    for _ in range(iters):
        # solve  sum_j c_j x^j - 2^x = (-1)^i E 2^x   (relative error E)
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :degree + 1] = x[i] ** np.arange(degree + 1)
            A[i, degree + 1] = -((-1) ** i) * 2.0 ** x[i]
        sol = np.linalg.solve(A, 2.0 ** x)
        c = sol[:degree + 1]
        err = np.polynomial.polynomial.polyval(grid, c) / 2.0 ** grid - 1.0
        # new reference: one extremum of the error per sign-alternating run
        idx = []
        sgn = np.sign(err)
        start = 0
        for i in range(1, len(grid) + 1):
            if i == len(grid) or sgn[i] != sgn[start]:
                seg = np.arange(start, i)
                idx.append(seg[np.argmax(np.abs(err[seg]))])
                start = i
        if len(idx) < n:
            break
        # keep the n consecutive extrema with the largest minimum magnitude
        best = max(range(len(idx) - n + 1), key=lambda s: np.min(np.abs(err[idx[s:s + n]])))
        x = grid[idx[best:best + n]]
    err = np.polynomial.polynomial.polyval(grid, c) / 2.0 ** grid - 1.0
    return c, float(np.max(np.abs(err)))


def coefficients_f32():
    c, e = remez()
    return [float(np.float32(v)) for v in c], e


if __name__ == "__main__":
    c, e = coefficients_f32()
    for i, v in enumerate(c):
        print("c%d = %.9ef" % (i, v))
    print("max relative error %.3e" % e)
