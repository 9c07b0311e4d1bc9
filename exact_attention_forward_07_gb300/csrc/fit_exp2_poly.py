"""Fit the polynomial the kernel uses for 2^f, f in [-1/2, 1/2].

The software exp2 of the attention kernel (an optional share of the
softmax's exponentials evaluated on the FMA pipes instead of the
special-function unit) splits x = n + f with n = round(x), evaluates
p(f) ~= 2^f with a polynomial, and adds n to the exponent bits of p(f).

This script computes the coefficients: a minimax fit of the RELATIVE error
of 2^f on [-1/2, 1/2] by the Remez exchange algorithm (equioscillation of
the weighted error at deg + 2 points), started from Chebyshev nodes, in
float64 with numpy.  It prints the coefficients as float32 literals and
the relative error of the float32-rounded polynomial (evaluated in float64)
on a dense grid.

    python fit_exp2_poly.py [degree ...]
"""
from __future__ import annotations

import sys

import numpy as np


def remez_relative(deg: int, lo: float = -0.5, hi: float = 0.5, iters: int = 50):
    f = lambda x: np.exp2(x)  # noqa: E731
    n = deg + 2
    k = np.arange(n)
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * (n - 1 - k) / (n - 1))
    grid = np.linspace(lo, hi, 200001)
    coef = None
    for _ in range(iters):
        # p(x_i) + (-1)^i E f(x_i) = f(x_i): unknowns c_0..c_deg and E
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = (-1) ** i * f(x[i])
        sol = np.linalg.solve(A, f(x))
        coef = sol[:deg + 1]
        err = (np.polyval(coef[::-1], grid) - f(grid)) / f(grid)
        # new reference: the extremum of each sign-alternating run
        sign = np.sign(err)
        breaks = np.flatnonzero(np.diff(sign) != 0) + 1
        runs = np.split(np.arange(grid.size), breaks)
        ext = [r[np.argmax(np.abs(err[r]))] for r in runs]
        while len(ext) > n:  # drop the smallest extremum at an end
            if abs(err[ext[0]]) < abs(err[ext[-1]]):
                ext = ext[1:]
            else:
                ext = ext[:-1]
        if len(ext) < n:
            break
        x = grid[np.asarray(ext)]
    return coef


def main(argv):
    degrees = [int(a) for a in argv] or [3, 4]
    grid = np.linspace(-0.5, 0.5, 1000001)
    for deg in degrees:
        c = remez_relative(deg).astype(np.float32)
        p = np.polyval(c.astype(np.float64)[::-1], grid)
        rel = np.max(np.abs(p / np.exp2(grid) - 1.0))
        print(f"degree {deg}: max relative error {rel:.3e}")
        for i, ci in enumerate(c):
            print(f"  c{i} = {float(ci):.9e}f")


if __name__ == "__main__":
    main(sys.argv[1:])
