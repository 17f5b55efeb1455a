#!/usr/bin/env python3
"""Writes exp2_poly.h: a minimax polynomial for 2^f on [-1/2, 1/2].

The prefill kernel evaluates part of its exponentials on the FMA pipe
instead of the special-function unit.  It splits x = n + f with n the
nearest integer (|f| <= 1/2), evaluates 2^f by a polynomial and adds n to the
float's exponent field.  The polynomial coefficients come from the Remez
exchange algorithm applied to the relative error |p(f) / 2^f - 1| (weight
2^-f), run here in numpy float64; the script prints the achieved bound.

Run:  python gen_exp2_poly.py [degree]   (default 3), from this directory.
"""
import os
import sys

import numpy as np


def remez_relative(degree, lo=-0.5, hi=0.5, iters=30):
    n = degree
    # Chebyshev points as the initial reference (n + 2 points)
    k = np.arange(n + 2)
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * (n + 1 - k) / (n + 1))
    f = lambda t: np.exp2(t)
    for _ in range(iters):
        # p(x_i) - 2^x_i = (-1)^i E 2^x_i  ->  linear system in (c_0..c_n, E)
        A = np.zeros((n + 2, n + 2))
        for i, xi in enumerate(x):
            A[i, :n + 1] = xi ** np.arange(n + 1)
            A[i, n + 1] = -((-1) ** i) * f(xi)
        sol = np.linalg.solve(A, f(x))
        c, E = sol[:n + 1], sol[n + 1]
        # new reference: extrema of the relative error on a fine grid
        g = np.linspace(lo, hi, 200001)
        err = np.polyval(c[::-1], g) / f(g) - 1.0
        # split the grid into sign-alternating runs, keep the extreme of each
        sgn = np.sign(err)
        idx, start = [], 0
        for t in range(1, len(g) + 1):
            if t == len(g) or sgn[t] != sgn[start]:
                seg = np.arange(start, t)
                idx.append(seg[np.argmax(np.abs(err[seg]))])
                start = t
        if len(idx) >= n + 2:
            # keep n + 2 alternating extrema with the largest error
            while len(idx) > n + 2:
                if abs(err[idx[0]]) < abs(err[idx[-1]]):
                    idx = idx[1:]
                else:
                    idx = idx[:-1]
            x = g[np.array(idx)]
    g = np.linspace(lo, hi, 400001)
    err = np.max(np.abs(np.polyval(c[::-1], g) / f(g) - 1.0))
    return c, err, abs(E)


def main():
    degree = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c, err, E = remez_relative(degree)
    c32 = [float(np.float32(v)) for v in c]
    here = os.path.dirname(os.path.abspath(__file__))
    lines = [
        "// exp2_poly.h — written by gen_exp2_poly.py; do not edit.",
        f"// Minimax (Remez, relative error) polynomial of degree {degree} for 2^f, f in [-1/2, 1/2].",
        f"// Max relative error in exact arithmetic: {err:.3e}.",
        "#pragma once",
        f"#define MHA_EXP2_POLY_DEGREE {degree}",
    ]
    for i, v in enumerate(c32):
        lines.append(f"#define MHA_EXP2_POLY_C{i} {v!r}f")
    open(os.path.join(here, "exp2_poly.h"), "w").write("\n".join(lines) + "\n")
    print(f"degree {degree}: coefficients {c32}, max rel err {err:.3e} (equioscillation {E:.3e})")


if __name__ == "__main__":
    main()
