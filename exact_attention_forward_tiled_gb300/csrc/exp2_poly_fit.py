#!/usr/bin/env python3
"""Fit the polynomial behind the FMA-pipe exp2 of the softmax and write
exp2_poly.h next to this file.

2^x is split as 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2]
(a Cody-Waite style range reduction; n goes straight into the exponent
field). 2^f is approximated by a cubic p(f) that minimises the maximum
*relative* error on [-1/2, 1/2]: a Remez exchange on the error
(p(f) - 2^f) / 2^f, started from Chebyshev nodes, run in float64 and then
rounded to fp32 coefficients (the error is re-measured after rounding).

Run: python exp2_poly_fit.py   (writes exp2_poly.h, prints the max error)
"""
import os

import numpy as np

DEG = 3
LO, HI = -0.5, 0.5


def remez(deg, iters=30):
    n = deg + 2
    k = np.arange(n)
    x = (LO + HI) / 2 + (HI - LO) / 2 * np.cos(np.pi * k / (n - 1))[::-1]
    grid = np.linspace(LO, HI, 200001)
    for _ in range(iters):
        # solve p(x_i) - 2^x_i = (-1)^i E 2^x_i for the coefficients and E
        A = np.zeros((n, n))
        for i, xi in enumerate(x):
            A[i, :deg + 1] = xi ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * 2.0 ** xi
        b = 2.0 ** x
        sol = np.linalg.solve(A, b)
        c = sol[:deg + 1]
        err = (np.polyval(c[::-1], grid) - 2.0 ** grid) / 2.0 ** grid
        # new reference: the extrema of the error between its sign changes
        s = np.sign(err)
        edges = np.flatnonzero(np.diff(s) != 0)
        segs = np.split(np.arange(len(grid)), edges + 1)
        ext = [seg[np.argmax(np.abs(err[seg]))] for seg in segs]
        if len(ext) != n:
            break
        x = grid[ext]
    return c, np.abs(err).max()


def main():
    c, e64 = remez(DEG)
    c32 = c.astype(np.float32)
    grid = np.linspace(LO, HI, 200001)
    p32 = np.zeros_like(grid, dtype=np.float32)
    for ck in c32[::-1]:
        p32 = (p32 * grid.astype(np.float32) + ck).astype(np.float32)
    e32 = np.abs((p32.astype(np.float64) - 2.0 ** grid) / 2.0 ** grid).max()
    here = os.path.dirname(os.path.abspath(__file__))
    lines = [
        "// Written by exp2_poly_fit.py -- do not edit by hand.",
        f"// 2^f on [-1/2, 1/2] by a degree-{DEG} minimax (relative error) polynomial,",
        f"// Remez exchange in float64; max relative error {e64:.3e} (float64 coefficients),",
        f"// {e32:.3e} with these fp32 coefficients evaluated in fp32 Horner form.",
        "#pragma once",
        "namespace fa {",
    ]
    for k, ck in enumerate(c32):
        lines.append(f"constexpr float kExp2C{k} = {float(ck)!r}f;")
    lines.append("}  // namespace fa")
    with open(os.path.join(here, "exp2_poly.h"), "w") as f:
        f.write("\n".join(lines) + "\n")
    print(f"degree {DEG}: max rel error {e64:.3e} (f64), {e32:.3e} (fp32 coefficients)")
    print("coefficients:", [float(x) for x in c32])


if __name__ == "__main__":
    main()
