"""Derives the polynomial used for part of the softmax exponentials.

Method: range reduction followed by a minimax polynomial (Remez exchange),
both computed here from first principles, never taken from a math library.

  2^x = 2^n * 2^f,   n = round-to-nearest(x),  f = x - n in [-1/2, 1/2]

2^n is formed by adding n to the float's exponent field; 2^f is approximated
by the degree-DEG polynomial p that minimises the maximum RELATIVE error
max |p(f) / 2^f - 1| over [-1/2, 1/2].  The Remez exchange solves, on DEG + 2
reference points x_i, the linear system p(x_i) - 2^{x_i} = (-1)^i E 2^{x_i},
moves the reference to the alternating extrema of the weighted error, and
repeats until the extrema level out.

Running this file prints the coefficients (float32, Horner order c0..cDEG)
and the achieved error; the values are written into exp2_poly.h.
"""
from __future__ import annotations

import sys

import numpy as np

LO, HI = -0.5, 0.5


def remez(deg: int, iters: int = 60):
    m = deg + 2
    # Chebyshev-distributed initial reference
    k = np.arange(m)
    x = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * (m - 1 - k) / (m - 1))
    grid = np.linspace(LO, HI, 200001)
    coef = None
    for _ in range(iters):
        A = np.zeros((m, m))
        for i in range(m):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * 2.0 ** x[i]
        sol = np.linalg.solve(A, 2.0 ** x)
        coef, E = sol[:deg + 1], sol[deg + 1]
        err = np.polyval(coef[::-1], grid) / 2.0 ** grid - 1.0
        # alternating extrema: split the grid at sign changes, take max |err| per run
        sign = np.sign(err)
        sign[sign == 0] = 1
        cuts = np.flatnonzero(np.diff(sign)) + 1
        runs = np.split(np.arange(grid.size), cuts)
        ext = [r[np.argmax(np.abs(err[r]))] for r in runs]
        if len(ext) > m:  # keep the m largest, in order
            order = np.sort(np.argsort(-np.abs(err[ext]))[:m])
            ext = [ext[i] for i in order]
        if len(ext) < m:
            break
        new_x = grid[ext]
        if np.max(np.abs(new_x - x)) < 1e-12:
            x = new_x
            break
        x = new_x
    err = np.polyval(coef[::-1], grid) / 2.0 ** grid - 1.0
    return coef, float(np.max(np.abs(err)))


def float32_error(coef32: np.ndarray) -> float:
    """Max relative error of the float32 Horner evaluation over [-1/2, 1/2]."""
    f = np.linspace(LO, HI, 2000001, dtype=np.float64).astype(np.float32)
    p = np.float32(coef32[-1])
    for c in coef32[-2::-1]:
        p = (p * f + np.float32(c)).astype(np.float32)
    return float(np.max(np.abs(p.astype(np.float64) / 2.0 ** f.astype(np.float64) - 1.0)))


def main(deg: int = 3):
    coef, e = remez(deg)
    c32 = coef.astype(np.float32)
    e32 = float32_error(c32)
    print(f"degree {deg}: minimax relative error {e:.3e} (float64), {e32:.3e} (float32 Horner)")
    for i, c in enumerate(c32):
        print(f"  c{i} = {float(c)!r}f  // {c.view(np.uint32):#010x}")
    return c32, e32


if __name__ == "__main__":
    main(int(sys.argv[1]) if len(sys.argv) > 1 else 3)
