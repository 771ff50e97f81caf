"""Fits the polynomial behind the FMA-pipe 2^x of the attention softmax
(exp2_fma / exp2_fma_x2 in skiparse_dev.cuh) and prints its float32 coefficients.

The device routine reduces x to j = round(x) and f = x - j in [-1/2, 1/2], so it
needs p(f) ~ 2^f on that interval. The coefficients here minimise the largest
RELATIVE error max |p(f) / 2^f - 1| (the quantity that survives the exact
scaling by 2^j), found by the Remez exchange algorithm: on n + 2 reference
points solve p(x_i) - 2^x_i = (-1)^i E 2^x_i for the n + 1 coefficients and the
levelled error E, move the references to the extrema of the error curve, and
repeat until the extrema are level. The float64 result is rounded to float32
and the error re-measured with float32 Horner steps (fused multiply-adds), which
is what the kernel evaluates.

Usage: python exp2_poly_fit.py [degree]   (the kernels use degree 3)
"""
from __future__ import annotations

import sys

import numpy as np

LO, HI = -0.5, 0.5


def remez(deg: int, iters: int = 30):
    """Coefficients c[0..deg] (ascending powers) and the levelled relative error."""
    n = deg + 2
    # start from the Chebyshev extrema
    x = 0.5 * (LO + HI) + 0.5 * (HI - LO) * -np.cos(np.pi * np.arange(n) / (n - 1))
    grid = np.linspace(LO, HI, 200001)
    c, E = None, None
    for _ in range(iters):
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * 2.0 ** x[i]
        sol = np.linalg.solve(A, 2.0 ** x)
        c, E = sol[:deg + 1], sol[deg + 1]
        err = np.polyval(c[::-1], grid) / 2.0 ** grid - 1.0
        # one extremum per sign-alternating run of the error curve
        sgn = np.sign(err)
        cuts = np.flatnonzero(np.diff(sgn) != 0) + 1
        runs = np.split(np.arange(len(grid)), cuts)
        ext = [r[np.argmax(np.abs(err[r]))] for r in runs]
        if len(ext) != n:
            break
        x_new = grid[ext]
        if np.max(np.abs(x_new - x)) < 1e-12:
            x = x_new
            break
        x = x_new
    return c, abs(E)


def float32_error(c32: np.ndarray, samples: int = 1 << 20) -> float:
    """Largest relative error of float32 Horner evaluation (one rounding per
    fused multiply-add step) against float64 2^f over [-1/2, 1/2]."""
    f = np.linspace(LO, HI, samples).astype(np.float32).astype(np.float64)
    p = np.full_like(f, float(c32[-1]))
    for ck in c32[-2::-1]:
        p = (p * f + float(ck)).astype(np.float32).astype(np.float64)   # fma: one rounding
    return float(np.max(np.abs(p / 2.0 ** f - 1.0)))


def main(deg: int = 3):
    c, E = remez(deg)
    c32 = c.astype(np.float32)
    print(f"degree {deg}: levelled relative error {E:.3e}, float32 evaluation {float32_error(c32):.3e}")
    for k, v in enumerate(c32):
        print(f"  c{k} = {float(v)!r:>24}  ({float(v).hex()})")


if __name__ == "__main__":
    main(int(sys.argv[1]) if len(sys.argv) > 1 else 3)
