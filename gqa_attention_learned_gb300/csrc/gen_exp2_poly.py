"""Coefficients of the cubic used for 2^f, f in [-1/2, 1/2], in prefill.cu.

Method: Remez exchange for the minimax *relative* error of a degree-3
polynomial p(f) ~ 2^f on [-1/2, 1/2] (equioscillation at 5 points), written
from the textbook algorithm.  Combined with round-to-nearest range reduction
x = n + f, 2^x = 2^n * p(f) (the 2^n applied by adding n to the exponent
field), this gives exp2 on the FMA pipe for the part of the softmax that the
MUFU unit does not take.  Run: python gen_exp2_poly.py
"""

import numpy as np


def remez(deg=3, lo=-0.5, hi=0.5, iters=30):
    n = deg + 2
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    f = lambda t: np.exp2(t)
    for _ in range(iters):
        # solve p(x_i) - f(x_i) = (-1)^i E f(x_i) for coefficients and E
        a = np.zeros((n, n))
        for i in range(n):
            a[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            a[i, deg + 1] = -((-1) ** i) * f(x[i])
        sol = np.linalg.solve(a, f(x))
        c = sol[:deg + 1]
        grid = np.linspace(lo, hi, 200001)
        err = (np.polyval(c[::-1], grid) - f(grid)) / f(grid)
        # new reference: extrema of the error between sign changes
        idx = [0]
        for k in range(1, len(grid) - 1):
            if (err[k] - err[k - 1]) * (err[k + 1] - err[k]) <= 0:
                idx.append(k)
        idx.append(len(grid) - 1)
        cand = sorted(idx, key=lambda k: -abs(err[k]))
        pts = sorted(cand[:n])
        x = grid[pts]
    return c, float(np.max(np.abs(err)))


if __name__ == "__main__":
    c, e = remez()
    for i, v in enumerate(c):
        print(f"c{i} = {np.float32(v)!r}  ({v:.12e})")
    print(f"max relative error {e:.3e}")
