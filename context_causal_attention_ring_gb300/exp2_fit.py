"""Derives the coefficients of the cubic used for 2^f, f in [-1/2, 1/2], in the
forward kernel's FMA-pipe exponential (the other exponentials use the MUFU
ex2 instruction).

Minimax fit of the relative error |p(f) / 2^f - 1| by the Remez exchange
algorithm (equioscillation at deg + 2 reference points), started from
Chebyshev nodes. Run it to reprint the coefficients:

    python -m context_causal_attention_ring_gb300.exp2_fit
"""
import numpy as np

DEG = 3
LO, HI = -0.5, 0.5


def remez(deg=DEG, iters=30):
    n = deg + 2
    k = np.arange(n)
    x = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * (n - 1 - k) / (n - 1))
    grid = np.linspace(LO, HI, 200001)
    for _ in range(iters):
        # solve p(x_i) - 2^x_i = (-1)^i E 2^x_i for the coefficients and E
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = -((-1) ** i) * 2.0 ** x[i]
        sol = np.linalg.solve(A, 2.0 ** x)
        c = sol[:deg + 1]
        err = np.polyval(c[::-1], grid) / 2.0 ** grid - 1.0
        # new reference: the extremum of each sign run
        idx = []
        sign = np.sign(err)
        start = 0
        for j in range(1, len(grid) + 1):
            if j == len(grid) or sign[j] != sign[start]:
                seg = np.arange(start, j)
                idx.append(seg[np.argmax(np.abs(err[seg]))])
                start = j
        if len(idx) >= n:
            # keep the n largest alternating extrema
            while len(idx) > n:
                drop = 0 if abs(err[idx[0]]) < abs(err[idx[-1]]) else len(idx) - 1
                idx.pop(drop)
            x = grid[idx]
    return c, float(np.abs(err).max())


if __name__ == "__main__":
    c, e = remez()
    print("coefficients c0..c3:", ", ".join(f"{v:.9g}" for v in c))
    print("max relative error:", e)
