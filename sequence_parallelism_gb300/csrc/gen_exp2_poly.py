"""Derive the polynomial used for 2^f on the FMA pipe (attn_bf16.cu).

Method: range reduction x = n + f with n = round-to-nearest(x) (so
f in [-1/2, 1/2]) and 2^x = 2^n * 2^f; 2^f is approximated by a degree-3
polynomial with minimum relative error on [-1/2, 1/2], found by the Remez
exchange algorithm on the relative-error equioscillation conditions.  Run:

    python sequence_parallelism_gb300/csrc/gen_exp2_poly.py

and paste the printed float32 coefficients into attn_bf16.cu.
"""

import numpy as np

DEG = 3
A, B = -0.5, 0.5


def remez(deg=DEG, iters=30):
    f = lambda x: np.exp2(x)
    n = deg + 2
    # start from Chebyshev extrema
    x = (A + B) / 2 + (B - A) / 2 * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    for _ in range(iters):
        # solve sum c_k x_i^k - f(x_i) = (-1)^i E f(x_i)  (relative error)
        M = np.zeros((n, n))
        for i in range(n):
            M[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            M[i, deg + 1] = -((-1) ** i) * f(x[i])
        sol = np.linalg.solve(M, f(x))
        c, E = sol[:deg + 1], sol[deg + 1]
        # new extrema of the relative error
        g = np.linspace(A, B, 200001)
        err = np.polyval(c[::-1], g) / f(g) - 1
        idx = [0]
        for k in range(1, len(g) - 1):
            if (err[k] - err[k - 1]) * (err[k + 1] - err[k]) < 0:
                idx.append(k)
        idx.append(len(g) - 1)
        if len(idx) != n:
            # keep the n largest alternating extrema
            idx = sorted(idx, key=lambda k: -abs(err[k]))[:n]
            idx.sort()
        x = g[idx]
    return c, abs(E)


if __name__ == "__main__":
    c, E = remez()
    c32 = c.astype(np.float32)
    g = np.linspace(A, B, 1000001)
    rel = np.abs(np.polyval(c32.astype(np.float64)[::-1], g) / np.exp2(g) - 1).max()
    for k, v in enumerate(c32):
        print(f"c{k} = {float(v)!r}f  ({v.view(np.uint32):#010x})")
    print(f"max relative error on [-1/2, 1/2]: {rel:.3e} (equioscillation level {E:.3e})")
