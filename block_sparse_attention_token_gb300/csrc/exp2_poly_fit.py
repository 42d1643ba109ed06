"""Coefficients of the cubic used for 2^f, f in [-1/2, 1/2], in attn_fwd_tc.cu.

Method: minimax fit in relative error by the Remez exchange algorithm (start:
the Chebyshev extrema), then each coefficient rounded to float32. 2^x is then
2^round(x) * p(x - round(x)), the power of two added to the exponent field.
bf16 probabilities need a relative error well below 2^-9.

    python exp2_poly_fit.py      # prints the coefficients and the error
"""
import numpy as np


def fit(deg=3, lo=-0.5, hi=0.5, iters=30):
    f = np.exp2
    n = deg + 2
    k = np.arange(n)
    x = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * (n - 1 - k) / (n - 1))
    grid = np.linspace(lo, hi, 200001)
    c = None
    for _ in range(iters):
        # p(x_i) + (-1)^i E f(x_i) = f(x_i): equioscillating relative error E
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = (-1) ** i * f(x[i])
        c = np.linalg.solve(A, f(x))[:deg + 1]
        err = np.polyval(c[::-1], grid) / f(grid) - 1.0
        # new reference: one extremum of largest magnitude per sign run
        runs, start = [], 0
        for j in range(1, len(grid) + 1):
            if j == len(grid) or np.sign(err[j]) != np.sign(err[start]):
                seg = slice(start, j)
                runs.append(start + int(np.argmax(np.abs(err[seg]))))
                start = j
        while len(runs) > n:
            runs.pop(0 if abs(err[runs[0]]) < abs(err[runs[-1]]) else -1)
        if len(runs) == n:
            x = grid[runs]
    return c


if __name__ == "__main__":
    c32 = fit().astype(np.float32)
    g = np.linspace(-0.5, 0.5, 1000001)
    rel = np.abs(np.polyval(c32.astype(np.float64)[::-1], g) / np.exp2(g) - 1).max()
    print("c0..c3 =", ", ".join(f"{v:.9e}f" for v in c32))
    print(f"max relative error on [-1/2, 1/2]: {rel:.3e}  (bf16 half-ulp {2.0 ** -9:.3e})")
