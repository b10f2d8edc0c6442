"""Fits the polynomial for 2^f, f in [-0.5, 0.5], used by the kernels'
FMA-pipe exponential (csrc/common.cuh, exp2_fma).

Degree-3 polynomial, Lawson-reweighted least squares on Chebyshev nodes
toward the minimax relative error.  Printed coefficients are rounded to
float32; the fitted maximum relative error is about 7.5e-5, well below the
bf16 rounding (2^-9) the probabilities undergo afterwards.
"""
import numpy as np


def fit(deg=3, n=2000, iters=200):
    f = 0.5 * np.cos(np.pi * (np.arange(n) + 0.5) / n)
    y = np.exp2(f)
    A = np.vstack([f ** k for k in range(deg + 1)]).T / y[:, None]
    rhs = np.ones(n)
    wt = np.ones(n)
    for _ in range(iters):
        s = np.sqrt(wt)
        c, *_ = np.linalg.lstsq(A * s[:, None], rhs * s, rcond=None)
        err = np.abs(A @ c - rhs)
        wt *= err / err.mean()
        wt /= wt.sum()
    return [np.float32(x) for x in c]


def max_rel_err(c):
    x = np.linspace(-0.5, 0.5, 200001).astype(np.float32)
    p = np.full_like(x, c[-1])
    for k in range(len(c) - 2, -1, -1):
        p = p * x + c[k]
    return float(np.max(np.abs(p.astype(np.float64) / np.exp2(x.astype(np.float64)) - 1)))


if __name__ == "__main__":
    c = fit()
    print("coefficients c0..c3:", ", ".join(f"{float(x):.9g}f" for x in c))
    print("max relative error:", max_rel_err(c))
