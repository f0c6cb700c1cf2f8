"""Fits the odd polynomial the softcap kernels use for tanh on [-T, T].

tanh(y) ~= y * P(y^2), P of degree n in y^2, fitted for minimum maximum
relative error with Lawson-weighted least squares on Chebyshev nodes (float64),
then checked in float32 Horner arithmetic.  Prints the coefficients as C
literals.  Run: python fit_tanh_poly.py [T] [n]
"""
import sys

import numpy as np


def fit(T: float, n: int, iters: int = 60):
    k = np.arange(4000)
    y = T * (0.5 + 0.5 * np.cos(np.pi * (k + 0.5) / len(k)))  # Chebyshev nodes on (0, T)
    y = y[y > 1e-6]
    f = np.tanh(y) / y                                         # target for P(y^2)
    A = np.stack([y ** (2 * j) for j in range(n + 1)], axis=1)
    w = np.ones_like(y)
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(A * sw[:, None], f * sw, rcond=None)
        err = np.abs(A @ c - f) / f
        w = w * err
        w /= w.sum()
    return c


def check_f32(c, T):
    y = np.linspace(-T, T, 200001).astype(np.float32)
    y2 = (y * y).astype(np.float32)
    acc = np.float32(c[-1])
    for cj in c[-2::-1]:
        acc = (acc * y2 + np.float32(cj)).astype(np.float32)
    t = (y * acc).astype(np.float32)
    ref = np.tanh(y.astype(np.float64))
    nz = np.abs(ref) > 0
    return float(np.max(np.abs(t[nz] - ref[nz]) / np.abs(ref[nz]))), float(np.max(np.abs(t - ref)))


if __name__ == "__main__":
    T = float(sys.argv[1]) if len(sys.argv) > 1 else 0.75
    n = int(sys.argv[2]) if len(sys.argv) > 2 else 5
    c = fit(T, n)
    rel, ab = check_f32(c, T)
    print(f"T={T} degree {2 * n + 1}: float32 max rel err {rel:.3e}, max abs err {ab:.3e}")
    for j, cj in enumerate(c):
        print(f"  c{j} = {float(np.float32(cj)):.9g}f  // y^{2 * j + 1}")
