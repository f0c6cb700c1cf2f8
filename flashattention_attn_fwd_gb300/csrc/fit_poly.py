"""Fits the two polynomials the attention kernels evaluate on the FMA pipe.

  tanh   tanh(y) ~= y * P(y^2) on |y| <= T, P of degree n in y^2
         (softcap score modification; default T = 0.5, n = 3)
  exp2   2^f ~= E(f) on 0 <= f < 1, E of degree n
         (the share of the softmax exponentials computed without the MUFU
         unit, after the Cody-Waite split x = j + f, j = floor(x);
         default n = 3)

Both are fitted for minimum maximum relative error by Lawson's iteratively
reweighted least squares on Chebyshev nodes (float64), then the float32-
rounded coefficients are checked in float32 Horner arithmetic.  The kernel
header holds the coefficients this script prints with its defaults.

    python fit_poly.py tanh [T] [n]
    python fit_poly.py exp2 [n]
"""
import sys

import numpy as np


def cheb_nodes(a: float, b: float, m: int = 4000) -> np.ndarray:
    k = np.arange(m)
    return a + (b - a) * (0.5 + 0.5 * np.cos(np.pi * (k + 0.5) / m))


def lawson(A: np.ndarray, f: np.ndarray, iters: int = 80) -> np.ndarray:
    """Coefficients c minimising max |A c - f| / |f| (Lawson's algorithm)."""
    w = np.ones(len(f))
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(A * (sw / np.abs(f))[:, None], f * sw / np.abs(f), rcond=None)
        err = np.abs(A @ c - f) / np.abs(f)
        w = w * err
        w /= w.sum()
    return c


def horner_f32(c, x):
    acc = np.float32(c[-1])
    for cj in c[-2::-1]:
        acc = (acc * x + np.float32(cj)).astype(np.float32)
    return acc


def fit_tanh(T: float, n: int):
    y = cheb_nodes(0.0, T)
    y = y[y > 1e-6]
    c = lawson(np.stack([y ** (2 * j) for j in range(n + 1)], axis=1), np.tanh(y) / y)
    c32 = np.float32(c)
    ys = np.linspace(-T, T, 400001).astype(np.float32)
    t = (ys * horner_f32(c32, (ys * ys).astype(np.float32))).astype(np.float32)
    ref = np.tanh(ys.astype(np.float64))
    nz = ref != 0
    rel = float(np.max(np.abs(t[nz] - ref[nz]) / np.abs(ref[nz])))
    return c32, rel


def fit_exp2(n: int):
    f = cheb_nodes(0.0, 1.0)
    c = lawson(np.stack([f ** j for j in range(n + 1)], axis=1), np.exp2(f))
    c32 = np.float32(c)
    fs = np.linspace(0.0, 1.0, 400001, endpoint=False).astype(np.float32)
    e = horner_f32(c32, fs)
    rel = float(np.max(np.abs(e - np.exp2(fs.astype(np.float64))) / np.exp2(fs.astype(np.float64))))
    return c32, rel


if __name__ == "__main__":
    what = sys.argv[1] if len(sys.argv) > 1 else "tanh"
    if what == "tanh":
        T = float(sys.argv[2]) if len(sys.argv) > 2 else 0.5
        n = int(sys.argv[3]) if len(sys.argv) > 3 else 3
        c, rel = fit_tanh(T, n)
        print(f"tanh on |y| <= {T}, degree {2 * n + 1}: float32 max rel err {rel:.3e}")
        for j, cj in enumerate(c):
            print(f"  p{j} = {float(cj):.9g}f  // y^{2 * j + 1}")
    elif what == "exp2":
        n = int(sys.argv[2]) if len(sys.argv) > 2 else 3
        c, rel = fit_exp2(n)
        print(f"2^f on [0, 1), degree {n}: float32 max rel err {rel:.3e}")
        for j, cj in enumerate(c):
            print(f"  e{j} = {float(cj):.9g}f  // f^{j}")
    else:
        raise SystemExit("usage: fit_poly.py tanh [T] [n] | exp2 [n]")
