"""Fit the polynomial used by exp2_poly() in sm100_ptx.cuh.

2^x = 2^n * 2^f with n = round(x), f = x - n in [-1/2, 1/2]; 2^f is replaced by
a cubic whose coefficients minimise the maximum RELATIVE error on [-1/2, 1/2]
(Remez exchange).  Run `python gen_exp2_poly.py` to print them; the kernel's
constants are these values rounded to fp32.
"""
import numpy as np


def remez_exp2(deg=3, a=-0.5, b=0.5, iters=40):
    n = deg + 2
    x = 0.5 * (a + b) + 0.5 * (b - a) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    t = np.linspace(a, b, 200001)
    for _ in range(iters):
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :deg + 1] = x[i] ** np.arange(deg + 1)
            A[i, deg + 1] = (-1) ** i * np.exp2(x[i])
        c = np.linalg.solve(A, np.exp2(x))[:deg + 1]
        err = (np.polyval(c[::-1], t) - np.exp2(t)) / np.exp2(t)
        ext = [0]
        for k in range(1, len(t)):
            if np.sign(err[k]) != np.sign(err[ext[-1]]):
                ext.append(k)
            elif abs(err[k]) > abs(err[ext[-1]]):
                ext[-1] = k
        if len(ext) > n:
            ext = sorted(sorted(ext, key=lambda k: -abs(err[k]))[:n])
        if len(ext) == n:
            x = t[ext]
    return c, float(np.max(np.abs(err)))


if __name__ == "__main__":
    c, e = remez_exp2()
    print("max relative error %.3e" % e)
    for i, v in enumerate(c):
        print("c%d = %.9ef" % (i, np.float32(v)))
