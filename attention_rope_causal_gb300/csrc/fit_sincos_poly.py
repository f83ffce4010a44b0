"""Fits the polynomials behind sincos_turns() in rope.cuh: minimax (absolute error)
approximations of sin(pi/2 r) (odd, degree 7) and cos(pi/2 r) (even, degree 8) for r in [-1/2, 1/2]
(a quarter-turn fraction after exact integer reduction to the nearest quarter turn), solved as
linear programs on a dense grid, rounded to fp32, and re-evaluated in fp32 Horner form.
Run: python fit_sincos_poly.py
"""
import numpy as np
from scipy.optimize import linprog


def minimax(f, powers, lo, hi, n=6001):
    r = np.linspace(lo, hi, n)
    y = f(r)
    V = np.vstack([r ** p for p in powers]).T
    A = np.vstack([np.hstack([V, -np.ones((n, 1))]), np.hstack([-V, -np.ones((n, 1))])])
    b = np.hstack([y, -y])
    c = np.zeros(len(powers) + 1)
    c[-1] = 1
    res = linprog(c, A_ub=A, b_ub=b, bounds=[(None, None)] * len(powers) + [(0, None)], method="highs")
    return res.x[:-1], res.x[-1]


def horner_f32(coef32, x, odd):
    x = x.astype(np.float32)
    z = (x * x).astype(np.float32)
    p = np.float32(coef32[-1])
    for k in range(len(coef32) - 2, -1, -1):
        p = (p * z + np.float32(coef32[k])).astype(np.float32)
    return (p * x).astype(np.float32) if odd else p


if __name__ == "__main__":
    rr = np.linspace(-0.5, 0.5, 400001)
    s_coef, s_err = minimax(lambda r: np.sin(np.pi / 2 * r), [1, 3, 5, 7], 0.0, 0.5)
    c_coef, c_err = minimax(lambda r: np.cos(np.pi / 2 * r), [0, 2, 4, 6, 8], 0.0, 0.5)
    s32, c32 = s_coef.astype(np.float32), c_coef.astype(np.float32)
    es = np.abs(horner_f32(s32, rr, True).astype(np.float64) - np.sin(np.pi / 2 * rr)).max()
    ec = np.abs(horner_f32(c32, rr, False).astype(np.float64) - np.cos(np.pi / 2 * rr)).max()
    print("sin coef", [repr(float(x)) for x in s32], "lp", s_err, "fp32 max abs", es)
    print("cos coef", [repr(float(x)) for x in c32], "lp", c_err, "fp32 max abs", ec)
