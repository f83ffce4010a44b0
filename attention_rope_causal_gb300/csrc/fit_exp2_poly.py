"""Fits the polynomial behind exp2_poly.cuh: a minimax (relative error) polynomial for 2^f on
[0, 1), solved as a linear program on a dense grid (minimise t subject to |p(f_i) - 2^f_i| <= t 2^f_i),
then rounded to fp32 and re-evaluated in fp32 Horner form to report the error actually realised.
Run: python fit_exp2_poly.py   (prints the coefficients for degrees 3 and 4)
"""
import numpy as np
from scipy.optimize import linprog
for deg in (3, 4):
    f = np.linspace(0.0, 1.0, 4001)
    y = np.exp2(f)
    # variables: c0..cdeg, t ; minimize t ; |sum c_k f^k - y| <= t*y
    V = np.vstack([f**k for k in range(deg + 1)]).T
    A = np.vstack([np.hstack([V, -y[:, None]]), np.hstack([-V, -y[:, None]])])
    b = np.hstack([y, -y])
    c = np.zeros(deg + 2); c[-1] = 1
    res = linprog(c, A_ub=A, b_ub=b, bounds=[(None, None)] * (deg + 1) + [(0, None)], method="highs")
    coef = res.x[:deg + 1]
    c32 = coef.astype(np.float32)
    ff = np.linspace(0, 1, 200001, dtype=np.float32)[:-1]
    p = np.float32(c32[deg])
    for k in range(deg - 1, -1, -1):
        p = (p * ff + c32[k]).astype(np.float32)
    rel = np.abs(p.astype(np.float64) - np.exp2(ff.astype(np.float64))) / np.exp2(ff.astype(np.float64))
    print(deg, "lp bound", res.x[-1], "fp32 max rel err", rel.max())
    print("   coef", [float(x) for x in c32], [x.view(np.uint32).item() for x in c32])
