"""Derives the coefficients of the cubic used by the kernels' FMA-pipe exp2.

Method: 2^x = 2^j * 2^f with j = round(x) and f = x - j in [-1/2, 1/2] (exact range
reduction in base 2); 2^f is approximated by the cubic c0 + c1 f + c2 f^2 + c3 f^3 that
minimises the maximum relative error on [-1/2, 1/2] -- a discretised Chebyshev (minimax)
approximation solved as a linear program: minimise t subject to
|p(f_i) - 2^f_i| <= t * 2^f_i on a dense grid of f_i.  The coefficients are then rounded to
float32 and the float32 evaluation (Horner, fused multiply-adds) is re-checked.

    python sparse_prefill_gqa_b300/csrc/exp2_poly_fit.py

prints the coefficients used in prefill_tc.cuh and the maximum relative error.
"""
import numpy as np
from scipy.optimize import linprog


def fit(degree=3, n=4001):
    f = np.linspace(-0.5, 0.5, n)
    y = np.exp2(f)
    V = np.vander(f, degree + 1, increasing=True)          # columns 1, f, f^2, f^3
    # variables: c_0..c_degree, t ; minimise t
    A_ub = np.vstack([np.hstack([V, -y[:, None]]), np.hstack([-V, -y[:, None]])])
    b_ub = np.concatenate([y, -y])
    cost = np.zeros(degree + 2)
    cost[-1] = 1.0
    res = linprog(cost, A_ub=A_ub, b_ub=b_ub, bounds=[(None, None)] * (degree + 1) + [(0, None)],
                  method="highs")
    assert res.success, res.message
    return res.x[:-1], res.x[-1]


def f32_eval(c, f):
    c = np.asarray(c, dtype=np.float32)
    f = np.asarray(f, dtype=np.float32)
    p = np.full_like(f, c[-1])
    for ck in c[-2::-1]:
        p = (p.astype(np.float64) * f + ck).astype(np.float32)   # one rounding per step, as FMA
    return p


if __name__ == "__main__":
    c, t = fit()
    c32 = np.asarray(c, dtype=np.float32)
    f = np.linspace(-0.5, 0.5, 200001).astype(np.float32)
    err = np.max(np.abs(f32_eval(c32, f).astype(np.float64) / np.exp2(f.astype(np.float64)) - 1))
    for i, ci in enumerate(c32):
        print(f"c{i} = {float(ci):.9e}f  ({ci.view(np.uint32):#010x})")
    print(f"minimax relative error {t:.3e}; float32 evaluation {err:.3e}")
