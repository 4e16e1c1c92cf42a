"""Fits the cubic used by the prefill kernel's software 2^x.

Method: Cody-Waite range reduction (W. J. Cody and W. Waite, "Software Manual
for the Elementary Functions", 1980): 2^x = 2^floor(x) * 2^f with
f = x - floor(x) in [0, 1). The power of two is applied by adding floor(x)
to the IEEE exponent field; 2^f is approximated by

    p(f) = 1 + c1 f + c2 f^2 + c3 f^3,   with c3 = 1 - c1 - c2

so that p(0) = 1 and p(1) = 2 exactly (the approximation is continuous
across integer x). c1, c2 minimise the maximum relative error on [0, 1]; the
minimax problem is solved as a linear program on a dense grid.

The probabilities this feeds are rounded to bf16 (8 significant bits,
relative spacing 2^-8) before the P.V product, so a relative error near
1e-4 is far below what the rounding already adds.

Run:  python gqa_flash_attention_02_gb300/csrc/fit_exp2_poly.py
"""
import numpy as np
from scipy.optimize import linprog


def fit(n=4097):
    f = np.linspace(0.0, 1.0, n)
    y = np.exp2(f)
    # p(f) - y = (f - f^3) c1 + (f^2 - f^3) c2 + (1 + f^3 - y)
    a1 = f - f ** 3
    a2 = f ** 2 - f ** 3
    r0 = 1.0 + f ** 3 - y
    # minimise t subject to |a1 c1 + a2 c2 + r0| <= t * y
    A = np.vstack([np.column_stack([a1, a2, -y]), np.column_stack([-a1, -a2, -y])])
    b = np.concatenate([-r0, r0])
    res = linprog(c=[0, 0, 1], A_ub=A, b_ub=b, bounds=[(None, None)] * 3, method="highs")
    c1, c2, t = res.x
    return c1, c2, 1.0 - c1 - c2, t


if __name__ == "__main__":
    c1, c2, c3, t = fit()
    f = np.linspace(0, 1, 100001)
    p = 1 + f * (c1 + f * (c2 + f * c3))
    rel = np.abs(p / np.exp2(f) - 1).max()
    print(f"c1 = {np.float32(c1)!r}f\nc2 = {np.float32(c2)!r}f\nc3 = {np.float32(c3)!r}f")
    print(f"max relative error on [0,1]: {rel:.3e}")
