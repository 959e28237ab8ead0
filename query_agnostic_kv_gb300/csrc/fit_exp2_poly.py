"""Coefficients of the software exp2 used by the row-LSE scoring pass.

Method (Cody-Waite range reduction with a minimax polynomial, the split of
the exponential between the MUFU unit and the FMA pipe popularised by
FlashAttention-4): 2^x = 2^n * 2^f with n = round(x), f = x - n in
[-0.5, 0.5]; 2^f is a degree-3 polynomial fitted here by linear
programming to minimise the maximum *relative* error on [-0.5, 0.5]; 2^n is
applied by adding n to the exponent field.

Run this to regenerate the constants of EXP2_C0..EXP2_C3 in kvc_recon.cu:
    python query_agnostic_kv_gb300/csrc/fit_exp2_poly.py
"""
import numpy as np
from scipy.optimize import linprog


def fit(deg: int = 3, npts: int = 4001):
    x = np.linspace(-0.5, 0.5, npts)
    y = np.exp2(x)
    A = np.vander(x, deg + 1, increasing=True) / y[:, None]
    n = deg + 1
    a_ub = np.vstack([np.hstack([A, -np.ones((npts, 1))]), np.hstack([-A, -np.ones((npts, 1))])])
    b_ub = np.concatenate([np.ones(npts), -np.ones(npts)])
    c = np.zeros(n + 1)
    c[-1] = 1.0
    r = linprog(c, A_ub=a_ub, b_ub=b_ub, bounds=[(None, None)] * n + [(0, None)], method="highs")
    return r.x[:n].astype(np.float32), float(r.x[-1])


if __name__ == "__main__":
    coef, bound = fit()
    for i, v in enumerate(coef):
        print(f"constexpr float EXP2_C{i} = {float(v)!r}f;")
    print(f"// max relative error of the fit: {bound:.3e}")
