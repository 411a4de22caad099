"""Fits the polynomial of the kernels' software exp2 (prints its coefficients).

Method (Cody and Waite style argument reduction, then a polynomial): for
x <= 8 write x = n + f with n = round(x) and f in [-1/2, 1/2]; then
2^x = 2^n * p(f), where p is a degree-3 polynomial approximating 2^f on
[-1/2, 1/2]. p is fitted here by iteratively reweighted least squares on
Chebyshev points toward minimax relative error; the coefficients are rounded
to float32 and the error is re-measured in double precision. 2^n is applied by
adding n to the float's exponent field.

    python fit_exp2_poly.py  ->  coefficients c0..c3 and max relative error
"""
import numpy as np


def fit(deg: int = 3):
    f = np.cos(np.linspace(0.0, np.pi, 4001)) * 0.5
    y = 2.0 ** f
    w = np.ones_like(f)
    for _ in range(60):
        a = np.vander(f, deg + 1, increasing=True) / y[:, None]
        c, *_ = np.linalg.lstsq(a * w[:, None], w, rcond=None)
        err = (np.vander(f, deg + 1, increasing=True) @ c) / y - 1.0
        w = w * (1.0 + 50.0 * np.abs(err) / np.abs(err).max())
    c32 = c.astype(np.float32)
    ff = np.linspace(-0.5, 0.5, 200001)
    p = np.polyval(c32[::-1].astype(np.float64), ff)
    return c32, float(np.max(np.abs(p / 2.0 ** ff - 1.0)))


if __name__ == "__main__":
    c, e = fit(3)
    print("coefficients:", ", ".join(f"{float(x):.9g}f" for x in c))
    print(f"max relative error on [-1/2, 1/2]: {e:.3e}")
