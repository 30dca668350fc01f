"""Fit the cubic used for 2^f, f in [-1/2, 1/2], by the prefill softmax.

Method: weighted least squares on the relative error, refined by Lawson's
iteration (reweighting by the current error) towards the minimax fit.  The
kernel computes 2^x = 2^round(x) * p(x - round(x)); round() is done by adding
1.5 * 2^23 in fp32 (the sum's low mantissa bits hold the integer), and
2^round(x) is applied by adding round(x) << 23 to p's bit pattern.  Run this
script to reproduce the constants in prefill.cu; the self-test entry point
pa_selftest_exp2 checks the device result against CUDA's exp2f.
"""
import numpy as np


def fit(degree: int = 3, iters: int = 60):
    f = np.linspace(-0.5, 0.5, 200001)
    y = np.exp2(f)
    A = np.stack([f ** k for k in range(degree + 1)], 1) / y[:, None]
    w = np.ones_like(f)
    c = None
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(A * w[:, None], w, rcond=None)
        err = np.abs(A @ c - 1)
        w = w * (err + 1e-18) ** 0.5
        w /= w.mean()
    rel = float(np.max(np.abs(A @ c - 1)))
    return c, rel


if __name__ == "__main__":
    c, rel = fit()
    print("coefficients (c0..c3):", ", ".join(f"{x:.9g}f" for x in c))
    print("max relative error on [-1/2, 1/2]:", rel)
