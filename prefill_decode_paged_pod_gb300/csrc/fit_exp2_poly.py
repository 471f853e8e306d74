"""Derive the polynomial the prefill softmax uses for 2^f, f in [-1/2, 1/2].

Method: Cody–Waite style range reduction 2^x = 2^n * 2^f with n = the integer
nearest to x (obtained on the FMA pipe by adding and subtracting 1.5 * 2^23)
and f = x - n in [-1/2, 1/2]; 2^f is approximated by a degree-3 polynomial
whose coefficients minimise the maximum RELATIVE error on that interval
(minimax, found by Lawson's iteratively reweighted least squares on a dense
grid), with p(0) = 1 imposed so that 2^n is exact at integers. 2^n is applied
by adding n to the exponent field. Run this file to reprint the coefficients
and the error bound the kernel relies on; its output is what pod_device.cuh
holds.
"""
import numpy as np


def fit(degree=3, iters=200, grid=20001):
    f = np.linspace(-0.5, 0.5, grid)
    y = np.exp2(f)
    # p(f) = 1 + c1 f + c2 f^2 + c3 f^3: fit c1..c3 on (y - 1) / y relative weights
    A = np.stack([f ** k for k in range(1, degree + 1)], axis=1)
    w = np.ones_like(f)
    for _ in range(iters):
        W = w / y                      # relative error weighting
        c, *_ = np.linalg.lstsq(A * W[:, None], (y - 1.0) * W, rcond=None)
        err = np.abs((1.0 + A @ c - y) / y)
        w = w * (err / err.max() + 1e-3)
        w = w / w.mean()
    p = 1.0 + A @ c
    rel = np.max(np.abs(p - y) / y)
    return c, rel


if __name__ == "__main__":
    c, rel = fit()
    # evaluate in fp32 Horner form, as the kernel does
    f = np.linspace(-0.5, 0.5, 200001, dtype=np.float32)
    c32 = c.astype(np.float32)
    p = ((c32[2] * f + c32[1]) * f + c32[0]) * f + np.float32(1.0)
    rel32 = np.max(np.abs(p.astype(np.float64) - np.exp2(f.astype(np.float64))) / np.exp2(f.astype(np.float64)))
    print("c1 = %.9e\nc2 = %.9e\nc3 = %.9e" % tuple(c32))
    print("max relative error: %.3e (fp64 fit), %.3e (fp32 Horner)" % (rel, rel32))
