"""Coefficients of the odd polynomial tanh used by the prefill kernel's
soft-cap on small arguments (prefill_kernel.cuh, kTanhC).

tanh(y) ~ y * sum_{i=0..6} c_i y^(2i) on |y| <= 1: a minimax fit (Lawson's
iteratively reweighted least squares on a dense grid of [0, 1], the error
of an odd function being symmetric), degree 13.  Prints the coefficients as
C float literals and the maximum error of the fit in fp64 and of its fp32
Horner evaluation against numpy's tanh.  Run: python gen_tanh_poly.py
"""
import numpy as np

T, K = 1.0, 6


def fit(T, k, iters=80):
    y = np.unique(np.concatenate([np.linspace(0, T, 40001),
                                  T * (1 - np.cos(np.linspace(0, np.pi / 2, 40001)))]))
    z = y * y
    t = np.tanh(y)
    w = np.ones_like(y)
    best = None
    for _ in range(iters):
        A = np.stack([y * z ** i for i in range(k + 1)], 1)
        c, *_ = np.linalg.lstsq(A * w[:, None], t * w, rcond=None)
        err = A @ c - t
        m = np.abs(err).max()
        if best is None or m < best[0]:
            best = (m, c)
        w = w * np.sqrt(np.abs(err) / m + 1e-4)
        w /= w.max()
    return best


def fp32_error(c, T):
    y = np.linspace(-T, T, 2_000_001).astype(np.float32)
    z = y * y
    p = np.float32(c[-1])
    for cc in c[-2::-1]:
        p = p * z + np.float32(cc)
    return float(np.abs((y * p).astype(np.float64) - np.tanh(y.astype(np.float64))).max())


if __name__ == "__main__":
    m, c = fit(T, K)
    c32 = [float(np.float32(x)) for x in c]
    print("constexpr float kTanhC[%d] = {%s};" % (K + 1, ", ".join("%.9ef" % x for x in c32)))
    print("fit max error %.3e (fp64), %.3e (fp32 evaluation) on |y| <= %g" % (m, fp32_error(c32, T), T))
