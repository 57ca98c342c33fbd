"""Fits the polynomial P(e) ~ log1p(e) / e on [0, 1/8] used by the kernels'
softplus for small e (so that softplus(v) = e * P(e), e = exp(v), needs no
reciprocal).  Method: linear least squares in the monomial basis on 4000
Chebyshev nodes of the interval, in fp64, rounded to fp32.  Running it
prints the coefficients (constant term first) that ssm_math.cuh holds, and
the maximum relative error of e * P(e) evaluated in fp32 by Horner's rule.
"""
import numpy as np

DEGREE = 5
LO, HI = 0.0, 0.125


def fit(degree: int = DEGREE, nodes: int = 4000):
    k = np.arange(nodes)
    xs = (LO + HI) / 2 + (HI - LO) / 2 * np.cos(np.pi * (k + 0.5) / nodes)
    f = np.log1p(xs) / xs
    V = np.vander(xs, degree + 1, increasing=True)
    c, *_ = np.linalg.lstsq(V, f, rcond=None)
    return c.astype(np.float32)


def max_rel_error(c32) -> float:
    e = np.linspace(LO, HI, 200001).astype(np.float32)[1:]
    p = np.float32(c32[-1])
    for ci in c32[-2::-1]:
        p = (p * e + ci).astype(np.float32)
    r = (e * p).astype(np.float32)
    ref = np.log1p(e.astype(np.float64))
    return float(np.max(np.abs(r - ref) / ref))


if __name__ == "__main__":
    c = fit()
    print("coefficients:", ", ".join(f"{float(v)!r}f" for v in c))
    print("max relative error:", max_rel_error(c))
