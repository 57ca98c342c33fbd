"""Fits the polynomial P(e) ~ log1p(e) / e on [0, 1/8] used by the kernels'
softplus for small e (so that softplus(v) = e * P(e), e = exp(v), needs no
reciprocal).  Method: linear least squares in the monomial basis on 4000
Chebyshev nodes of the interval, in fp64, rounded to fp32.  Running it
prints the coefficients (constant term first) that ssm_math.cuh holds, and
the maximum relative error of e * P(e) evaluated in fp32 the way the kernels
do (Estrin's scheme, fused multiply-adds).
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


def _fma32(a, b, c):
    """fp32 fused multiply-add: the exact a*b+c (fp64 holds it for fp32 inputs
    up to the last bits that matter here) rounded once to fp32."""
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def estrin32(c32, e):
    """P(e) = (c0 + c1 e) + e^2 ((c2 + c3 e) + e^2 (c4 + c5 e)) in fp32."""
    c = [np.full_like(e, v) for v in c32]
    e2 = (e * e).astype(np.float32)
    q0 = _fma32(e, c[1], c[0])
    q1 = _fma32(e, c[3], c[2])
    q2 = _fma32(e, c[5], c[4])
    return _fma32(_fma32(q2, e2, q1), e2, q0)


def max_rel_error(c32) -> float:
    e = np.linspace(LO, HI, 200001).astype(np.float32)[1:]
    r = (e * estrin32(c32, e)).astype(np.float32)
    ref = np.log1p(e.astype(np.float64))
    return float(np.max(np.abs(r - ref) / ref))


if __name__ == "__main__":
    c = fit()
    print("coefficients:", ", ".join(f"{float(v)!r}f" for v in c))
    print("max relative error:", max_rel_error(c))
