"""Pins of the oracle's backward (oracle.scan_bwd) against something other
than itself: central finite differences of the forward oracle, on every
coordinate of every input of small problems, in fp64.  The loss is
sum(y*dy) + sum(final_h*dfinal_h) + sum(final_conv_state*dfinal_conv_state)
with random weights, so every output and every path through the layer
(conv, SiLU, softplus on both sides of its threshold, decay, input, read-out,
skip, gate, initial and final states) contributes.  A second test plants
plausible mistakes in a copy of the backward and checks that the finite
differences reject each."""
import numpy as np
import pytest
from hypothesis import given, settings, strategies as st

import oracle

N = 16
NAMES_IN = ("x", "z", "dt_raw", "Bm", "Cm", "A_log", "Dskip", "conv_w", "conv_b", "h0",
            "conv_state0")
GRAD_OF = {"x": "dx", "z": "dz", "dt_raw": "ddt_raw", "Bm": "dB", "Cm": "dC", "A_log": "dA_log",
           "Dskip": "dD", "conv_w": "dconv_w", "conv_b": "dconv_b", "h0": "dh0",
           "conv_state0": "dconv_state0"}


def problem(B, L, D, seed, big_dt=False):
    rng = np.random.default_rng(seed)
    p = dict(x=rng.normal(size=(B, L, D)), z=rng.normal(size=(B, L, D)),
             dt_raw=rng.uniform(-4.0, 0.5, size=(B, L, D)),
             Bm=rng.normal(size=(B, L, N)), Cm=rng.normal(size=(B, L, N)),
             A_log=np.log(np.arange(1, N + 1, dtype=float))[None, :].repeat(D, 0)
             + rng.normal(scale=0.3, size=(D, N)),
             Dskip=rng.normal(size=D), conv_w=rng.uniform(-0.5, 0.5, size=(D, 4)),
             conv_b=rng.normal(scale=0.2, size=D), h0=rng.normal(scale=0.3, size=(B, D, N)),
             conv_state0=rng.normal(size=(B, 3, D)))
    if big_dt:  # some dt_raw past softplus's threshold (20): identity branch
        p["dt_raw"][..., 0] = 20.5 + rng.uniform(size=(B, L))
        p["A_log"][0] = -8.0  # keep exp(dt*A) away from underflow there
    w = dict(dy=rng.normal(size=(B, L, D)), dfinal_h=rng.normal(size=(B, D, N)),
             dfinal_conv_state=rng.normal(size=(B, 3, D)))
    return p, w


def loss(p, w, lib=None):
    y, fh, fcs = oracle.scan(**p, lib=lib)
    return float(np.sum(y * w["dy"]) + np.sum(fh * w["dfinal_h"])
                 + np.sum(fcs * w["dfinal_conv_state"]))


def fd_check(p, w, lib=None, rel=2e-6):
    g = oracle.scan_bwd(**p, **w, lib=lib)
    worst = 0.0
    for name in NAMES_IN:
        a = p[name]
        ga = g[GRAD_OF[name]]
        for idx in np.ndindex(a.shape):
            v = a[idx]
            eps = 1e-6 * max(1.0, abs(v))
            a[idx] = v + eps
            lp = loss(p, w)
            a[idx] = v - eps
            lm = loss(p, w)
            a[idx] = v
            fd = (lp - lm) / (2 * eps)
            scale = max(1.0, abs(fd))
            err = abs(fd - ga[idx]) / scale
            worst = max(worst, err)
            if err > rel:
                return False, f"{name}{idx}: finite difference {fd:.9g} vs backward {ga[idx]:.9g}"
    return True, f"worst relative gap {worst:.2e}"


@pytest.mark.parametrize("B,L,D,big_dt", [(1, 1, 2, False), (1, 2, 2, False), (2, 5, 2, False),
                                          (1, 7, 3, True)])
def test_backward_matches_finite_differences(B, L, D, big_dt):
    p, w = problem(B, L, D, seed=10 * L + D, big_dt=big_dt)
    ok, msg = fd_check(p, w)
    assert ok, msg



@settings(max_examples=40, deadline=None, derandomize=True)
@given(st.integers(1, 2), st.integers(1, 40), st.integers(1, 4), st.booleans(), st.integers(0, 2 ** 31 - 1))
def test_backward_matches_a_directional_derivative(B, L, D, big_dt, seed):
    """On random shapes (longer sequences than the per-coordinate check
    reaches): the loss's central difference along one random direction in
    all inputs at once equals the gradients' inner product with it."""
    p, w = problem(B, L, D, seed=seed, big_dt=big_dt)
    g = oracle.scan_bwd(**p, **w)
    rng = np.random.default_rng(seed + 1)
    v = {k: rng.normal(size=p[k].shape) for k in NAMES_IN}
    eps = 1e-6
    plus = {k: p[k] + eps * v[k] for k in NAMES_IN}
    minus = {k: p[k] - eps * v[k] for k in NAMES_IN}
    fd = (loss(plus, w) - loss(minus, w)) / (2 * eps)
    an = sum(float(np.sum(g[GRAD_OF[k]] * v[k])) for k in NAMES_IN)
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (fd, an)


MUTANTS = [
    ("skip term of du dropped", "double du = dyss * Dskip[c];", "double du = 0.0;"),
    ("gate derivative sign", "return s * (1.0 + v * (1.0 - s));", "return s * (1.0 - v * (1.0 - s));"),
    ("adjoint not decayed", "lam[n] *= dA;", "lam[n] *= 1.0;"),
    ("read-out before the adjoint update", "lam[n] += Cm[r + n] * dyss;", "lam[n] += 0.0 * dyss;"),
    ("decay gradient uses h_t", "double gA = lam[n] * hs[(size_t)t * N + n];",
     "double gA = lam[n] * hs[(size_t)(t + 1) * N + n];"),
    ("A_log chain rule missing A", "dA_log[(size_t)c * N + n] += gA * dA * dt[t] * A;",
     "dA_log[(size_t)c * N + n] += gA * dA * dt[t];"),
    ("softplus derivative", "static double dsoftplus(double v) { return v > 20.0 ? 1.0 : sigmoid(v); }",
     "static double dsoftplus(double v) { return v > 20.0 ? 1.0 : sigmoid(-v); }"),
    ("conv taps reversed in dx", "din[tau + (K - 1)] += dpre * w[k];",
     "din[tau + (K - 1)] += dpre * w[K - 1 - k];"),
    ("final h gradient ignored", "lam[n] = dfinal_h ? dfinal_h[((size_t)b * D + c) * N + n] : 0.0;",
     "lam[n] = 0.0;"),
]


@pytest.mark.parametrize("what,old,new", MUTANTS)
def test_finite_differences_catch_planted_backward_mistakes(tmp_path, what, old, new):
    src = oracle.source()
    assert old in src, what
    lib = oracle.compile_variant(src.replace(old, new, 1), str(tmp_path / "liboracle_mut.so"))
    p, w = problem(1, 6, 2, seed=3)
    ok, msg = fd_check(p, w, lib=lib)
    assert not ok, f"mutant '{what}' survived ({msg})"
