"""Pins of the Mamba-2 scan oracle (oracle.ssd) against computations other
than its recurrence.

1. The quadratic ("dual") form: with cum_t = sum_{k<=t} dt_k and the
   per-head decay A, the state after token t is
     S_t = sum_{s<=t} exp(A (cum_t - cum_s)) dt_s B_s x_s^T + exp(A cum_t) S_0
   so y is a masked (L x L) matrix product (numpy einsum), not a loop over t.
2. A = 0 (A_log = -inf): the state is a running sum (numpy cumsum).
3. A -> -inf: no memory, y_t = dt_t (C_t . B_t) x_t + D x_t.
4. Planted mistakes in copies of the C code are each rejected by pin 1.
"""
import numpy as np
import pytest
from hypothesis import given, settings, strategies as st

import oracle


def softplus(v):
    return np.where(v > 20.0, v, np.log1p(np.exp(np.minimum(v, 20.0))))


def silu(v):
    return v / (1.0 + np.exp(-v))


def problem(B=2, L=37, H=4, P=3, G=2, N=5, seed=0, gate=True, state=True):
    rng = np.random.default_rng(seed)
    return dict(x=rng.normal(size=(B, L, H, P)), dt_raw=rng.uniform(-4.0, 1.0, size=(B, L, H)),
                A_log=rng.normal(scale=0.5, size=H), Bm=rng.normal(size=(B, L, G, N)),
                Cm=rng.normal(size=(B, L, G, N)), Dskip=rng.normal(size=H),
                z=rng.normal(size=(B, L, H, P)) if gate else None,
                h0=rng.normal(scale=0.3, size=(B, H, N, P)) if state else None)


def dual_form(p):
    x, dtr, Al, Bm, Cm, Dk, z, h0 = (p[k] for k in ("x", "dt_raw", "A_log", "Bm", "Cm", "Dskip", "z", "h0"))
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    dt = softplus(dtr)                                   # (B, L, H)
    A = -np.exp(Al)                                      # (H,)
    cum = np.cumsum(dt, axis=1)                          # (B, L, H)
    g = np.arange(H) // (H // G)
    Bh, Ch = Bm[:, :, g, :], Cm[:, :, g, :]              # (B, L, H, N)
    diff = cum[:, :, None, :] - cum[:, None, :, :]       # (B, t, s, H)
    mask = np.tril(np.ones((L, L)))[None, :, :, None]
    W = np.exp(A * np.where(mask > 0, diff, 0.0)) * mask  # decay from s to t
    CB = np.einsum("bthn,bshn->btsh", Ch, Bh)
    y = np.einsum("btsh,bsh,bshp->bthp", W * CB, dt, x)
    S = np.einsum("btsh,bsh,bshn,bshp->bthnp", W, dt, Bh, x)
    if h0 is not None:
        dec = np.exp(A * cum)                            # (B, L, H)
        y = y + np.einsum("bthn,bhnp,bth->bthp", Ch, h0, dec)
        S = S + np.einsum("bhnp,bth->bthnp", h0, dec)
    y = y + Dk[None, None, :, None] * x
    if z is not None:
        y = y * silu(z)
    return y, S[:, -1]


@pytest.mark.parametrize("kw", [dict(), dict(gate=False, state=False), dict(G=1, H=3, P=4), dict(L=1)])
def test_dual_form(kw):
    p = problem(**kw)
    y, fs = oracle.ssd(**p)
    yr, fsr = dual_form(p)
    np.testing.assert_allclose(y, yr, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(fs, fsr, rtol=1e-10, atol=1e-12)


def test_no_decay_is_a_running_sum():
    p = problem(gate=False, state=False, G=1)
    p["A_log"] = np.full_like(p["A_log"], -np.inf)  # A = -exp(-inf) = 0
    y, fs = oracle.ssd(**p)
    dt = softplus(p["dt_raw"])
    inc = np.einsum("blh,bln,blhp->blhnp", dt, p["Bm"][:, :, 0], p["x"])
    S = np.cumsum(inc, axis=1)
    yr = np.einsum("bln,blhnp->blhp", p["Cm"][:, :, 0], S) + p["Dskip"][None, None, :, None] * p["x"]
    np.testing.assert_allclose(y, yr, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(fs, S[:, -1], rtol=1e-11, atol=1e-12)


def test_fast_decay_forgets():
    p = problem(gate=False, G=1)
    p["A_log"] = np.full_like(p["A_log"], 60.0)  # A = -1e26: every earlier state is gone
    y, _ = oracle.ssd(**p)
    dt = softplus(p["dt_raw"])
    cb = np.einsum("bln,bln->bl", p["Cm"][:, :, 0], p["Bm"][:, :, 0])
    yr = (dt * cb[:, :, None])[..., None] * p["x"] + p["Dskip"][None, None, :, None] * p["x"]
    np.testing.assert_allclose(y, yr, rtol=1e-12, atol=1e-12)


MUTANTS = [
    ("input without dt", "= a * S[n * P + p] + dt * Br[n] * xr[p];", "= a * S[n * P + p] + Br[n] * xr[p];"),
    ("decay sign", "double a = exp(dt * A);", "double a = exp(-dt * A);"),
    ("group index by modulo", "int g = h / hpg;", "int g = h % G;"),
    ("skip term dropped", "double v = acc + Dskip[h] * xr[p];", "double v = acc;"),
    ("gate without SiLU", "if (z) v *= silu(z[", "if (z) v *= (z["),
    ("read-out from B", "for (int n = 0; n < N; ++n) acc += Cr[n] * S[n * P + p];",
     "for (int n = 0; n < N; ++n) acc += Br[n] * S[n * P + p];"),
]


@pytest.mark.parametrize("what,old,new", MUTANTS)
def test_dual_form_rejects_planted_mistakes(tmp_path, what, old, new):
    src = oracle.source()
    start = src.index("void oracle_ssd_f64(")
    assert old in src[start:], what
    lib = oracle.compile_variant(src[:start] + src[start:].replace(old, new, 1), str(tmp_path / "mut.so"))
    p = problem(G=2, H=4)
    y, fs = oracle.ssd(**p, lib=lib)
    yr, fsr = dual_form(p)
    assert not (np.allclose(y, yr, rtol=1e-8, atol=1e-10) and np.allclose(fs, fsr, rtol=1e-8, atol=1e-10)), what


@settings(max_examples=60, deadline=None, derandomize=True)
@given(st.integers(1, 2), st.integers(1, 40), st.integers(1, 3), st.integers(1, 3), st.integers(1, 5),
       st.integers(1, 8), st.booleans(), st.booleans(), st.integers(0, 2 ** 31 - 1))
def test_dual_form_over_shapes(B, L, G, hpg, P, N, gate, state, seed):
    """The quadratic form on random small shapes: any number of groups and
    heads per group, head and state widths, with and without gate and
    initial state."""
    p = problem(B=B, L=L, H=G * hpg, P=P, G=G, N=N, seed=seed, gate=gate, state=state)
    y, fs = oracle.ssd(**p)
    yr, fsr = dual_form(p)
    np.testing.assert_allclose(y, yr, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(fs, fsr, rtol=1e-9, atol=1e-11)
