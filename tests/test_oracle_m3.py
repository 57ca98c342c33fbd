"""Pins of the complex-valued scan oracle (mamba3_oracle.c: Mamba-3's state
update, as read from "Jamba -- SSM-Transformer Hibrido", section "Mamba-3: a
linha de base de SSM puro em 2026", items 1 and 2), against facts fixed
outside it:

* the page's own equivalence: a complex state update is a data-dependent
  rotary embedding -- turning B by -Phi_t and C by +Phi_t (Phi_t the
  accumulated angle dt*theta) gives a real-decay scan, which the real-valued
  oracle (pinned separately) computes, the whole layer included;
* theta = 0 with real B and C is exactly the real-valued scan;
* a pure rotation (no decay, no input) keeps |h| and turns h0 by Phi_t;
* constant dt, B, C make the layer a causal convolution with kernel
  Re(sum_n C_n alpha_n^k dt B_n) (Euler; the trapezoid halves the k = 0 tap);
* the exponential-trapezoidal rule converges at second order to the exact
  solution of h' = lambda h + B u(tau) (Euler at first order);
* splitting a sequence into calls that carry (h, conv state, previous input)
  gives the one-call result.

Planted mistakes in a copy of the C source (sign of the rotation, read-out of
the imaginary part, conjugated C, trapezoid without the decay on the earlier
input, wrong trapezoid weight, previous input not kept, final v not written)
are each rejected by a pin.
"""
import numpy as np
import pytest

import oracle

LIB = {"lib": None}  # a mutated copy's path while a mutant is checked
M = 8


def _m3(*a, **k):
    return oracle.m3_scan(*a, lib=LIB["lib"], **k)


def _core(*a, **k):
    return oracle.m3_core(*a, lib=LIB["lib"], **k)


def _softplus(v):
    return np.where(v > 20.0, v, np.log1p(np.exp(np.minimum(v, 20.0))))


def _case(rng, B=2, L=37, D=3, K=4, theta_scale=3.0, state=True):
    c = dict(x=rng.normal(size=(B, L, D)), z=rng.normal(size=(B, L, D)),
             dt_raw=np.log(np.expm1(np.exp(rng.uniform(np.log(1e-3), np.log(3e-1), size=(B, L, D))))),
             Bm=rng.normal(size=(B, L, 2 * M)), Cm=rng.normal(size=(B, L, 2 * M)),
             A_log=rng.normal(scale=0.7, size=(D, M)), theta=rng.normal(scale=theta_scale, size=(D, M)),
             Dskip=rng.normal(size=D), conv_w=rng.uniform(-0.5, 0.5, size=(D, K)), conv_b=rng.normal(size=D))
    if state:
        c["h0"] = rng.normal(size=(B, D, 2 * M))
        c["conv_state0"] = rng.normal(size=(B, K - 1, D))
    return c


def _run(c, **k):
    return _m3(c["x"], c["z"], c["dt_raw"], c["Bm"], c["Cm"], c["A_log"], c["theta"], c["Dskip"],
               c["conv_w"], c.get("conv_b"), c.get("h0"), c.get("conv_state0"), c.get("v0"), **k)


def _cplx(a):
    return a[..., 0::2] + 1j * a[..., 1::2]


def _pairs(z):
    out = np.empty(z.shape[:-1] + (2 * z.shape[-1],))
    out[..., 0::2] = z.real
    out[..., 1::2] = z.imag
    return out


def pin_rotary_equivalence_with_the_real_scan():
    """Complex scan == real-decay scan of the real-valued oracle on B turned by
    -Phi_t and C by +Phi_t, Phi_t = sum_{s<=t} dt_s theta (per channel and
    mode); the final state turned back by Phi_L."""
    rng = np.random.default_rng(1)
    c = _case(rng)
    y, fh, fcs, _ = _run(c)
    B_, L, D = c["x"].shape
    dt = _softplus(c["dt_raw"])
    for ch in range(D):
        phi = np.cumsum(dt[:, :, ch:ch + 1] * c["theta"][ch][None, None, :], axis=1)  # (B, L, M)
        Bt = _cplx(c["Bm"]) * np.exp(-1j * phi)
        Ct = _cplx(c["Cm"]) * np.exp(1j * phi)
        # real states (Re h~_n, Im h~_n): the read-out Re(C~ h~) = Re C~ Re h~ - Im C~ Im h~
        Bp = _pairs(Bt)
        Cp = _pairs(Ct.real - 1j * Ct.imag)
        A2 = np.repeat(c["A_log"][ch], 2)[None, :]
        yr, hr, csr = oracle.scan(c["x"][:, :, ch:ch + 1], c["z"][:, :, ch:ch + 1], c["dt_raw"][:, :, ch:ch + 1],
                                  Bp, Cp, A2, c["Dskip"][ch:ch + 1], c["conv_w"][ch:ch + 1], c["conv_b"][ch:ch + 1],
                                  c["h0"][:, ch:ch + 1], c["conv_state0"][:, :, ch:ch + 1])
        np.testing.assert_allclose(y[:, :, ch:ch + 1], yr, rtol=1e-10, atol=1e-12)
        hL = _cplx(hr[:, 0]) * np.exp(1j * phi[:, -1])
        np.testing.assert_allclose(_cplx(fh[:, ch]), hL, rtol=1e-10, atol=1e-12)
        np.testing.assert_array_equal(fcs[:, :, ch:ch + 1], csr)


def pin_theta_zero_real_inputs_is_the_real_scan():
    rng = np.random.default_rng(2)
    c = _case(rng)
    c["theta"][:] = 0.0
    c["Bm"][..., 1::2] = 0.0
    c["Cm"][..., 1::2] = 0.0
    c["h0"][..., 1::2] = 0.0
    y, fh, fcs, _ = _run(c)
    yr, hr, csr = oracle.scan(c["x"], c["z"], c["dt_raw"], c["Bm"][..., 0::2], c["Cm"][..., 0::2], c["A_log"],
                              c["Dskip"], c["conv_w"], c["conv_b"], c["h0"][..., 0::2], c["conv_state0"])
    np.testing.assert_allclose(y, yr, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fh[..., 0::2], hr, rtol=1e-12, atol=1e-13)
    assert np.all(fh[..., 1::2] == 0.0)
    np.testing.assert_array_equal(fcs, csr)


def pin_pure_rotation_closed_form():
    """No decay (A_log = -inf), no input (B = 0): h_t = e^{i Phi_t} h0, |h_t| = |h0|."""
    rng = np.random.default_rng(3)
    L = 50
    dt = rng.uniform(0.01, 0.5, size=L)
    theta = rng.normal(scale=2.0, size=M)
    h0 = rng.normal(size=2 * M)
    C = rng.normal(size=(L, 2 * M))
    for trap in (False, True):
        ys, h, _ = _core(rng.normal(size=L), dt, np.zeros((L, 2 * M)), C, np.full(M, -np.inf), theta, h0=h0,
                         trapezoidal=trap)
        phi = np.cumsum(dt)[:, None] * theta[None, :]
        ht = _cplx(h0)[None, :] * np.exp(1j * phi)
        np.testing.assert_allclose(ys, np.real(np.sum(_cplx(C) * ht, axis=1)), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(np.abs(_cplx(h)), np.abs(_cplx(h0)), rtol=1e-12)
        np.testing.assert_allclose(_cplx(h), ht[-1], rtol=1e-11, atol=1e-12)


def pin_constant_dt_B_C_is_a_causal_convolution():
    """ys_t = sum_k K_k u_{t-k}: Euler K_k = Re sum_n C_n alpha_n^k dt B_n;
    trapezoid the same for k >= 1 and half of it at k = 0 (numpy.convolve)."""
    rng = np.random.default_rng(4)
    L = 64
    u = rng.normal(size=L)
    dt = 0.07
    A_log = rng.normal(scale=0.5, size=M)
    theta = rng.normal(scale=2.0, size=M)
    Bc = rng.normal(size=2 * M)
    Cc = rng.normal(size=2 * M)
    alpha = np.exp(dt * (-np.exp(A_log) + 1j * theta))
    k = np.arange(L)
    kern = np.real(np.sum(_cplx(Cc)[None, :] * alpha[None, :] ** k[:, None] * dt * _cplx(Bc)[None, :], axis=1))
    for trap in (False, True):
        kk = kern.copy()
        if trap:
            kk[0] *= 0.5
        ys, _, _ = _core(u, np.full(L, dt), np.tile(Bc, (L, 1)), np.tile(Cc, (L, 1)), A_log, theta,
                         trapezoidal=trap)
        np.testing.assert_allclose(ys, np.convolve(u, kk)[:L], rtol=1e-10, atol=1e-12)


def _ode_errors(trap, lam, omega, T, h0, steps):
    """|h_n - h(T)| of the scheme with n steps of T/n on h' = lam h + cos(omega tau),
    against the exact solution."""
    errs = []
    exact = np.exp(lam * T) * h0 + 0.5 * ((np.exp(1j * omega * T) - np.exp(lam * T)) / (1j * omega - lam)
                                          + (np.exp(-1j * omega * T) - np.exp(lam * T)) / (-1j * omega - lam))
    for n in steps:
        d = T / n
        tau = d * np.arange(1, n + 1)
        Bm = np.zeros((n, 2 * M))
        Bm[:, 0] = 1.0  # mode 0 only, B = 1
        _, h, _ = _core(np.cos(omega * tau), np.full(n, d), Bm, np.zeros((n, 2 * M)),
                        np.r_[np.log(-lam.real), np.zeros(M - 1)], np.r_[lam.imag, np.zeros(M - 1)],
                        h0=np.r_[h0.real, h0.imag, np.zeros(2 * M - 2)],
                        v0=np.r_[1.0, 0.0, np.zeros(2 * M - 2)],  # u(0) = cos(0) = 1
                        trapezoidal=trap)
        errs.append(abs((h[0] + 1j * h[1]) - exact))
    return np.array(errs)


def pin_trapezoid_second_order_euler_first_order():
    lam, omega, T, h0 = -0.8 + 2.0j, 3.0, 2.0, 0.3 - 0.2j
    steps = [40, 80, 160, 320]
    et = _ode_errors(True, lam, omega, T, h0, steps)
    ee = _ode_errors(False, lam, omega, T, h0, steps)
    rt, re = et[:-1] / et[1:], ee[:-1] / ee[1:]
    assert np.all(np.abs(rt - 4.0) < 0.2), rt  # error / 4 per halving
    assert np.all(np.abs(re - 2.0) < 0.2), re  # error / 2 per halving
    assert et[-1] < 1e-3 * ee[-1] * 20


def pin_split_calls_carry_state_and_previous_input():
    rng = np.random.default_rng(5)
    c = _case(rng, L=41)
    for trap in (False, True):
        c["v0"] = rng.normal(size=c["h0"].shape)
        y, fh, fcs, fv = _run(c, trapezoidal=trap)
        parts, h, cs, v = [], c["h0"], c["conv_state0"], c["v0"]
        for t0, t1 in [(0, 1), (1, 17), (17, 41)]:
            p = dict(c, h0=h, conv_state0=cs, v0=v)
            for k in ("x", "z", "dt_raw", "Bm", "Cm"):
                p[k] = c[k][:, t0:t1]
            yp, h, cs, v = _run(p, trapezoidal=trap)
            parts.append(yp)
        np.testing.assert_allclose(np.concatenate(parts, 1), y, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(h, fh, rtol=1e-13, atol=1e-14)
        np.testing.assert_array_equal(cs, fcs)
        np.testing.assert_array_equal(v, fv)


PINS = [pin_rotary_equivalence_with_the_real_scan, pin_theta_zero_real_inputs_is_the_real_scan,
        pin_pure_rotation_closed_form, pin_constant_dt_B_C_is_a_causal_convolution,
        pin_trapezoid_second_order_euler_first_order, pin_split_calls_carry_state_and_previous_input]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


MUTANTS = {
    "rotation_sign": ("double complex lam = -exp(A_log_c[n]) + I * theta_c[n];",
                      "double complex lam = -exp(A_log_c[n]) - I * theta_c[n];"),
    "readout_imaginary_part": ("ys += creal((Ct[2 * n] + I * Ct[2 * n + 1]) * h[n]);",
                               "ys += cimag((Ct[2 * n] + I * Ct[2 * n + 1]) * h[n]);"),
    "readout_conjugated_C": ("ys += creal((Ct[2 * n] + I * Ct[2 * n + 1]) * h[n]);",
                             "ys += creal((Ct[2 * n] - I * Ct[2 * n + 1]) * h[n]);"),
    "trapezoid_earlier_input_not_decayed": ("h[n] = alpha * (h[n] + 0.5 * dt * vprev[n]) + 0.5 * dt * v;",
                                            "h[n] = alpha * h[n] + 0.5 * dt * vprev[n] + 0.5 * dt * v;"),
    "trapezoid_weight": ("h[n] = alpha * (h[n] + 0.5 * dt * vprev[n]) + 0.5 * dt * v;",
                         "h[n] = alpha * (h[n] + dt * vprev[n]) + 0.5 * dt * v;"),
    "previous_input_not_kept": ("        vprev[n] = v;\n", ""),
    "final_v_not_written": ("final_v[hs + 2 * n] = creal(vp[n]);", "final_v[hs + 2 * n] = 0.0;"),
    "state_input_without_dt": ("h[n] = alpha * h[n] + dt * v;", "h[n] = alpha * h[n] + v;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.source_m3()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = oracle.compile_variant(src.replace(old, new), str(tmp_path / f"libm3_{name}.so"))
    failed = []
    try:
        LIB["lib"] = oracle._load_m3(path)
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
                break
    finally:
        LIB["lib"] = None
    assert failed, f"no pin rejects the mutant {name}"
