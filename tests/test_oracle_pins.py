"""Pins of the fp64 oracle against facts fixed outside it (CPU only).

The pages print no worked values of y, so the oracle is pinned by closed
forms and special cases that a mistake in any term would break:

* brute-force closed form of the recurrence (decay products written as
  exponentials of cumulative dt, the conv done by torch's conv1d, softplus and
  SiLU by torch.nn.functional) on tiny inputs with non-zero h0/conv_state0;
* A -> 0 (dA = 1): the state is a cumulative sum (numpy.cumsum);
* constant dt, B, C: the layer is LTI and equals a causal convolution with
  kernel K_k = sum_n C_n a_n^k dt B_n (numpy.convolve) -- the S4 view in the
  lesson's "Um SSM em uma pagina";
* A -> -inf: the state forgets everything (h_t = dt_t B_t u_t);
* B = 0: pure decay of h0, and y = D*u*silu(z);
* conv taps/bias/state against torch conv1d, softplus (incl. the threshold)
  against torch softplus, SiLU against torch silu;
* z = 0 or (C = 0 and D = 0) give exactly zero;
* the chunked evaluation equals the sequential one;
* L decode steps equal one scan bit for bit;
* the state size is independent of L and matches the pages' memory budget.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from hypothesis import given, settings, strategies as st

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(B=2, L=12, D=3, N=4, K=4, seed=0, with_state=True):
    r = np.random.default_rng(seed)
    c = dict(
        x=r.standard_normal((B, L, D)),
        z=r.standard_normal((B, L, D)),
        dt_raw=np.log(np.expm1(np.exp(r.uniform(np.log(1e-3), np.log(0.5), (B, L, D))))),
        Bm=r.standard_normal((B, L, N)),
        Cm=r.standard_normal((B, L, N)),
        A_log=r.uniform(-1.0, 1.5, (D, N)),
        Dskip=r.standard_normal(D),
        conv_w=r.uniform(-0.5, 0.5, (D, K)),
        conv_b=r.standard_normal(D) * 0.1,
    )
    if with_state:
        c["h0"] = r.standard_normal((B, D, N)) * 0.5
        c["conv_state0"] = r.standard_normal((B, K - 1, D))
    return c


def torch_u(c):
    """u = silu(conv1d(x)) with torch's conv1d in fp64: the K-1 earlier inputs
    (conv_state0, or zeros) are prepended and a valid convolution taken."""
    x = torch.from_numpy(c["x"])                      # (B,L,D)
    B, L, D = x.shape
    K = c["conv_w"].shape[1]
    prev = torch.from_numpy(c["conv_state0"]) if c.get("conv_state0") is not None \
        else torch.zeros(B, K - 1, D, dtype=torch.float64)
    xx = torch.cat([prev, x], dim=1).transpose(1, 2)  # (B,D,K-1+L)
    w = torch.from_numpy(c["conv_w"])[:, None, :]     # (D,1,K)
    bias = torch.from_numpy(c["conv_b"]) if c.get("conv_b") is not None else None
    pre = F.conv1d(xx, w, bias, groups=D)             # (B,D,L)
    return F.silu(pre).transpose(1, 2).numpy()


def torch_softplus(a):
    return F.softplus(torch.from_numpy(a)).numpy()   # beta=1, threshold=20


def torch_silu(a):
    return F.silu(torch.from_numpy(a)).numpy()


# Each pin_* function checks one fact against the oracle library `lib`
# (None: the real one).  The test_* wrappers run them on the real oracle;
# test_oracle_mutants.py runs them on mutated copies and expects failures.
LIB = {"lib": None}


def run(c, **kw):
    return oracle.scan(c["x"], c["z"], c["dt_raw"], c["Bm"], c["Cm"], c["A_log"],
                       c["Dskip"], c["conv_w"], c.get("conv_b"), c.get("h0"),
                       c.get("conv_state0"), lib=LIB["lib"], **kw)


def relerr(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


def brute_force(c):
    """y_t = silu(z_t) [ sum_n C_tn exp(A_n S_t) h0_n
                         + sum_{s<=t} sum_n C_tn exp(A_n (S_t - S_s)) dt_s B_sn u_s
                         + D u_t ],   S_t = dt_0 + ... + dt_t,  A = -exp(A_log)."""
    u = torch_u(c)
    dt = torch_softplus(c["dt_raw"])
    A = -np.exp(c["A_log"])                          # (D,N)
    B_, L, D = c["x"].shape
    N = A.shape[1]
    h0 = c.get("h0")
    y = np.zeros((B_, L, D))
    fh = np.zeros((B_, D, N))
    for b in range(B_):
        for ch in range(D):
            S = np.cumsum(dt[b, :, ch])
            for t in range(L):
                h = np.zeros(N)
                if h0 is not None:
                    h += np.exp(A[ch] * S[t]) * h0[b, ch]
                for s in range(t + 1):
                    h += np.exp(A[ch] * (S[t] - S[s])) * dt[b, s, ch] * c["Bm"][b, s] * u[b, s, ch]
                y[b, t, ch] = (c["Cm"][b, t] @ h + c["Dskip"][ch] * u[b, t, ch]) \
                    * torch_silu(np.array(c["z"][b, t, ch]))
                if t == L - 1:
                    fh[b, ch] = h
    return y, fh


def pin_brute_force_closed_form():
    for seed, kw in [(0, {}), (1, dict(B=1, L=20, D=2, N=16, K=4)), (2, dict(K=2, N=3)),
                     (3, dict(with_state=False))]:
        c = rand_case(seed=seed, **kw)
        y, fh, fcs = run(c)
        yb, fhb = brute_force(c)
        assert relerr(y, yb) < 1e-12
        assert relerr(fh, fhb) < 1e-12


def pin_final_conv_state_is_last_inputs():
    c = rand_case(L=12)
    _, _, fcs = run(c)
    np.testing.assert_array_equal(fcs, c["x"][:, -3:, :])
    # L shorter than K-1: older entries come from conv_state0
    c = rand_case(L=2, seed=5)
    _, _, fcs = run(c)
    np.testing.assert_array_equal(fcs[:, 0, :], c["conv_state0"][:, 2, :])
    np.testing.assert_array_equal(fcs[:, 1:, :], c["x"])


def pin_A_to_zero_is_cumsum():
    c = rand_case(seed=7, L=30)
    c["A_log"][:] = -np.inf          # A = -exp(-inf) = -0, dA = 1
    y, fh, _ = run(c)
    u = torch_u(c)
    dt = torch_softplus(c["dt_raw"])
    inc = dt[..., None] * c["Bm"][:, :, None, :] * u[..., None]   # (B,L,D,N)
    h = c["h0"][:, None] + np.cumsum(inc, axis=1)
    yr = (np.einsum("bln,bldn->bld", c["Cm"], h) + c["Dskip"] * u) * torch_silu(c["z"])
    assert relerr(y, yr) < 1e-12
    assert relerr(fh, h[:, -1]) < 1e-12


def pin_constant_dt_B_C_is_lti_convolution():
    r = np.random.default_rng(11)
    c = rand_case(seed=11, L=64, D=3, N=16, with_state=False)
    B_, L, D = c["x"].shape
    N = 16
    c["dt_raw"][:] = r.uniform(-4, -1, D)[None, None, :]
    c["Bm"][:] = r.standard_normal(N)
    c["Cm"][:] = r.standard_normal(N)
    c["A_log"] = np.log(np.arange(1, N + 1, dtype=np.float64))[None, :].repeat(D, 0)
    y, _, _ = run(c)
    u = torch_u(c)
    gate = torch_silu(c["z"])
    for b in range(B_):
        for ch in range(D):
            dt = torch_softplus(c["dt_raw"][0, 0, ch:ch + 1])[0]
            a = np.exp(dt * -np.exp(c["A_log"][ch]))
            k = np.arange(L)
            kern = (c["Cm"][0, 0] * dt * c["Bm"][0, 0] * a[None, :] ** k[:, None]).sum(1)
            conv = np.convolve(u[b, :, ch], kern)[:L]
            yr = (conv + c["Dskip"][ch] * u[b, :, ch]) * gate[b, :, ch]
            assert relerr(y[b, :, ch], yr) < 1e-11


def pin_A_to_minus_infinity_forgets():
    c = rand_case(seed=13, L=10)
    c["A_log"][:] = 60.0              # A = -e^60: dA underflows to exactly 0
    y, fh, _ = run(c)
    u = torch_u(c)
    dt = torch_softplus(c["dt_raw"])
    h = dt[..., None] * c["Bm"][:, :, None, :] * u[..., None]
    yr = (np.einsum("bln,bldn->bld", c["Cm"], h) + c["Dskip"] * u) * torch_silu(c["z"])
    assert relerr(y, yr) < 1e-13
    assert relerr(fh, h[:, -1]) < 1e-13


def pin_B_zero_decays_h0_and_skips():
    c = rand_case(seed=17, L=25)
    c["Bm"][:] = 0.0
    y, fh, _ = run(c)
    S = torch_softplus(c["dt_raw"]).sum(1)            # (B,D)
    A = -np.exp(c["A_log"])
    np.testing.assert_allclose(fh, c["h0"] * np.exp(A[None] * S[..., None]), rtol=1e-12)
    c["h0"] = None
    y, fh, _ = run(c)
    u = torch_u(c)
    assert relerr(y, c["Dskip"] * u * torch_silu(c["z"])) < 1e-14
    assert np.all(fh == 0.0)


def pin_conv_taps_bias_and_state_against_torch_conv1d():
    c = rand_case(seed=19, L=16, D=5, N=2)
    c["Cm"][:] = 0.0
    c["Dskip"][:] = 1.0
    c["z"][:] = 1.0
    y, _, _ = run(c)
    u = y / torch_silu(np.array(1.0))
    assert relerr(u, torch_u(c)) < 1e-14
    # identity taps, zero bias: u = silu(x), y = silu(x) silu(z)
    c = rand_case(seed=23, L=9, D=4, N=2)
    c["conv_w"][:] = [0.0, 0.0, 0.0, 1.0]
    c["conv_b"][:] = 0.0
    c["Cm"][:] = 0.0
    c["Dskip"][:] = 1.0
    y, _, _ = run(c)
    assert relerr(y, torch_silu(c["x"]) * torch_silu(c["z"])) < 1e-15


def pin_softplus_including_threshold():
    # N=1, dA=1, B=C=1, D=0, h0=0, identity taps: y_t = silu(z_t) sum_{s<=t} dt_s u_s
    c = rand_case(seed=29, B=1, L=40, D=2, N=1, with_state=False)
    c["dt_raw"][0, :, 0] = np.linspace(-30, 30, 40)
    c["dt_raw"][0, :, 1] = np.linspace(19.0, 21.0, 40)
    c["A_log"][:] = -np.inf
    c["Bm"][:] = 1.0
    c["Cm"][:] = 1.0
    c["Dskip"][:] = 0.0
    c["conv_w"][:] = [0, 0, 0, 1.0]
    c["conv_b"][:] = 0.0
    y, _, _ = run(c)
    u = torch_silu(c["x"])
    yr = np.cumsum(torch_softplus(c["dt_raw"]) * u, axis=1) * torch_silu(c["z"])
    assert relerr(y, yr) < 1e-13


def pin_zero_gate_and_zero_readout_are_exact_zero():
    c = rand_case(seed=31)
    c["z"][:] = 0.0
    y, _, _ = run(c)
    assert np.all(y == 0.0)
    c = rand_case(seed=32)
    c["Cm"][:] = 0.0
    c["Dskip"][:] = 0.0
    y, _, _ = run(c)
    assert np.all(y == 0.0)


def pin_chunked_equals_sequential(chunk=16):
    c = rand_case(seed=37, B=2, L=64, D=3, N=16)
    y, fh, fcs = run(c)
    yc, fhc, fcsc = oracle.scan_chunked(c["x"], c["z"], c["dt_raw"], c["Bm"], c["Cm"],
                                        c["A_log"], c["Dskip"], c["conv_w"], c["conv_b"],
                                        c["h0"], c["conv_state0"], chunk=chunk,
                                        lib=LIB["lib"])
    assert relerr(yc, y) < 1e-12
    assert relerr(fhc, fh) < 1e-12
    np.testing.assert_array_equal(fcsc, fcs)


def pin_decode_steps_equal_scan_bitwise():
    c = rand_case(seed=41, B=2, L=33, D=4, N=16)
    y, fh, fcs = run(c)
    h, s = c["h0"], c["conv_state0"]
    for t in range(c["x"].shape[1]):
        yt, h, s = oracle.step(h, s, c["x"][:, t], c["z"][:, t], c["dt_raw"][:, t],
                               c["Bm"][:, t], c["Cm"][:, t], c["A_log"], c["Dskip"],
                               c["conv_w"], c["conv_b"], lib=LIB["lib"])
        np.testing.assert_array_equal(yt, y[:, t])
    np.testing.assert_array_equal(h, fh)
    np.testing.assert_array_equal(s, fcs)


def pin_host_chunked_calls_with_carried_state_equal_one_call():
    c = rand_case(seed=43, B=1, L=48, D=3, N=16)
    y, fh, fcs = run(c)
    h, s = c["h0"], c["conv_state0"]
    ys = []
    for t0 in range(0, 48, 12):
        part = {k: (v[:, t0:t0 + 12] if k in ("x", "z", "dt_raw", "Bm", "Cm") else v)
                for k, v in c.items()}
        part["h0"], part["conv_state0"] = h, s
        yp, h, s = run(part)
        ys.append(yp)
    np.testing.assert_array_equal(np.concatenate(ys, 1), y)
    np.testing.assert_array_equal(h, fh)
    np.testing.assert_array_equal(s, fcs)


def pin_state_size_independent_of_L_and_memory_budget():
    g = json.load(open(os.path.join(GOLDEN, "memory_budget.json")))
    shapes = set()
    for L in (1, 3, 256, 2048):
        c = rand_case(seed=47, B=1, L=L, D=4, N=16)
        _, fh, fcs = run(c)
        shapes.add((fh.shape, fcs.shape))
    assert shapes == {((1, 4, 16), (1, 3, 4))}
    st = g["ssm_state"]
    # per layer and token-independent: hidden channels x state_size values
    assert st["layers"] * st["hidden"] * st["state_size"] * st["bytes_per_value"] == st["bytes"]
    assert round(st["bytes"] / 1e6, 1) == float(st["printed"].split()[0])
    ctx = g["context_tokens"]
    for key, (layers, heads) in {"kv_cache_hybrid_mha": (4, 32), "kv_cache_hybrid_gqa8": (4, 8),
                                 "kv_cache_transformer_mha": (32, 32),
                                 "kv_cache_transformer_gqa8": (32, 8)}.items():
        b = 2 * layers * heads * 128 * ctx * 2
        assert b == g[key]["bytes"]
        assert b // 2**30 == int(g[key]["printed"].split()[0])


def pin_oracle_threads_do_not_change_results():
    c = rand_case(seed=53, B=3, L=40, D=7, N=16)
    a = run(c, n_threads=1)
    b = run(c, n_threads=4)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


PINS = [pin_brute_force_closed_form, pin_final_conv_state_is_last_inputs,
        pin_A_to_zero_is_cumsum, pin_constant_dt_B_C_is_lti_convolution,
        pin_A_to_minus_infinity_forgets, pin_B_zero_decays_h0_and_skips,
        pin_conv_taps_bias_and_state_against_torch_conv1d,
        pin_softplus_including_threshold, pin_zero_gate_and_zero_readout_are_exact_zero,
        pin_chunked_equals_sequential, pin_decode_steps_equal_scan_bitwise,
        pin_host_chunked_calls_with_carried_state_equal_one_call,
        pin_state_size_independent_of_L_and_memory_budget,
        pin_oracle_threads_do_not_change_results]


@pytest.mark.parametrize("pin", [p for p in PINS if p is not pin_chunked_equals_sequential],
                         ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


@pytest.mark.parametrize("chunk", [1, 5, 16, 37, 64, 100])
def test_chunked_equals_sequential(chunk):
    pin_chunked_equals_sequential(chunk)



@settings(max_examples=60, deadline=None, derandomize=True)
@given(st.integers(1, 2), st.integers(1, 20), st.integers(1, 3), st.integers(1, 16), st.integers(2, 4),
       st.booleans(), st.booleans(), st.integers(0, 2 ** 31 - 1))
def test_brute_force_closed_form_over_shapes(B, L, D, N, K, with_state, with_bias, seed):
    """The closed form of the recurrence on random small shapes: every
    sequence length from 1 (conv state only), every state and conv width the
    oracle accepts, with and without initial states and conv bias."""
    c = rand_case(B=B, L=L, D=D, N=N, K=K, seed=seed, with_state=with_state)
    if not with_bias:
        c["conv_b"] = None
    y, fh, fcs = run(c)
    yb, fhb = brute_force(c)
    assert relerr(y, yb) < 1e-11
    assert relerr(fh, fhb) < 1e-11
    prev = c["conv_state0"] if with_state else np.zeros((B, K - 1, D))
    np.testing.assert_array_equal(fcs, np.concatenate([prev, c["x"]], axis=1)[:, -(K - 1):])
