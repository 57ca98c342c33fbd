"""The complex-valued scan (mamba3_scan_fwd: Mamba-3's state update, Euler and
exponential-trapezoidal) on the GPU through the C ABI, against the fp64
complex-scan oracle (mamba3_oracle.c).  Tolerances as for the real scan
(parity.py): max|gpu - oracle| / rms(oracle) <= 1e-4 for fp32 I/O, <= 1e-2
for bf16 I/O after each bf16 output's half-ulp allowance; the final conv
state is a copy and must be exact."""
import math

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, io_name, sample_channels
from selective_state_space_118_b300 import inputs, ops

pytestmark = pytest.mark.gpu

RULES = {"euler": False, "trapezoidal": True}


def run_gpu(inp, trap, **kw):
    return ops.mamba3_scan_fwd(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"],
                               inp["theta"], inp["Dskip"], inp["conv_w"], inp.get("conv_b"), inp.get("h0"),
                               inp.get("conv_state0"), inp.get("v0"), trapezoidal=trap, **kw)


def oracle_run(inp, trap, channels=None):
    cs = slice(None) if channels is None else channels

    def ch(t, axis):
        if t is None:
            return None
        a = oracle.f64(t)
        return np.take(a, np.arange(a.shape[axis])[cs], axis=axis)

    return oracle.m3_scan(ch(inp["x"], 2), ch(inp["z"], 2), ch(inp["dt_raw"], 2), oracle.f64(inp["Bm"]),
                          oracle.f64(inp["Cm"]), ch(inp["A_log"], 0), ch(inp["theta"], 0), ch(inp["Dskip"], 0),
                          ch(inp["conv_w"], 0), ch(inp.get("conv_b"), 0), ch(inp.get("h0"), 1),
                          ch(inp.get("conv_state0"), 2), ch(inp.get("v0"), 1), trapezoidal=trap)


def check(inp, outs, trap, what, channels=None):
    y, fh, fcs, fv = outs
    torch.cuda.synchronize()
    if channels is not None:
        idx = torch.as_tensor(channels, device=y.device)
        y, fh, fcs, fv = y.index_select(2, idx), fh.index_select(1, idx), fcs.index_select(2, idx), \
            fv.index_select(1, idx)
    yr, fhr, fcsr, fvr = oracle_run(inp, trap, channels)
    io = io_name(inp["x"])
    assert_close(y, yr, io, f"{what} y")
    assert_close(fh, fhr, io, f"{what} final_h", fp32_output=True)
    assert_close(fv, fvr, io, f"{what} final_v", fp32_output=True)
    np.testing.assert_array_equal(fcs.double().cpu().numpy(), fcsr)


def make(B, L, D, io, seed, with_state=True, v0=True, conv_b=True, bc_std=1.0):
    inp = inputs.complex_scan_inputs(B, L, D, io, seed=seed, bc_std=bc_std, device="cuda", with_state=with_state)
    g = torch.Generator(device="cuda").manual_seed(seed + 7)
    if with_state and v0:
        inp["v0"] = torch.randn(B, D, 16, device="cuda", generator=g)
    inp["conv_b"] = (torch.randn(D, device="cuda", generator=g) * 0.1) if conv_b else None
    return inp


EDGE = [
    # (B, L, D, io, with_state, n_chunks)
    (1, 1, 16, "f32", False, 1),
    (1, 2, 16, "bf16", True, 1),
    (2, 3, 32, "f32", True, 1),
    (1, 5, 16, "bf16", False, 1),
    (3, 63, 48, "f32", True, 1),
    (2, 65, 32, "bf16", True, 1),
    (1, 130, 16, "f32", True, 1),
    (2, 257, 48, "bf16", True, 2),
    (1, 337, 16, "f32", True, 3),
    (2, 337, 32, "bf16", True, 5),
    (3, 1000, 64, "f32", True, 7),
    (1, 4096, 32, "bf16", True, 0),
    # widths that are not multiples of 16
    (2, 300, 40, "bf16", True, 1),
    (1, 337, 36, "f32", True, 3),
]


@pytest.mark.parametrize("rule", sorted(RULES))
@pytest.mark.parametrize("B,L,D,io,with_state,n_chunks", EDGE)
def test_against_oracle(rule, B, L, D, io, with_state, n_chunks):
    inp = make(B, L, D, io, seed=500 + L + D, with_state=with_state)
    check(inp, run_gpu(inp, RULES[rule], n_chunks=n_chunks), RULES[rule], f"{rule} B{B} L{L} D{D} {io} nc{n_chunks}")


@pytest.mark.parametrize("rule", sorted(RULES))
def test_wide_softplus_range(rule):
    """dt_raw across [-30, 30]: softplus's three regions, in tiles wholly in
    one region and tiles that mix them."""
    B, L, D = 2, 600, 32
    inp = make(B, L, D, "f32", seed=601)
    inp["dt_raw"] = inputs.wide_dt_raw(B, L, D, "f32", seed=602, device="cuda")
    check(inp, run_gpu(inp, RULES[rule], n_chunks=3), RULES[rule], f"{rule} wide dt")


@pytest.mark.parametrize("rule", sorted(RULES))
def test_fast_turns(rule):
    """Rotation frequencies up to +-40 with dt log-uniform in [1e-2, 1]: up to
    40 radians (several whole turns) per token, reduced to [-pi, pi] before
    the sine and cosine.  (The angle dt theta carries dt's fp32 rounding, a
    few 1e-8 of it: turns of thousands of radians per token are beyond the
    fp32 bound.)"""
    B, L, D = 2, 600, 32
    inp = make(B, L, D, "f32", seed=611)
    g = torch.Generator(device="cuda").manual_seed(612)
    inp["theta"] = (torch.rand(D, 8, device="cuda", generator=g) - 0.5) * 80.0
    dt = torch.exp(math.log(1e-2) + torch.rand(B, L, D, device="cuda", generator=g) * math.log(100.0))
    inp["dt_raw"] = torch.log(torch.expm1(dt))
    check(inp, run_gpu(inp, RULES[rule], n_chunks=3), RULES[rule], f"{rule} fast turns")


@pytest.mark.parametrize("rule", sorted(RULES))
def test_fast_turns_in_small_dt_tiles(rule):
    """dt log-uniform in [1e-3, 1e-1] (every tile in softplus's small region,
    so the tokens go two at a time) with rotation frequencies up to +-200:
    a token takes its angle dt theta directly only when dt <= pi / max|theta|
    of its channel, so within one warp and one token pair some lanes take
    the angle directly and others reduce whole turns (up to 20 radians per
    token).  Chunked, so the carry walks take both paths too."""
    B, L, D = 2, 700, 64
    inp = make(B, L, D, "f32", seed=621)
    g = torch.Generator(device="cuda").manual_seed(622)
    inp["theta"] = (torch.rand(D, 8, device="cuda", generator=g) - 0.5) * 400.0
    inp["theta"][::4] *= 0.05  # a quarter of the channels turn slowly: every token direct
    dt = torch.exp(math.log(1e-3) + torch.rand(B, L, D, device="cuda", generator=g) * math.log(100.0))
    inp["dt_raw"] = torch.log(torch.expm1(dt))
    assert float(inp["dt_raw"].max()) < -2.08  # softplus's small region: token pairs
    check(inp, run_gpu(inp, RULES[rule], n_chunks=3), RULES[rule], f"{rule} fast turns, small dt")


@pytest.mark.parametrize("rule", sorted(RULES))
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_split_calls_equal_one_call_bitwise(rule, io):
    """One pass == the same sequence fed as calls that carry (final_h,
    final_conv_state, final_v) into (h0, conv_state0, v0), bit for bit."""
    inp = make(1, 1024, 64, io, seed=611)
    y, fh, fcs, fv = [t.clone() for t in run_gpu(inp, RULES[rule], n_chunks=1)]
    h, cs, v, ys = inp["h0"], inp["conv_state0"], inp["v0"], []
    for t0, t1 in [(0, 64), (64, 65), (65, 300), (300, 1024)]:
        part = dict(inp, h0=h, conv_state0=cs, v0=v)
        for k in ("x", "z", "dt_raw", "Bm", "Cm"):
            part[k] = inp[k][:, t0:t1].contiguous()
        yp, h, cs, v = run_gpu(part, RULES[rule], n_chunks=1)
        ys.append(yp)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(ys, 1), y)
    assert torch.equal(h, fh) and torch.equal(cs, fcs) and torch.equal(v, fv)


@pytest.mark.parametrize("rule", sorted(RULES))
@pytest.mark.parametrize("n_chunks", [1, 3, 7])
def test_final_states_may_alias_initial_states(rule, n_chunks):
    """final_h, final_conv_state and final_v given the buffers of h0,
    conv_state0 and v0 (the header allows it): the same bits as with separate
    buffers, one pass and chunked."""
    inp = make(2, 300, 64, "bf16", seed=631)
    ref = [t.clone() for t in run_gpu(inp, RULES[rule], n_chunks=n_chunks)]
    h, cs, v = inp["h0"].clone(), inp["conv_state0"].clone(), inp["v0"].clone()
    out = run_gpu(dict(inp, h0=h, conv_state0=cs, v0=v), RULES[rule], final_h=h, final_conv_state=cs, final_v=v,
                  n_chunks=n_chunks)
    torch.cuda.synchronize()
    assert torch.equal(out[0], ref[0])
    assert torch.equal(h, ref[1]) and torch.equal(cs, ref[2]) and torch.equal(v, ref[3])


@pytest.mark.parametrize("rule", sorted(RULES))
def test_exact_carry_flag_against_oracle(rule):
    """MAMBA_FLAG_EXACT_CARRY: every chunk summarised and folded, nothing
    dropped (three launches) -- against the oracle, and against the default
    walked carries, which stop after ~1,100 tokens of these 2,048-token chunks
    (the slowest mode's decay passes 2^-32) and drop what lies before."""
    inp = make(1, 8192, 32, "f32", seed=651)
    exact = [t.clone() for t in run_gpu(inp, RULES[rule], n_chunks=4, flags=ops.MAMBA_FLAG_EXACT_CARRY)]
    check(inp, exact, RULES[rule], f"{rule} exact carries")
    walked = run_gpu(inp, RULES[rule], n_chunks=4)
    torch.cuda.synchronize()
    assert_close(walked[0], exact[0].double().cpu().numpy(), "f32", "walked vs exact y")
    assert_close(walked[1], exact[1].double().cpu().numpy(), "f32", "walked vs exact h", fp32_output=True)
    assert torch.equal(walked[2], exact[2]) and torch.equal(walked[3], exact[3])


@pytest.mark.parametrize("rule", sorted(RULES))
def test_chunked_equals_one_pass_within_tolerance(rule):
    inp = make(1, 64 * 40 + 7, 32, "f32", seed=621)
    y1, fh1, fcs1, fv1 = [t.clone() for t in run_gpu(inp, RULES[rule], n_chunks=1)]
    for nc in (2, 7, 40):
        y, fh, fcs, fv = run_gpu(inp, RULES[rule], n_chunks=nc)
        torch.cuda.synchronize()
        assert_close(y, y1.double().cpu().numpy(), "f32", f"nc={nc} y")
        assert_close(fh, fh1.double().cpu().numpy(), "f32", f"nc={nc} h", fp32_output=True)
        assert torch.equal(fcs, fcs1) and torch.equal(fv, fv1)


def test_seqlen_zero_returns_initial_state():
    inp = make(2, 0, 32, "bf16", seed=631)
    y, fh, fcs, fv = run_gpu(inp, True)
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert torch.equal(fh, inp["h0"]) and torch.equal(fv, inp["v0"]) and torch.equal(fcs, inp["conv_state0"])


def test_rejects_bad_arguments_on_device():
    inp = make(1, 64, 32, "bf16", seed=641)
    with pytest.raises(ops.MambaError) as e:
        run_gpu(inp, False, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == ops.MAMBA_ERR_WORKSPACE


@pytest.mark.parametrize("rule", sorted(RULES))
def test_full_size_sampled_channels(rule):
    """The Jamba-shaped workload (1 x 32768 tokens x 8192 channels, bf16,
    B, C ~ N(0, 1/16)), the default plan: sampled channels against the
    oracle (channels are independent; B and C rows are per token)."""
    w = inputs.JAMBA_PREFILL
    inp = inputs.complex_scan_inputs(w.batch, w.seqlen, w.d_inner, w.io, w.seed, w.bc_std, device="cuda")
    outs = run_gpu(inp, RULES[rule])
    plan_chunks = ops.mamba3_scan_workspace_size(1, w.seqlen, w.d_inner, 0) > \
        ops.mamba3_scan_workspace_size(1, w.seqlen, w.d_inner, 1)
    assert plan_chunks  # the default plan is chunked at batch 1
    check(inp, outs, RULES[rule], f"{rule} full size", channels=sample_channels(w.d_inner, 24))
