"""Backward of the prefill scan on the GPU (through the C ABI) against the
fp64 backward oracle.

Tolerance: the forward's bounds (parity.py: max error / rms of the oracle,
1e-4 for fp32 I/O, 1e-2 for bf16 I/O, bf16 outputs first allowed their own
rounding).  The per-token gradients (dx, dz, ddt_raw) and the state
gradients (dh0, dconv_state0) are measured channel by channel: channels are
independent recurrences whose gradients can differ in scale by large
factors (a slowly decaying channel accumulates a larger state and adjoint),
and a channel's rounding error scales with its own magnitude, so against
the rms of the whole tensor one large channel among small ones would look
worse than it is and a small channel's errors would be drowned.  Each
channel's rms is floored at 1e-3 of the tensor's.  The parameter gradients
(one sum over all tokens per element, which may cancel to near zero) and dB,
dC (sums over all channels) are measured against the whole tensor.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import BF16_HALF_ULP, TOL, assert_close, io_name, sample_channels
from selective_state_space_118_b300 import inputs, ops

pytestmark = pytest.mark.gpu

# C-ABI output name -> oracle name
NAMES = {"dx": "dx", "dz": "dz", "ddt_raw": "ddt_raw", "dB": "dB", "dC": "dC", "dA_log": "dA_log",
         "dDskip": "dD", "dconv_w": "dconv_w", "dconv_b": "dconv_b", "dh0": "dh0",
         "dconv_state0": "dconv_state0"}
IO_OUTPUTS = ("dx", "dz", "ddt_raw")
CHANNEL_AXIS = {"dx": 2, "dz": 2, "ddt_raw": 2, "dh0": 1, "dconv_state0": 2}
PARAM_AXIS = {"dA_log": 0, "dDskip": 0, "dconv_w": 0, "dconv_b": 0}


def assert_close_per_channel(gpu, ref, axis, io, what, rounded_bf16):
    """max over channels of (max |gpu - oracle| / rms of the oracle) within the
    channel, the rms floored at 1e-3 of the tensor's; bf16 outputs first get
    their half-ulp allowance, as in parity.py."""
    g = oracle.f64(gpu)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = np.abs(g - ref)
    if rounded_bf16:
        err = np.maximum(err - BF16_HALF_ULP * np.abs(ref), 0.0)
    if err.size == 0:
        return 0.0
    err = np.moveaxis(err, axis, 0).reshape(ref.shape[axis], -1)
    r = np.moveaxis(ref, axis, 0).reshape(ref.shape[axis], -1)
    rms_all = float(np.sqrt(np.mean(ref * ref))) or 1.0
    rms = np.maximum(np.sqrt(np.mean(r * r, axis=1)), 1e-3 * rms_all)
    worst = float(np.max(err.max(axis=1) / rms))
    assert worst <= TOL[io], f"{what}: per-channel error {worst:.3e} > {TOL[io]:g}"
    return worst


def make_case(B, L, D, io, seed, with_state=True, conv_b=True, dfinal=True, bc_std=1.0):
    inp = inputs.scan_inputs(B, L, D, io, seed=seed, bc_std=bc_std, device="cuda", with_state=with_state)
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    dt = inputs.torch_dtype(io)
    inp["conv_b"] = (torch.randn(D, device="cuda", generator=g) * 0.1) if conv_b else None
    inp["dy"] = torch.randn(B, L, D, device="cuda", generator=g).to(dt)
    if dfinal:
        inp["dfinal_h"] = torch.randn(B, D, 16, device="cuda", generator=g)
        inp["dfinal_conv_state"] = torch.randn(B, 3, D, device="cuda", generator=g).to(dt)
    return inp


def run_gpu(inp, **kw):
    return ops.mamba_scan_bwd(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"],
                              inp["Dskip"], inp["conv_w"], inp.get("conv_b"), inp.get("h0"),
                              inp.get("conv_state0"), dy=inp["dy"], dfinal_h=inp.get("dfinal_h"),
                              dfinal_conv_state=inp.get("dfinal_conv_state"), **kw)


def oracle_bwd(inp, channels=None):
    cs = slice(None) if channels is None else channels

    def ch(t, axis):
        if t is None:
            return None
        a = oracle.f64(t)
        return np.take(a, np.arange(a.shape[axis])[cs], axis=axis)

    return oracle.scan_bwd(ch(inp["x"], 2), ch(inp["z"], 2), ch(inp["dt_raw"], 2),
                           oracle.f64(inp["Bm"]), oracle.f64(inp["Cm"]), ch(inp["A_log"], 0),
                           ch(inp["Dskip"], 0), ch(inp["conv_w"], 0), ch(inp.get("conv_b"), 0),
                           ch(inp.get("h0"), 1), ch(inp.get("conv_state0"), 2), dy=ch(inp["dy"], 2),
                           dfinal_h=ch(inp.get("dfinal_h"), 1),
                           dfinal_conv_state=ch(inp.get("dfinal_conv_state"), 2))


def check(inp, g, what, channels=None, skip=()):
    torch.cuda.synchronize()
    ref = oracle_bwd(inp, channels)
    io = io_name(inp["x"])
    worst = {}
    for k, rk in NAMES.items():
        if k in skip or g.get(k) is None:
            continue
        t = g[k]
        axis = CHANNEL_AXIS.get(k, PARAM_AXIS.get(k))
        if channels is not None and axis is not None:
            t = torch.index_select(t, axis, torch.as_tensor(channels, device=t.device))
        if k in CHANNEL_AXIS:
            worst[k] = assert_close_per_channel(t, ref[rk], axis, io, f"{what} {k}",
                                                rounded_bf16=io == "bf16" and k in IO_OUTPUTS)
        else:
            worst[k] = assert_close(t, ref[rk], io, f"{what} {k}", fp32_output=True)[1]
    return worst


CASES = [
    # (B, L, D, io, with_state, conv_b, dfinal, n_chunks)
    (1, 1, 16, "f32", False, True, True, 1),
    (1, 2, 16, "f32", True, True, True, 1),
    (2, 3, 32, "bf16", True, False, True, 1),
    (1, 5, 16, "f32", True, True, False, 1),
    (2, 16, 32, "f32", True, True, True, 1),
    (1, 17, 48, "f32", True, True, True, 1),
    (2, 65, 32, "bf16", True, False, True, 1),
    (3, 130, 48, "f32", True, True, True, 1),
    (1, 337, 16, "f32", True, True, True, 2),
    (2, 337, 32, "bf16", True, True, True, 3),
    (1, 337, 48, "f32", False, False, False, 6),
    (1, 49, 16, "f32", True, True, True, 3),
    (3, 1000, 64, "f32", True, True, True, 5),
    (1, 4096, 32, "bf16", True, True, True, 0),
    # widths that are not multiples of 16
    (2, 300, 40, "bf16", True, True, True, 1),
    (1, 337, 40, "bf16", True, True, True, 3),
    (1, 300, 36, "f32", True, True, True, 1),
    (2, 337, 36, "f32", True, False, True, 4),
]


@pytest.mark.parametrize("B,L,D,io,with_state,conv_b,dfinal,n_chunks", CASES)
def test_bwd_against_oracle(B, L, D, io, with_state, conv_b, dfinal, n_chunks):
    inp = make_case(B, L, D, io, seed=300 + L + D, with_state=with_state, conv_b=conv_b, dfinal=dfinal)
    g = run_gpu(inp, n_chunks=n_chunks)
    check(inp, g, f"B{B} L{L} D{D} {io} nc{n_chunks}")


@pytest.mark.parametrize("case", ["fast_decay", "slow_decay", "mixed"])
def test_bwd_adjoint_carries(case):
    """The adjoint-carry walk: with fast decay it stops after a few pieces,
    with slow decay every boundary chains onto the next one, a warp mixing
    both follows its slowest channel."""
    B, L, D = 1, 8192, 64
    inp = make_case(B, L, D, "f32", seed=41)
    if case == "slow_decay":
        inp["A_log"] = torch.full_like(inp["A_log"], -1.5)
    elif case == "mixed":
        inp["A_log"][5] = -1.5
        inp["A_log"][40, :4] = -1.0
    plan = ops.mamba_scan_plan(B, L, D, 4)
    assert plan["n_chunks"] == 4 and plan["pieces"] > 1
    g = run_gpu(inp, n_chunks=4)
    check(inp, g, f"adjoint carries {case}")
    g1 = run_gpu(inp, n_chunks=1)
    torch.cuda.synchronize()
    for k in ("dh0", "dA_log", "dB"):
        assert_close(g[k], g1[k].double().cpu().numpy(), "f32", f"{case}: chunked vs one pass {k}",
                     fp32_output=True)


def test_bwd_deterministic():
    inp = make_case(1, 2000, 64, "bf16", seed=43)
    a = run_gpu(inp, n_chunks=4)
    a = {k: (v.clone() if v is not None else None) for k, v in a.items()}
    b = run_gpu(inp, n_chunks=4)
    torch.cuda.synchronize()
    for k in ops.BWD_OUTPUTS:
        if a[k] is not None:
            assert torch.equal(a[k], b[k]), k


def test_bwd_seqlen_zero():
    inp = make_case(2, 0, 32, "bf16", seed=45)
    g = run_gpu(inp)
    torch.cuda.synchronize()
    assert torch.equal(g["dh0"], inp["dfinal_h"])
    assert torch.equal(g["dconv_state0"], inp["dfinal_conv_state"].float())
    for k in ("dA_log", "dDskip", "dconv_w", "dconv_b"):
        assert torch.all(g[k] == 0), k


def test_bwd_rejects_bad_arguments():
    inp = make_case(1, 64, 20, "bf16", seed=47)  # bf16 rows of 40 bytes
    with pytest.raises(ops.MambaError) as e:
        run_gpu(inp)
    assert e.value.status == ops.MAMBA_ERR_UNSUPPORTED
    inp = make_case(1, 4096, 16, "bf16", seed=47)
    with pytest.raises(ops.MambaError) as e:
        run_gpu(inp, n_chunks=4, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == ops.MAMBA_ERR_WORKSPACE


def test_bwd_fullsize_sampled_channels():
    """The benchmark's shape (1 x 32768 tokens x 8192 channels, bf16, the
    default plan): every per-channel gradient on sampled channels (the oracle
    runs on those channels alone; channels are independent except through dB
    and dC, which sum over all of them and are checked at smaller sizes)."""
    w = inputs.JAMBA_PREFILL
    inp = inputs.workload_inputs(w, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(49)
    inp["dy"] = torch.randn(inp["x"].shape, device="cuda", generator=g).to(inp["x"].dtype)
    out = run_gpu(inp)
    chans = sample_channels(w.d_inner, 12)
    check(inp, out, "full size", channels=chans, skip=("dB", "dC", "dconv_b"))


@pytest.mark.parametrize("io,n_chunks", [("bf16", 0), ("f32", 1), ("bf16", 4)])
def test_bwd_from_forward_tile_states_is_bitwise_the_same(io, n_chunks):
    """A forward call that stores the tile states, then a backward given them
    (no recomputation), equals a backward that recomputes them, bit for bit:
    both passes compute the states with the same operations."""
    inp = make_case(2, 700, 48, io, seed=51)
    B, L, D = inp["x"].shape
    ts = torch.empty(ops.tile_states_shape(B, L, D), device="cuda")
    ops.mamba_scan_fwd(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"], inp["Dskip"],
                       inp["conv_w"], inp["conv_b"], inp["h0"], inp["conv_state0"], n_chunks=n_chunks,
                       tile_states=ts)
    a = run_gpu(inp, n_chunks=n_chunks)
    a = {k: (v.clone() if v is not None else None) for k, v in a.items()}
    b = run_gpu(inp, n_chunks=n_chunks, tile_states=ts)
    torch.cuda.synchronize()
    for k in ops.BWD_OUTPUTS:
        if a[k] is not None:
            assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("io,n_chunks", [("f32", 1), ("f32", 3), ("bf16", 3)])
def test_bwd_softplus_regions(io, n_chunks):
    """dt_raw across [-30, 30]: the softplus derivative (sigmoid below the
    threshold, 1 above it) and the three regions of softplus itself, in
    the recomputed forward, the adjoint walk and the reverse sweep."""
    B, L, D = 2, 700, 48
    inp = make_case(B, L, D, io, seed=97)
    inp["dt_raw"] = inputs.wide_dt_raw(B, L, D, io, seed=98, device="cuda")
    g = run_gpu(inp, n_chunks=n_chunks)
    check(inp, g, f"wide dt {io} nc{n_chunks}")


def test_bwd_exact_carry_flag():
    """MAMBA_FLAG_EXACT_CARRY in the backward: both carry walks cover whole
    chunks; the gradients match the oracle and the one-pass backward."""
    B, L, D = 1, 8192, 32
    inp = make_case(B, L, D, "f32", seed=99)
    g = run_gpu(inp, n_chunks=4, flags=ops.MAMBA_FLAG_EXACT_CARRY)
    check(inp, g, "exact carries")
    g1 = run_gpu(inp, n_chunks=1)
    torch.cuda.synchronize()
    for k in ("dh0", "dA_log", "dB", "dx"):
        assert_close(g[k], g1[k].double().cpu().numpy(), "f32", f"exact chunked vs one pass {k}",
                     fp32_output=True)
