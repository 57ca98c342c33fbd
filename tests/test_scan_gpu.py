"""Prefill scan on the GPU (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from parity import assert_close, io_name, oracle_scan, to_device
from selective_state_space_118_b300 import inputs, ops

pytestmark = pytest.mark.gpu


def run_gpu(inp, **kw):
    return ops.mamba_scan_fwd(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"],
                              inp["A_log"], inp["Dskip"], inp["conv_w"], inp.get("conv_b"),
                              inp.get("h0"), inp.get("conv_state0"), **kw)


def check_against_oracle(inp, outs, what=""):
    y, fh, fcs = outs
    torch.cuda.synchronize()
    yr, fhr, fcsr = oracle_scan(inp)
    io = io_name(inp["x"])
    assert_close(y, yr, io, f"{what} y")
    assert_close(fh, fhr, io, f"{what} final_h", fp32_output=True)
    np.testing.assert_array_equal(fcs.double().cpu().numpy(), fcsr)


def test_tiny_f32_workload():
    w = inputs.TINY_F32
    inp = inputs.workload_inputs(w, device="cuda")
    check_against_oracle(inp, run_gpu(inp), w.name)


@pytest.mark.parametrize("n_chunks", [0, 1, 4])
def test_small_bf16_workload(n_chunks):
    w = inputs.SMALL_BF16
    inp = inputs.workload_inputs(w, device="cuda")
    check_against_oracle(inp, run_gpu(inp, n_chunks=n_chunks), f"{w.name} n_chunks={n_chunks}")


EDGE = [
    # (B, L, D, io, with_state, conv_b, n_chunks)
    (1, 1, 16, "f32", False, True, 1),
    (1, 2, 16, "bf16", True, True, 1),
    (2, 3, 32, "f32", True, False, 1),
    (1, 5, 16, "bf16", False, True, 1),
    (3, 63, 48, "f32", True, True, 1),
    (1, 64, 16, "bf16", True, True, 1),
    (2, 65, 32, "bf16", True, False, 1),
    (1, 130, 16, "f32", True, True, 1),
    (2, 257, 48, "bf16", True, True, 1),
    (1, 337, 16, "f32", True, True, 2),
    (2, 337, 32, "bf16", True, True, 3),
    (1, 337, 16, "bf16", False, False, 6),
    (3, 1000, 64, "f32", True, True, 5),
    (1, 4096, 16, "bf16", True, True, 0),
    # widths that are not multiples of 16: a last group of 8 (bf16) or 4 (fp32) channels
    (2, 300, 40, "bf16", True, True, 1),
    (2, 300, 40, "bf16", True, True, 3),
    (1, 300, 36, "f32", True, True, 1),
    (1, 337, 36, "f32", True, False, 4),
    (2, 130, 8, "bf16", True, True, 2),
    (1, 65, 4, "f32", True, True, 1),
]


@pytest.mark.parametrize("B,L,D,io,with_state,conv_b,n_chunks", EDGE)
def test_edge_shapes(B, L, D, io, with_state, conv_b, n_chunks):
    inp = inputs.scan_inputs(B, L, D, io, seed=100 + L + D, bc_std=1.0, device="cuda",
                             with_state=with_state)
    if not conv_b:
        inp["conv_b"] = None
    else:
        inp["conv_b"] = torch.randn(D, device="cuda") * 0.1
    check_against_oracle(inp, run_gpu(inp, n_chunks=n_chunks), f"B{B} L{L} D{D} {io} nc{n_chunks}")


def test_seqlen_zero_returns_initial_state():
    inp = inputs.scan_inputs(2, 0, 32, "bf16", seed=5, device="cuda", with_state=True)
    y, fh, fcs = run_gpu(inp)
    torch.cuda.synchronize()
    assert y.numel() == 0
    assert torch.equal(fh, inp["h0"])
    assert torch.equal(fcs, inp["conv_state0"])
    del inp["h0"], inp["conv_state0"]
    y, fh, fcs = run_gpu(inp)
    torch.cuda.synchronize()
    assert torch.all(fh == 0) and torch.all(fcs == 0)


@pytest.mark.parametrize("L,n_chunks", [(300, 1), (300, 3), (1000, 9), (4096, 4)])
def test_final_state_may_alias_initial_state(L, n_chunks):
    """final_h and final_conv_state given the buffers of h0 and conv_state0:
    the same bits as with separate buffers.  In the chunked launch chunk 0's
    main warp and boundary 1's carry walk read h0 and conv_state0 while the
    last chunk runs (walks of several pieces; at L = 4096 the walks stop
    early on the decay)."""
    inp = inputs.scan_inputs(2, L, 32, "bf16", seed=7, device="cuda", with_state=True)
    ref = [t.clone() for t in run_gpu(inp, n_chunks=n_chunks)]
    h, cs = inp["h0"].clone(), inp["conv_state0"].clone()
    inp2 = dict(inp, h0=h, conv_state0=cs)
    y, fh, fcs = run_gpu(inp2, final_h=h, final_conv_state=cs, n_chunks=n_chunks)
    torch.cuda.synchronize()
    assert torch.equal(y, ref[0]) and torch.equal(h, ref[1]) and torch.equal(cs, ref[2])


def test_carried_calls_in_place_equal_separate_buffers():
    """A sequence fed as chunked calls back to back (their launches overlap
    the previous call's end), each call's final_h and final_conv_state
    written over its own h0 and conv_state0 in place, as a serving loop
    does: the same bits as with fresh buffers for every call."""
    B, L, D, calls = 1, 16384, 256, 4
    inp = inputs.scan_inputs(B, L, D, "bf16", seed=29, device="cuda", with_state=True)
    step = L // calls

    def part(i, h, cs):
        q = dict(inp, h0=h, conv_state0=cs)
        for k in ("x", "z", "dt_raw", "Bm", "Cm"):
            q[k] = inp[k][:, i * step:(i + 1) * step]
        return q

    ys, h, cs = [], inp["h0"].clone(), inp["conv_state0"].clone()
    for i in range(calls):
        y, h, cs = run_gpu(part(i, h, cs), n_chunks=0)
        ys.append(y)
    h_in, cs_in = inp["h0"].clone(), inp["conv_state0"].clone()
    ys_in = [run_gpu(part(i, h_in, cs_in), final_h=h_in, final_conv_state=cs_in, n_chunks=0)[0]
             for i in range(calls)]
    torch.cuda.synchronize()
    assert ops.mamba_scan_plan(B, step, D, 0)["n_chunks"] > 1
    assert all(torch.equal(a, b) for a, b in zip(ys, ys_in))
    assert torch.equal(h_in, h) and torch.equal(cs_in, cs)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_host_split_calls_equal_one_call_bitwise(io):
    """One sequential pass == the same sequence fed as several calls that carry
    (final_h, final_conv_state) into (h0, conv_state0) -- bit for bit."""
    inp = inputs.scan_inputs(1, 1024, 64, io, seed=11, device="cuda", with_state=True)
    y, fh, fcs = run_gpu(inp, n_chunks=1)
    h, cs, ys = inp["h0"], inp["conv_state0"], []
    for t0, t1 in [(0, 64), (64, 65), (65, 300), (300, 1024)]:
        part = dict(inp, h0=h, conv_state0=cs)
        for k in ("x", "z", "dt_raw", "Bm", "Cm"):
            part[k] = inp[k][:, t0:t1].contiguous()
        yp, h, cs = run_gpu(part, n_chunks=1)
        ys.append(yp)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat(ys, 1), y)
    assert torch.equal(h, fh) and torch.equal(cs, fcs)


def test_chunked_matches_sequential_within_tolerance():
    inp = inputs.scan_inputs(1, 64 * 40 + 7, 32, "f32", seed=13, device="cuda", with_state=True)
    y1, fh1, fcs1 = [t.clone() for t in run_gpu(inp, n_chunks=1)]
    for nc in (2, 7, 40):
        y, fh, fcs = run_gpu(inp, n_chunks=nc)
        torch.cuda.synchronize()
        assert_close(y, oracle_like(y1), "f32", f"nc={nc} y")
        assert_close(fh, oracle_like(fh1), "f32", f"nc={nc} h", fp32_output=True)
        assert torch.equal(fcs, fcs1)


def oracle_like(t):
    return t.double().cpu().numpy()


def test_timeout_is_reported_and_gpu_stays_usable():
    inp = inputs.scan_inputs(1, 256, 16, "bf16", seed=17, device="cuda")
    assert ops.mamba_last_error() == ops.MAMBA_OK
    run_gpu(inp, flags=ops.MAMBA_FLAG_TEST_STALL_FIRST_LOAD, wait_timeout_ns=20_000_000)
    assert ops.mamba_last_error() == ops.MAMBA_ERR_TIMEOUT
    assert ops.mamba_last_error() == ops.MAMBA_OK  # cleared by the read
    check_against_oracle(inp, run_gpu(inp), "after timeout")
    assert ops.mamba_last_error() == ops.MAMBA_OK


def test_rejects_bad_arguments_on_device():
    inp = inputs.scan_inputs(1, 64, 20, "bf16", seed=19, device="cuda")  # bf16 rows of 40 bytes
    with pytest.raises(ops.MambaError) as e:
        run_gpu(inp)
    assert e.value.status == ops.MAMBA_ERR_UNSUPPORTED
    inp = inputs.scan_inputs(1, 64, 32, "bf16", seed=19, device="cuda")
    x = torch.empty(inp["x"].numel() * 2 + 8, dtype=torch.bfloat16, device="cuda")[1:1 + inp["x"].numel()]
    x = x.view(inp["x"].shape)
    with pytest.raises(ops.MambaError) as e:
        run_gpu(dict(inp, x=x))
    assert e.value.status == ops.MAMBA_ERR_INVALID_ARG
    inp = inputs.scan_inputs(1, 4096, 16, "bf16", seed=19, device="cuda")
    with pytest.raises(ops.MambaError) as e:
        run_gpu(inp, n_chunks=4, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == ops.MAMBA_ERR_WORKSPACE


@pytest.mark.parametrize("case", ["fast_decay", "slow_decay", "mixed", "very_slow_bf16"])
def test_chunk_carries_against_oracle(case):
    """The chunk-carry walk: with fast decay it stops after a few pieces (the
    carried state from far back is below 2^-32 of its size); with slow decay
    it must chain every boundary onto the previous one; a warp mixing both
    follows its slowest channel.  Each case is checked against the oracle and
    against the GPU's own one-pass scan (same fp32 arithmetic but for the
    carry sums).  A very slow leak (A = -0.0025, ~1/20000 per token) is
    checked in bf16: there the fp32 rounding of dA = 2^(dt A2) near 1 alone
    misstates the leak rate by ~0.1 %, beyond the fp32-I/O bound for any fp32
    recurrence, one pass included."""
    B, L, D = 1, 8192, 64
    io = "bf16" if case == "very_slow_bf16" else "f32"
    inp = inputs.scan_inputs(B, L, D, io, seed=23, device="cuda", with_state=True)
    if case == "slow_decay":
        inp["A_log"] = torch.full_like(inp["A_log"], -1.5)  # A = -0.22: no 2^-32 decay within a chunk
    elif case == "mixed":
        inp["A_log"][5] = -1.5
        inp["A_log"][40, :4] = -1.0
    elif case == "very_slow_bf16":
        inp["A_log"] = torch.full_like(inp["A_log"], -6.0)
    plan = ops.mamba_scan_plan(B, L, D, 4)
    assert plan["n_chunks"] == 4 and plan["pieces"] > 1
    outs = [t.clone() for t in run_gpu(inp, n_chunks=4)]
    check_against_oracle(inp, outs, f"carries {case}")
    y1, fh1, fcs1 = run_gpu(inp, n_chunks=1)
    torch.cuda.synchronize()
    if io == "f32":  # bf16 outputs of the two may round one ulp apart
        assert_close(outs[0], oracle_like(y1), "f32", f"{case}: chunked vs one pass, y")
    assert_close(outs[1], oracle_like(fh1), "f32", f"{case}: chunked vs one pass, h", fp32_output=True)
    assert torch.equal(outs[2], fcs1)


def _tile_regions(dt_raw):
    """Per 16-token tile of every batch row (over all channels): whether all of
    it lies below the softplus's small-argument bound, and whether it holds
    values above the threshold 20 and values in between."""
    v = dt_raw.float().cpu()
    B, L, D = v.shape
    tiles = [(b, t) for b in range(B) for t in range(0, L, 16)]
    small = sum(bool((v[b, t:t + 16] < -2.08).all()) for b, t in tiles)
    mixed = sum(bool((v[b, t:t + 16] > 20).any() and ((v[b, t:t + 16] > -2.08) & (v[b, t:t + 16] < 20)).any()
                     and (v[b, t:t + 16] < -2.08).any()) for b, t in tiles)
    return small, mixed


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("n_chunks", [1, 3])
def test_softplus_regions_against_oracle(io, n_chunks):
    """dt_raw across [-30, 30]: softplus's small-argument polynomial, its
    log2 region (up to the threshold) and the identity above 20, in tiles
    that lie wholly in the small region (the fast path) and tiles that mix
    all three (the per-value path), one pass and chunked (the carry walk
    takes the same two paths)."""
    B, L, D = 2, 1000, 64
    inp = inputs.scan_inputs(B, L, D, io, seed=71, device="cuda", with_state=True)
    inp["dt_raw"] = inputs.wide_dt_raw(B, L, D, io, seed=72, device="cuda")
    small, mixed = _tile_regions(inp["dt_raw"])
    assert small >= 5 and mixed >= 5, (small, mixed)
    check_against_oracle(inp, run_gpu(inp, n_chunks=n_chunks), f"wide dt {io} nc{n_chunks}")


def _large_range_case(seed):
    return inputs.scan_inputs(1, 8192, 64, "f32", seed=seed, device="cuda", with_state=True)


@pytest.mark.parametrize("case", ["h0_x1e6", "first_chunk_x_x1e3"])
def test_chunked_carry_large_dynamic_range(case):
    """Chunked mode (4 chunks, the carry walks stop early on these decays)
    with an initial state a million times the inputs' scale, or the first
    chunk's inputs a thousand times the later ones': against the oracle at
    the fp32 bound, and against the one-pass scan."""
    inp = _large_range_case(81)
    if case == "h0_x1e6":
        inp["h0"] = inp["h0"] * 1e6
    else:
        inp["x"][:, :2048] *= 1e3
    plan = ops.mamba_scan_plan(1, 8192, 64, 4)
    assert plan["n_chunks"] == 4 and plan["pieces"] > 1
    outs = [t.clone() for t in run_gpu(inp, n_chunks=4)]
    check_against_oracle(inp, outs, f"carries {case}")
    y1, fh1, fcs1 = run_gpu(inp, n_chunks=1)
    torch.cuda.synchronize()
    assert_close(outs[0], oracle_like(y1), "f32", f"{case}: chunked vs one pass, y")
    assert_close(outs[1], oracle_like(fh1), "f32", f"{case}: chunked vs one pass, h", fp32_output=True)


def test_exact_carry_flag_with_hidden_large_state():
    """A state 1e8 times the inputs' scale built up early in chunk 0 and hidden
    from y there (gate input z = 0 over chunk 0), decaying towards the
    boundary: the default carry walk stops where every state has decayed
    below 2^-32 and drops what lies before, which here is still visible in
    the next chunk's y.  With MAMBA_FLAG_EXACT_CARRY the walks cover whole
    chunks and the chunked scan matches the oracle at the fp32 bound."""
    B, L, D = 1, 8192, 32
    inp = inputs.scan_inputs(B, L, D, "f32", seed=83, device="cuda", with_state=True)
    inp["A_log"] = torch.zeros_like(inp["A_log"])  # A = -1: every state decays at the same rate
    # dt = 0.02 on every token: the walk over chunk 0 stops once the decay
    # to the boundary passes 2^-32 (1,109 tokens), after 18 pieces of 64, at
    # token 896, and drops tokens 0..895
    inp["dt_raw"] = torch.full_like(inp["dt_raw"], float(np.log(np.expm1(0.02))))
    inp["x"][:, 700:768] *= 1e8
    inp["z"][:, :2048] = 0.0
    plan = ops.mamba_scan_plan(B, L, D, 4)
    assert plan["n_chunks"] == 4 and plan["piece_len"] == 64
    y, fh, fcs = run_gpu(inp, n_chunks=4, flags=ops.MAMBA_FLAG_EXACT_CARRY)
    check_against_oracle(inp, (y, fh, fcs), "exact carries, hidden large state")
    y1, fh1, _ = run_gpu(inp, n_chunks=1)
    torch.cuda.synchronize()
    assert_close(y, oracle_like(y1), "f32", "exact chunked vs one pass, y")
    assert_close(fh, oracle_like(fh1), "f32", "exact chunked vs one pass, h", fp32_output=True)
