"""Decode step on the GPU (through the C ABI): against the fp64 oracle, and
bit-identical to the single-pass prefill scan on the same tokens."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close
from selective_state_space_118_b300 import inputs, ops

pytestmark = pytest.mark.gpu


def step(st, tok, t):
    return ops.mamba_step(st["h"], st["conv_state"], tok["x_t"][t], tok["z_t"][t],
                          tok["dt_raw_t"][t], tok["B_t"][t], tok["C_t"][t], st["A_log"],
                          st["Dskip"], st["conv_w"], st.get("conv_b"))


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L,D", [(1, 48), (37, 48), (130, 48), (37, 80), (130, 208), (37, 40), (130, 72)])
def test_steps_equal_single_pass_scan_bitwise(io, L, D):
    """D = 48: one partial block of 64 channels (the step moves h in blocks
    of 64 channels of a row); 80, 208: full blocks and a partial one; 40, 72:
    widths that are not multiples of 16 (a last scan group of 8 channels)."""
    B = 2
    inp = inputs.scan_inputs(B, L, D, io, seed=L, device="cuda", with_state=True)
    y, fh, fcs = ops.mamba_scan_fwd(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"],
                                    inp["A_log"], inp["Dskip"], inp["conv_w"], inp["conv_b"],
                                    inp["h0"], inp["conv_state0"], n_chunks=1)
    st = dict(h=inp["h0"].clone(), conv_state=inp["conv_state0"].clone(), A_log=inp["A_log"],
              Dskip=inp["Dskip"], conv_w=inp["conv_w"], conv_b=inp["conv_b"])
    tok = {"x_t": inp["x"].transpose(0, 1).contiguous(), "z_t": inp["z"].transpose(0, 1).contiguous(),
           "dt_raw_t": inp["dt_raw"].transpose(0, 1).contiguous(),
           "B_t": inp["Bm"].transpose(0, 1).contiguous(), "C_t": inp["Cm"].transpose(0, 1).contiguous()}
    ys = [step(st, tok, t) for t in range(L)]
    torch.cuda.synchronize()
    assert torch.equal(torch.stack(ys, 1), y)
    assert torch.equal(st["h"], fh)
    assert torch.equal(st["conv_state"], fcs)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_steps_against_oracle(io):
    w = inputs.DECODE
    B, D, T = 8, 256, 24
    st = inputs.decode_layer_state(w, 0, device="cuda")
    st["h"] = st["h"][:B, :D].contiguous()
    st["conv_state"] = st["conv_state"][:B, :, :D].contiguous()
    for k in ("A_log", "Dskip", "conv_w", "conv_b"):
        st[k] = st[k][:D].contiguous()
    tok = inputs.decode_token_inputs(w, 0, T, device="cuda", batch=B, d_inner=D)
    if io == "f32":
        st["conv_state"] = st["conv_state"].float()
        tok = {k: v.float() for k, v in tok.items()}
    h_ref, cs_ref = oracle.f64(st["h"]), oracle.f64(st["conv_state"])
    for t in range(T):
        y = step(st, tok, t)
        yr, h_ref, cs_ref = oracle.step(h_ref, cs_ref, tok["x_t"][t], tok["z_t"][t],
                                        tok["dt_raw_t"][t], tok["B_t"][t], tok["C_t"][t],
                                        st["A_log"], st["Dskip"], st["conv_w"], st["conv_b"])
        torch.cuda.synchronize()
        assert_close(y, yr, io, f"y step {t}")
    assert_close(st["h"], h_ref, io, "h", fp32_output=True)
    np.testing.assert_array_equal(oracle.f64(st["conv_state"]), cs_ref)


def test_step_rejects_bad_arguments():
    B, D = 2, 32
    h = torch.zeros(B, D, 16, device="cuda")
    cs = torch.zeros(B, 3, D, device="cuda", dtype=torch.bfloat16)
    v = torch.zeros(B, D, device="cuda", dtype=torch.bfloat16)
    bc = torch.zeros(B, 16, device="cuda", dtype=torch.bfloat16)
    A = torch.zeros(D, 8, device="cuda")
    with pytest.raises(ops.MambaError) as e:
        ops.mamba_step(h, cs, v, v, v, bc, bc, A, torch.zeros(D, device="cuda"),
                       torch.zeros(D, 4, device="cuda"))
    assert e.value.status == ops.MAMBA_ERR_UNSUPPORTED


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_steps_wide_softplus_range(io):
    """dt_raw across [-30, 30] (softplus's three regions): steps against the
    oracle, and bit for bit equal to a one-pass scan of the same tokens (the
    scan's per-tile fast path and per-value path give softplus's bits)."""
    B, L, D = 2, 96, 48
    inp = inputs.scan_inputs(B, L, D, io, seed=91, device="cuda", with_state=True)
    inp["dt_raw"] = inputs.wide_dt_raw(B, L, D, io, seed=92, device="cuda")
    y, fh, fcs = ops.mamba_scan_fwd(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"],
                                    inp["A_log"], inp["Dskip"], inp["conv_w"], inp["conv_b"],
                                    inp["h0"], inp["conv_state0"], n_chunks=1)
    st = dict(h=inp["h0"].clone(), conv_state=inp["conv_state0"].clone(), A_log=inp["A_log"],
              Dskip=inp["Dskip"], conv_w=inp["conv_w"], conv_b=inp["conv_b"])
    tok = {"x_t": inp["x"].transpose(0, 1).contiguous(), "z_t": inp["z"].transpose(0, 1).contiguous(),
           "dt_raw_t": inp["dt_raw"].transpose(0, 1).contiguous(),
           "B_t": inp["Bm"].transpose(0, 1).contiguous(), "C_t": inp["Cm"].transpose(0, 1).contiguous()}
    h_ref, cs_ref = oracle.f64(inp["h0"]), oracle.f64(inp["conv_state0"])
    ys = []
    for t in range(L):
        ys.append(step(st, tok, t))
        yr, h_ref, cs_ref = oracle.step(h_ref, cs_ref, tok["x_t"][t], tok["z_t"][t], tok["dt_raw_t"][t],
                                        tok["B_t"][t], tok["C_t"][t], st["A_log"], st["Dskip"],
                                        st["conv_w"], st["conv_b"])
        torch.cuda.synchronize()
        assert_close(ys[-1], yr, io, f"y step {t}")
    assert_close(st["h"], h_ref, io, "h", fp32_output=True)
    assert torch.equal(torch.stack(ys, 1), y)
    assert torch.equal(st["h"], fh)
    assert torch.equal(st["conv_state"], fcs)
