"""Mamba-2's chunked scan (mamba2_scan_fwd: tensor-core chunk products) on
the GPU against the fp64 recurrence oracle (oracle.ssd), with the bf16 bound
of parity.py (y first allowed its own bf16 rounding; the final state is
fp32).  The tensor cores take bf16 operands: the inputs are bf16 already,
and the fp32 quantities the kernels feed them (the decay-weighted C B^T
entries, the decay-weighted B rows, the entering state) go in as two bf16
terms each (hi + lo, ~16 significant bits), so the products keep near-fp32
accuracy."""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close
from selective_state_space_118_b300 import ops

pytestmark = pytest.mark.gpu


def case(B, L, H, G, seed, gate=True, state=True, dt_lo=1e-3, dt_hi=1e-1):
    g = torch.Generator(device="cuda").manual_seed(seed)
    bf = torch.bfloat16

    def n(*shape, std=1.0):
        return (torch.randn(shape, generator=g, device="cuda") * std).to(bf)
    u = torch.rand((B, L, H), generator=g, device="cuda")
    dt = torch.exp(np.log(dt_lo) + u * (np.log(dt_hi) - np.log(dt_lo)))
    return dict(x=n(B, L, H, 64), dt_raw=torch.log(torch.expm1(dt)).to(bf),
                A_log=torch.log(torch.arange(1, H + 1, device="cuda", dtype=torch.float32) % 16 + 1),
                Bm=n(B, L, G, 16, std=0.5), Cm=n(B, L, G, 16, std=0.5),
                Dskip=torch.rand(H, generator=g, device="cuda"),
                z=n(B, L, H, 64) if gate else None,
                h0=(torch.randn((B, H, 16, 64), generator=g, device="cuda") * 0.1) if state else None)


def run(p):
    return ops.mamba2_scan_fwd(p["x"], p["dt_raw"], p["A_log"], p["Bm"], p["Cm"], p["Dskip"], p["z"], p["h0"])


@pytest.mark.parametrize("B,L,H,G,gate,state", [
    (1, 1, 1, 1, True, True),
    (1, 64, 2, 1, False, False),
    (2, 65, 4, 2, True, True),
    (1, 200, 3, 3, True, False),
    (2, 1000, 8, 1, True, True),
    (1, 4096, 16, 4, True, True),
])
def test_ssd_against_oracle(B, L, H, G, gate, state):
    p = case(B, L, H, G, seed=B * 1000 + L + H, gate=gate, state=state)
    y, fs = run(p)
    torch.cuda.synchronize()
    yr, fsr = oracle.ssd(**p)
    what = f"B{B} L{L} H{H} G{G}"
    assert_close(y, yr, "bf16", f"{what} y")
    assert_close(fs, fsr, "bf16", f"{what} final state", fp32_output=True)


def test_ssd_slow_decay():
    """dt ~ 1e-3 and A = -1: the state lives across hundreds of chunks."""
    p = case(1, 8192, 2, 1, seed=7, dt_lo=1e-3, dt_hi=2e-3)
    p["A_log"] = torch.zeros_like(p["A_log"])
    y, fs = run(p)
    torch.cuda.synchronize()
    yr, fsr = oracle.ssd(**p)
    assert_close(y, yr, "bf16", "slow decay y")
    assert_close(fs, fsr, "bf16", "slow decay final state", fp32_output=True)


def test_ssd_seqlen_zero_and_errors():
    p = case(1, 0, 2, 1, seed=9)
    y, fs = run(p)
    torch.cuda.synchronize()
    assert torch.equal(fs, p["h0"])
    p = case(1, 64, 2, 1, seed=9)
    x = torch.empty(1, 64, 2, 32, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ops.MambaError) as e:
        ops.mamba2_scan_fwd(x, p["dt_raw"], p["A_log"], p["Bm"], p["Cm"], p["Dskip"])
    assert e.value.status == ops.MAMBA_ERR_UNSUPPORTED


def test_ssd_large_dt_fast_decay():
    """dt up to ~5 with A down to -16: a 16-token row block spans far more
    than 2^60 of decay, so the output kernel takes its exact per-pair decay
    path (the split path covers the other cases above)."""
    p = case(2, 300, 4, 2, seed=11, dt_lo=0.5, dt_hi=5.0)
    p["A_log"] = torch.log(torch.tensor([1.0, 4.0, 10.0, 16.0], device="cuda"))
    y, fs = run(p)
    torch.cuda.synchronize()
    yr, fsr = oracle.ssd(**p)
    assert_close(y, yr, "bf16", "large dt y")
    assert_close(fs, fsr, "bf16", "large dt final state", fp32_output=True)


def test_ssd_fullsize_sampled_heads():
    """The benchmark's configuration (1 x 32768 tokens, 128 heads of 64, one
    group, the gate), in the launch configuration bench.py times: 6 sampled
    heads against the oracle (heads are independent given B and C)."""
    p = case(1, 32768, 128, 1, seed=3)
    y, fs = run(p)
    torch.cuda.synchronize()
    heads = [0, 1, 37, 64, 100, 127]
    idx = torch.tensor(heads, device="cuda")
    sub = dict(p, x=p["x"][:, :, idx].contiguous(), z=p["z"][:, :, idx].contiguous(),
               dt_raw=p["dt_raw"][:, :, idx].contiguous(), A_log=p["A_log"][idx].contiguous(),
               Dskip=p["Dskip"][idx].contiguous(), h0=p["h0"][:, idx].contiguous())
    yr, fsr = oracle.ssd(**sub)
    assert_close(y[:, :, idx], yr, "bf16", "full size y (sampled heads)")
    assert_close(fs[:, idx], fsr, "bf16", "full size final state (sampled heads)", fp32_output=True)
