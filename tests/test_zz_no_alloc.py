"""mamba_scan_fwd_noalloc, the prefill entry point for callers that cannot
allocate device memory (for example a plugin whose host framework owns all
device memory through its own pool, or a path that must not take
cudaMalloc's implicit synchronisation).  It runs the same kernels with the
same plan as mamba_scan_fwd, which takes a caller-allocated workspace, so
its results must be the same bits, on consecutive calls that share its fixed
scratch array (whatever an earlier call left there), and must refuse sizes
that do not fit that array.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from parity import assert_close, oracle_scan
from selective_state_space_118_b300 import inputs, ops

pytestmark = pytest.mark.gpu


def _outputs_like(inp):
    B, L, D = inp["x"].shape
    return dict(y=torch.empty_like(inp["x"]),
                final_h=torch.empty(B, D, 16, device="cuda"),
                final_conv_state=torch.empty(B, 3, D, device="cuda", dtype=inp["x"].dtype))


def _args(inp):
    return (inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"], inp["Dskip"],
            inp["conv_w"], inp["conv_b"], inp.get("h0"), inp.get("conv_state0"))


def test_noalloc_equals_workspace_entry_point_on_consecutive_calls():
    # two chunked calls of different sizes back to back (the second starts on
    # the counters and carries the first left in the scratch), then a
    # one-pass call; every call must give mamba_scan_fwd's bits
    cases = [(inputs.scan_inputs(2, 2048, 1024, "bf16", seed=61, device="cuda", with_state=True), 4),
             (inputs.scan_inputs(1, 3000, 256, "f32", seed=63, device="cuda", with_state=True), 3),
             (inputs.scan_inputs(1, 700, 48, "f32", seed=62, device="cuda", with_state=True), 1)]
    for i, (inp, n_chunks) in enumerate(cases):
        B, L, D = inp["x"].shape
        assert ops.mamba_scan_plan(B, L, D, n_chunks)["n_chunks"] == n_chunks
        ref = ops.mamba_scan_fwd(*_args(inp), n_chunks=n_chunks)
        got = ops.mamba_scan_fwd_noalloc(*_args(inp), n_chunks=n_chunks, **_outputs_like(inp))
        torch.cuda.synchronize()
        for g, r, name in zip(got, ref, ("y", "final_h", "final_conv_state")):
            assert torch.equal(g, r), f"call {i + 1}: {name} differs from mamba_scan_fwd"
        assert ops.mamba_last_error() == ops.MAMBA_OK


def test_noalloc_against_oracle():
    inp = inputs.scan_inputs(1, 1500, 64, "f32", seed=64, device="cuda", with_state=True)
    y, fh, fcs = ops.mamba_scan_fwd_noalloc(*_args(inp), n_chunks=3, **_outputs_like(inp))
    torch.cuda.synchronize()
    yr, fhr, fcsr = oracle_scan(inp)
    assert_close(y, yr, "f32", "noalloc y")
    assert_close(fh, fhr, "f32", "noalloc final_h", fp32_output=True)
    np.testing.assert_array_equal(fcs.double().cpu().numpy(), fcsr)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = ops.load_library()
    fake = 0x10000  # never dereferenced: the size check comes first
    too_long = ops.MAMBA_NOALLOC_SCRATCH_BYTES // 128 + 64  # tokens: widened B/C alone exceed it
    a = ops.ScanArgs(batch=1, seqlen=too_long, d_inner=16, d_state=16, d_conv=4, io=ops.MAMBA_BF16,
                     x=fake, z=fake, dt_raw=fake, Bm=fake, Cm=fake, A_log=fake, Dskip=fake,
                     conv_w=fake, y=fake, n_chunks=1)
    assert ops.mamba_scan_workspace_size(1, too_long, 16, 1) > ops.MAMBA_NOALLOC_SCRATCH_BYTES
    assert lib.mamba_scan_fwd_noalloc(ctypes.byref(a), None) == ops.MAMBA_ERR_WORKSPACE
    assert lib.mamba_scan_fwd_noalloc(None, None) == ops.MAMBA_ERR_INVALID_ARG
