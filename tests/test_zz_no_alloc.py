"""mamba_scan_fwd_noalloc, the prefill entry point for callers that cannot
allocate device memory (for example a plugin whose host framework owns all
device memory through its own pool, or a path that must not take
cudaMalloc's implicit synchronisation).  It must give the same results as
mamba_scan_fwd, which takes a caller-allocated workspace, on consecutive
calls that share its fixed scratch array, and must refuse sizes that do not
fit that array.  This file is collected last on purpose."""
import ctypes

import pytest
import torch

from parity import assert_close
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


def _compare(io, got, ref, what):
    for g, r, name, fp32 in zip(got, ref, ("y", "final_h", "final_conv_state"), (False, True, False)):
        torch.cuda.synchronize()
        assert_close(g, r.double().cpu().numpy(), io, f"{what} {name}", fp32_output=fp32)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    # call 1: a chunked plan (carries live in the scratch); call 2: one pass
    cases = [(inputs.scan_inputs(2, 2048, 1024, "bf16", seed=61, device="cuda", with_state=True), 0),
             (inputs.scan_inputs(1, 700, 48, "f32", seed=62, device="cuda", with_state=True), 1)]
    for i, (inp, n_chunks) in enumerate(cases):
        io = "bf16" if inp["x"].dtype == torch.bfloat16 else "f32"
        ref = ops.mamba_scan_fwd(*_args(inp), n_chunks=n_chunks)
        out = _outputs_like(inp)
        got = ops.mamba_scan_fwd_noalloc(*_args(inp), n_chunks=n_chunks, **out)
        _compare(io, got, ref, f"call {i + 1}")
        assert ops.mamba_last_error() == ops.MAMBA_OK


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
