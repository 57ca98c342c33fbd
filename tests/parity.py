"""Helpers of the GPU-vs-oracle parity tests.

Tolerance (per output tensor): err = max|gpu - oracle| / rms(oracle) must be
<= 1e-4 for fp32 I/O and <= 1e-2 for bf16 I/O with fp32 state.  A bf16
output is itself a rounding of the fp32 result to 8 significant bits, which
alone moves an element by up to 2^-8 of its magnitude -- more than 1e-2 of
the rms at the tails of a large tensor.  For bf16 outputs each element is
therefore first allowed its own half-ulp rounding, 2^-8 |oracle|, and the
tolerance applies to what is left (the arithmetic error).  fp32 outputs
(final_h) and the conv state copies get no allowance; conv states must be
exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {"f32": 1e-4, "bf16": 1e-2}
BF16_HALF_ULP = 2.0 ** -8


def io_name(t: torch.Tensor) -> str:
    return {torch.float32: "f32", torch.bfloat16: "bf16"}[t.dtype]


def errors(gpu, ref: np.ndarray, rounded_bf16: bool):
    """(plain, arithmetic) relative errors as defined above."""
    g = oracle.f64(gpu)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    err = np.abs(g - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    if rms == 0.0:
        rms = 1.0
    plain = float(err.max()) / rms if err.size else 0.0
    if rounded_bf16:
        excess = np.maximum(err - BF16_HALF_ULP * np.abs(ref), 0.0)
        arith = float(excess.max()) / rms if err.size else 0.0
    else:
        arith = plain
    return plain, arith


def assert_close(gpu, ref, io: str, what: str = "", fp32_output: bool = False):
    plain, arith = errors(gpu, ref, rounded_bf16=(io == "bf16" and not fp32_output))
    tol = TOL[io]
    assert arith <= tol, f"{what}: error {arith:.3e} (plain {plain:.3e}) > {tol:g}"
    return plain, arith


def oracle_scan(inp: dict, channels=None, n_threads: int = 0):
    """Oracle on the inputs of one scan call, optionally on a subset of channels
    (channels are independent, B and C rows are shared)."""
    cs = slice(None) if channels is None else channels

    def ch(t, axis):
        if t is None:
            return None
        a = oracle.f64(t)
        return np.take(a, np.arange(a.shape[axis])[cs], axis=axis)

    return oracle.scan(ch(inp["x"], 2), ch(inp["z"], 2), ch(inp["dt_raw"], 2),
                       oracle.f64(inp["Bm"]), oracle.f64(inp["Cm"]),
                       ch(inp["A_log"], 0), ch(inp["Dskip"], 0), ch(inp["conv_w"], 0),
                       ch(inp.get("conv_b"), 0), ch(inp.get("h0"), 1),
                       ch(inp.get("conv_state0"), 2), n_threads=n_threads)


def to_device(inp: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def sample_channels(D: int, n: int) -> np.ndarray:
    """n channels spread over [0, D), always including the first and last."""
    return np.unique(np.linspace(0, D - 1, n).round().astype(np.int64))


def sample_scan_inputs(inp: dict, channels) -> dict:
    """The inputs restricted (on the device) to some channels; B and C rows
    are per token and kept whole."""
    idx = torch.as_tensor(channels, device=inp["x"].device)
    out = {}
    for k, v in inp.items():
        if v is None or k in ("Bm", "Cm"):
            out[k] = v
        elif k in ("x", "z", "dt_raw", "conv_state0"):
            out[k] = v.index_select(2, idx)
        elif k == "h0":
            out[k] = v.index_select(1, idx)
        else:  # per-channel parameters
            out[k] = v.index_select(0, idx)
    return out
