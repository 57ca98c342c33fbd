"""Seeded synthetic inputs for the selective-scan workloads.

This module only draws random tensors with the shapes and value
distributions of the workloads; it holds none of the scan's arithmetic, so
both the CUDA path and the fp64 oracle can be fed from it.

Distributions (the same for every workload unless noted):
  x, z            ~ N(0, 1)
  B, C            ~ N(0, bc_std^2)   (bc_std = 1 for the small cases,
                                      0.25 i.e. variance 1/16 for the
                                      Jamba-shaped cases)
  dt              log-uniform in [1e-3, 1e-1]; dt_raw = log(expm1(dt)), so
                  that softplus(dt_raw) = dt (computed in fp32, then rounded
                  to the I/O dtype; consumers use the rounded dt_raw)
  A_log[c, n]     = log(n + 1)             (n is 0-based: A in {-1..-16})
  D               = 1
  conv_w          ~ U(-0.5, 0.5)
  conv_b          = 0
  h (decode)      ~ N(0, 0.1^2); conv_state ~ N(0, 1)

Tensors are drawn with a ``torch.Generator`` on the requested device, seeded
with the workload's seed, in a fixed order.  CPU and CUDA generators give
different values for the same seed; every consumer of one draw uses that one
draw.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

D_STATE = 16
D_CONV = 4


@dataclass(frozen=True)
class ScanWorkload:
    name: str
    batch: int
    seqlen: int
    d_inner: int
    io: str          # "f32" or "bf16"
    seed: int
    bc_std: float
    host_chunks: int = 1   # >1: the sequence is fed as this many calls with carried state


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    layers: int
    batch: int
    d_inner: int
    steps: int
    io: str
    seed: int
    bc_std: float
    h_std: float


# The five workloads: a tiny fp32 case, a small bf16 layer, a Jamba-shaped
# layer (hidden 4096, expand 2), a 256k-token prefill fed in 64 carried
# chunks, and 28-layer batched decode.
TINY_F32 = ScanWorkload("tiny_scan_f32_b1_l256_d64", 1, 256, 64, "f32", 0, 1.0)
SMALL_BF16 = ScanWorkload("small_layer_bf16_b2_l2048_d1024", 2, 2048, 1024, "bf16", 1, 1.0)
JAMBA_PREFILL = ScanWorkload("jamba_prefill_bf16_b1_l32768_d8192", 1, 32768, 8192, "bf16", 2, 0.25)
PREFILL_256K = ScanWorkload("prefill_256k_bf16_b1_l262144_d8192", 1, 262144, 8192, "bf16", 3, 0.25,
                            host_chunks=64)
DECODE = DecodeWorkload("decode_bf16_28layers_b64_d8192_256steps", 28, 64, 8192, 256, "bf16", 4,
                        0.25, 0.1)

SCAN_WORKLOADS = {w.name: w for w in (TINY_F32, SMALL_BF16, JAMBA_PREFILL, PREFILL_256K)}


def torch_dtype(io: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[io]


def _normal(g, shape, std, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _dt_raw(g, shape, device, lo=1e-3, hi=1e-1):
    r = torch.rand(shape, generator=g, device=device, dtype=torch.float32)
    dt = torch.exp(math.log(lo) + r * (math.log(hi) - math.log(lo)))
    return torch.log(torch.expm1(dt))


# dt_raw ranges of the wide-range draw (one per 16-token block): every value
# below the softplus's small-argument bound; the full range across the
# threshold 20; a narrow band around the small-argument bound (-2.08); and
# values past the threshold only or near it.
WIDE_DT_RANGES = ((-9.0, -2.2), (-30.0, 30.0), (-2.3, -1.85), (12.0, 30.0))


def wide_dt_raw(batch: int, seqlen: int, d_inner: int, io: str, seed: int, device="cpu") -> torch.Tensor:
    """dt_raw (B, L, D) in the I/O dtype spanning [-30, 30]: each block of 16
    consecutive tokens draws uniformly from one of WIDE_DT_RANGES, the range
    chosen at random per block, so that some 16-token tiles lie entirely in
    one region and others mix all of them."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    blocks = (seqlen + 15) // 16
    mode = torch.randint(0, len(WIDE_DT_RANGES), (batch, blocks), generator=g, device=dev)
    lo = torch.tensor([r[0] for r in WIDE_DT_RANGES], device=dev)[mode]
    hi = torch.tensor([r[1] for r in WIDE_DT_RANGES], device=dev)[mode]
    lo = lo.repeat_interleave(16, dim=1)[:, :seqlen, None]
    hi = hi.repeat_interleave(16, dim=1)[:, :seqlen, None]
    r = torch.rand((batch, seqlen, d_inner), generator=g, device=dev, dtype=torch.float32)
    return (lo + r * (hi - lo)).to(torch_dtype(io))


def layer_params(d_inner: int, g: torch.Generator, device) -> dict:
    """Per-layer parameters (fp32): A_log, D, conv_w, conv_b."""
    n = torch.arange(D_STATE, device=device, dtype=torch.float32)
    A_log = torch.log(n + 1.0).expand(d_inner, D_STATE).contiguous()
    Dskip = torch.ones(d_inner, device=device, dtype=torch.float32)
    conv_w = torch.rand((d_inner, D_CONV), generator=g, device=device,
                        dtype=torch.float32) - 0.5
    conv_b = torch.zeros(d_inner, device=device, dtype=torch.float32)
    return dict(A_log=A_log, Dskip=Dskip, conv_w=conv_w, conv_b=conv_b)


def scan_inputs(batch: int, seqlen: int, d_inner: int, io: str, seed: int,
                bc_std: float = 1.0, device="cpu", with_state: bool = False,
                h_std: float = 0.1) -> dict:
    """All inputs of one scan call.  Activations are in the I/O dtype,
    parameters in fp32.  with_state=True also draws h0 (B,D,16) fp32 and
    conv_state0 (B,3,D) in the I/O dtype."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    dt = torch_dtype(io)
    shape = (batch, seqlen, d_inner)
    out = {}
    out["x"] = _normal(g, shape, 1.0, dev).to(dt)
    out["z"] = _normal(g, shape, 1.0, dev).to(dt)
    out["dt_raw"] = _dt_raw(g, shape, dev).to(dt)
    out["Bm"] = _normal(g, (batch, seqlen, D_STATE), bc_std, dev).to(dt)
    out["Cm"] = _normal(g, (batch, seqlen, D_STATE), bc_std, dev).to(dt)
    out.update(layer_params(d_inner, g, dev))
    if with_state:
        out["h0"] = _normal(g, (batch, d_inner, D_STATE), h_std, dev)
        out["conv_state0"] = _normal(g, (batch, D_CONV - 1, d_inner), 1.0, dev).to(dt)
    return out


def complex_scan_inputs(batch: int, seqlen: int, d_inner: int, io: str, seed: int,
                        bc_std: float = 1.0, device="cpu", with_state: bool = False,
                        h_std: float = 0.1) -> dict:
    """Inputs of one call of the complex-valued scan: those of scan_inputs
    (B and C rows of 16 reals read as 8 complex numbers, (re, im) pairs; h0
    (B,D,16) likewise), with 8 modes per channel: A_log[c, n] = log(n + 1)
    and rotation frequencies theta[c, n] = pi * n, n = 0..7."""
    out = scan_inputs(batch, seqlen, d_inner, io, seed, bc_std, device, with_state, h_std)
    modes = D_STATE // 2
    n = torch.arange(modes, device=out["A_log"].device, dtype=torch.float32)
    out["A_log"] = torch.log(n + 1.0).expand(d_inner, modes).contiguous()
    out["theta"] = (math.pi * n).expand(d_inner, modes).contiguous()
    return out


def workload_inputs(w: ScanWorkload, device="cpu", **kw) -> dict:
    return scan_inputs(w.batch, w.seqlen, w.d_inner, w.io, w.seed, w.bc_std, device, **kw)


def decode_layer_state(w: DecodeWorkload, layer: int, device="cpu") -> dict:
    """Initial state and parameters of one decode layer."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 1000 + layer)
    dt = torch_dtype(w.io)
    st = {}
    st["h"] = _normal(g, (w.batch, w.d_inner, D_STATE), w.h_std, dev)
    st["conv_state"] = _normal(g, (w.batch, D_CONV - 1, w.d_inner), 1.0, dev).to(dt)
    st.update(layer_params(w.d_inner, g, dev))
    return st


def decode_token_inputs(w: DecodeWorkload, layer: int, steps: int, device="cpu",
                        batch: int | None = None, d_inner: int | None = None) -> dict:
    """Per-token inputs of one layer for `steps` consecutive tokens:
    x_t, z_t, dt_raw_t (steps,B,D) and B_t, C_t (steps,B,16), I/O dtype."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 1000 + 500 + layer)
    dt = torch_dtype(w.io)
    B = w.batch if batch is None else batch
    D = w.d_inner if d_inner is None else d_inner
    shape = (steps, B, D)
    return dict(
        x_t=_normal(g, shape, 1.0, dev).to(dt),
        z_t=_normal(g, shape, 1.0, dev).to(dt),
        dt_raw_t=_dt_raw(g, shape, dev).to(dt),
        B_t=_normal(g, (steps, B, D_STATE), w.bc_std, dev).to(dt),
        C_t=_normal(g, (steps, B, D_STATE), w.bc_std, dev).to(dt),
    )
