#!/usr/bin/env python
"""Benchmark of the selective-scan library on synthetic Jamba-shaped inputs.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--seqlen L] [--n-chunks K]
                [--no-e2e] [--no-cpu-baseline] [--no-decode] [--no-ssd]
                [--no-layer] [--no-backward]
                [--no-prefill | --backward-only | --layer-only | --ssd-only]

A step is one prefill pass of the layer (conv, SiLU, softplus, discretised
scan, D skip, SiLU(z) gate; final h and conv state) over the workload's whole
batch, through the C ABI, inputs resident in HBM (larger than L2).  Prints
one JSON line on rank 0.  Under torchrun every rank runs an independent
replica (the scan has no cross-device exchange): value = elements all ranks
processed / max-over-ranks time.  The line also carries, unless switched
off, the end-to-end number (host copies in the timed region), the decode
block, Mamba-2's scan, the whole layer and the backward, each with its own
timing, roofline and clocks; the --*-only switches print one block alone
(profiling).

--impl reference times the fp64 CPU oracle (the definition the library is
checked against) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_118_b300 import inputs  # noqa: E402

METRIC = "selective-scan elements/s (B*L*d_inner), HBM GB/s vs B300 peak; decode steps/s"
UNIT = "elements/s"
D_STATE, D_CONV = 16, 4


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


# ---------------------------------------------------------------- distributed
# The scan has no cross-device exchange: N ranks run N independent replicas
# (one per GPU); only the timing is combined (a barrier on both sides of the
# timed region and the maximum time over ranks).
def dist_setup(n_gpus: int, backend: str | None = None):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    else:
        torch.cuda.set_device(0) if torch.cuda.is_available() else None
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank_step: int, steps: int, world: int, t_max_ms: float) -> float:
    """Whole-job throughput: the units all ranks processed / the slowest rank's time."""
    return units_per_rank_step * steps * world / (t_max_ms / 1e3)


# ---------------------------------------------------------------- clocks
class _Nvml:
    """Minimal read-only NVML access through the driver's libnvidia-ml (ctypes):
    SM clock, max SM clock and the active clock-event reasons."""

    def __init__(self, device_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self._check(self.lib.nvmlInit_v2())
        props = torch.cuda.get_device_properties(device_index)
        self.h = ctypes.c_void_p()
        uuid = str(getattr(props, "uuid", ""))
        rc = 1
        if uuid:
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            rc = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h))
        if rc != 0:
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            self._check(self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)))

    @staticmethod
    def _check(rc):
        if rc != 0:
            raise RuntimeError(f"NVML error {rc}")

    def sm_clock(self):
        v = self.ct.c_uint()
        self._check(self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(v)))  # NVML_CLOCK_SM
        return v.value

    def max_sm_clock(self):
        v = self.ct.c_uint()
        self._check(self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, self.ct.byref(v)))
        return v.value

    def reasons(self):
        v = self.ct.c_ulonglong()
        self._check(self.lib.nvmlDeviceGetCurrentClocksEventReasons(self.h, self.ct.byref(v)))
        return v.value


class ClockSampler:
    """Polls NVML (read-only) every millisecond while the timed region runs."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting"}

    def __init__(self, device_index: int, period_s: float = 0.001):
        self.samples, self.reasons, self.max_mhz, self.error = [], 0, None, None
        self.period = period_s
        self._stop = threading.Event()
        self.nv = None
        try:
            self.nv = _Nvml(device_index)
            self.max_mhz = self.nv.max_sm_clock()
        except Exception as e:  # report, do not guess
            self.nv, self.error = None, f"{type(e).__name__}: {e}"

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.sm_clock())
                self.reasons |= int(self.nv.reasons())
            except Exception as e:
                self.error = f"{type(e).__name__}: {e}"
            time.sleep(self.period)

    def __enter__(self):
        if self.nv is not None:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self.nv is not None:
            self.t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"],
                    "samples": 0, "error": self.error}
        reasons = [n for bit, n in self.REASONS.items() if self.reasons & bit]
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples)}


# ---------------------------------------------------------------- ncu traffic record
def sources_digest() -> str:
    """sha256 over the CUDA/C++ sources of the library: a DRAM-traffic figure
    measured by ncu is reported only for the sources it was measured on."""
    import hashlib
    csrc = os.path.join(ROOT, "selective_state_space_118_b300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".cpp", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def measured_traffic(key: str):
    """DRAM bytes per call from profiles/dram_traffic.json (written from an ncu
    capture, see the profiles' command lines), or None when absent or taken on
    other sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f)
        if rec.get("sources_sha256") != sources_digest():
            return None
        return rec["per_call_bytes"].get(key)
    except Exception:
        return None


# ---------------------------------------------------------------- byte counts
def scan_algorithmic_bytes(B, L, D, es):
    """Minimum HBM bytes of one prefill call: x, z, dt_raw read and y written
    once; B, C rows; parameters; final h (fp32) and final conv state."""
    act = 4 * B * L * D * es
    bc = 2 * B * L * D_STATE * es
    params = D * (D_STATE + 1 + D_CONV + 1) * 4
    state = B * D * D_STATE * 4 + B * (D_CONV - 1) * D * es
    return act + bc + params + state


def bwd_algorithmic_bytes(B, L, D, es):
    """Minimum HBM bytes of one backward call: x, z, dt_raw, dy read and dx,
    dz, ddt_raw written once; B, C rows read and dB, dC (fp32) written; the
    parameters read and their gradients written."""
    act = 7 * B * L * D * es
    bc = 2 * B * L * D_STATE * es + 2 * B * L * D_STATE * 4
    params = 2 * D * (D_STATE + 1 + D_CONV + 1) * 4
    return act + bc + params


def decode_algorithmic_bytes(B, D, es):
    """Minimum HBM bytes of one decode step of one layer: h read and written
    (fp32), x_t, z_t, dt_raw_t read and y_t written, the conv state's 3
    values read and one written, B_t and C_t."""
    return B * D * (2 * D_STATE * 4 + 4 * es + 4 * es) + 2 * B * D_STATE * es


# ---------------------------------------------------------------- our arm
def scan_call(ops, inp, out, ws, stream, n_chunks=0):
    ops.mamba_scan_fwd(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"],
                       inp["Dskip"], inp["conv_w"], inp["conv_b"], None, None, y=out["y"],
                       final_h=out["fh"], final_conv_state=out["fcs"], workspace=ws,
                       n_chunks=n_chunks, stream=stream)


def bench_prefill(w, steps, warmup, world, local, n_chunks_req=0):
    from selective_state_space_118_b300 import ops
    dev = torch.device("cuda", local)
    inp = inputs.workload_inputs(w, device=dev)
    B, L, D = w.batch, w.seqlen, w.d_inner
    es = 2 if w.io == "bf16" else 4
    out = {"y": torch.empty_like(inp["x"]),
           "fh": torch.empty(B, D, D_STATE, device=dev),
           "fcs": torch.empty(B, D_CONV - 1, D, device=dev, dtype=inp["x"].dtype)}
    nbytes = ops.mamba_scan_workspace_size(B, L, D, n_chunks_req)
    ws = torch.empty(max(nbytes, 1), device=dev, dtype=torch.uint8) if nbytes else None
    plan = ops.mamba_scan_plan(B, L, D, n_chunks_req)
    n_chunks = plan["n_chunks"]
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        scan_call(ops, inp, out, ws, stream, n_chunks_req)
    torch.cuda.synchronize(dev)
    assert ops.mamba_last_error(stream) == ops.MAMBA_OK
    barrier(world)
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(dev.index) as clk:
        ev[0].record(stream)
        for i in range(steps):
            scan_call(ops, inp, out, ws, stream, n_chunks_req)
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    assert ops.mamba_last_error(stream) == ops.MAMBA_OK
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    t_total_ms = ev[0].elapsed_time(ev[steps])
    t_max_ms = max_over_ranks(t_total_ms, world)
    elems = B * L * D
    alg = scan_algorithmic_bytes(B, L, D, es)
    res = dict(elems=elems, t_ms=t_max_ms, per_launch_ms=statistics.mean(per),
               per_launch_min_ms=min(per), alg_bytes=alg, n_chunks=n_chunks, plan=plan,
               launches_per_step=2 if n_chunks == 1 else 3, clocks=clk.summary(),
               in_bytes=sum(inp[k].numel() * inp[k].element_size()
                            for k in ("x", "z", "dt_raw", "Bm", "Cm")),
               out_bytes=out["y"].numel() * out["y"].element_size())
    return res, inp, out, ws


def bench_e2e(w, inp, out, ws, steps, local):
    """Same metric through the C ABI with the inputs in pinned HOST memory:
    every step copies x, z, dt_raw, B, C host->device, scans, and copies y
    device->host, all inside the timed region.  Steps are pipelined the way a
    serving loop would run independent requests: uploads on one stream, the
    scan on another, downloads on a third, with two device buffer sets, so
    that step i+1's upload overlaps step i's scan and download (the host
    link's two directions work at the same time)."""
    from selective_state_space_118_b300 import ops
    dev = torch.device("cuda", local)
    names = ("x", "z", "dt_raw", "Bm", "Cm")
    host = {k: torch.empty(inp[k].shape, dtype=inp[k].dtype, pin_memory=True) for k in names}
    for k in host:
        host[k].copy_(inp[k])
    y_host = [torch.empty(out["y"].shape, dtype=out["y"].dtype, pin_memory=True) for _ in range(2)]
    bufs = [{k: torch.empty_like(inp[k]) for k in names} for _ in range(2)]
    outs = [dict(out, y=torch.empty_like(out["y"])) for _ in range(2)]
    up, comp, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    uploaded = [torch.cuda.Event() for _ in range(2)]
    scanned = [torch.cuda.Event() for _ in range(2)]
    downloaded = [torch.cuda.Event() for _ in range(2)]
    for e in downloaded:
        e.record(down)

    def step(i):
        s = i % 2
        up.wait_event(downloaded[s])  # buffer set s is free once its last y left
        with torch.cuda.stream(up):
            for k in names:
                bufs[s][k].copy_(host[k], non_blocking=True)
        uploaded[s].record(up)
        comp.wait_event(uploaded[s])
        scan_call(ops, dict(inp, **bufs[s]), outs[s], ws, comp)
        scanned[s].record(comp)
        down.wait_event(scanned[s])
        with torch.cuda.stream(down):
            y_host[s].copy_(outs[s]["y"], non_blocking=True)
        downloaded[s].record(down)

    step(0)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
    torch.cuda.synchronize(dev)
    t = time.perf_counter() - t0
    bi = sum(h.numel() * h.element_size() for h in host.values())
    bo = y_host[0].numel() * y_host[0].element_size()
    return {"t": t, "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "steps": steps, "ms_per_step": t * 1e3 / steps,
            "pipelining": "uploads / scan / downloads on three streams, two buffer sets"}


def bench_backward(w, steps, warmup, local, n_chunks_req=0):
    """The backward of the prefill (mamba_scan_bwd: it recomputes the forward
    with tile checkpoints, then the reverse sweep) on the same workload, with
    a seeded random dy; elements/s over B * L * D, like the forward."""
    from selective_state_space_118_b300 import ops
    dev = torch.device("cuda", local)
    inp = inputs.workload_inputs(w, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 1000)
    dy = torch.randn(inp["x"].shape, generator=g, device=dev).to(inp["x"].dtype)
    B, L, D = w.batch, w.seqlen, w.d_inner
    ws = torch.empty(ops.mamba_scan_bwd_workspace_size(B, L, D, n_chunks_req), device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)
    out = None

    def call():
        return ops.mamba_scan_bwd(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"],
                                  inp["Dskip"], inp["conv_w"], inp["conv_b"], dy=dy, out=out, workspace=ws,
                                  n_chunks=n_chunks_req, stream=stream)

    out = call()
    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    assert ops.mamba_last_error(stream) == ops.MAMBA_OK
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(dev.index) as clk:
        ev[0].record(stream)
        for i in range(steps):
            call()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
    assert ops.mamba_last_error(stream) == ops.MAMBA_OK
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    t = ev[0].elapsed_time(ev[steps]) / 1e3 / steps
    es = 2 if w.io == "bf16" else 4
    alg = bwd_algorithmic_bytes(B, L, D, es)
    hbm, src = peaks()
    n_chunks = ops.mamba_scan_plan(B, L, D, n_chunks_req)["n_chunks"]
    launches = 7 if n_chunks > 1 else 5
    reuse = bench_tile_state_reuse(ops, inp, dy, out, ws, n_chunks_req, stream, steps, warmup, dev)
    res = {"metric": "backward elements/s", "value": B * L * D / t, "unit": UNIT,
           "config": {"workload": w.name, "batch": B, "seqlen": L, "d_inner": D, "n_chunks": n_chunks,
                      "dy": "seeded N(0,1) in the I/O dtype"},
           "ms_per_call": t * 1e3, "ms_per_call_min": min(per),
           "roofline": {"bound": "issue", "hbm_achieved": alg / t / 1e9, "hbm_peak": hbm, "unit": "GB/s",
                        "hbm_frac": alg / t / 1e9 / hbm, "peak_source": src,
                        "algorithmic_bytes_per_call": alg,
                        "note": "instruction-issue bound (forward recomputed from tile checkpoints, "
                                "then the reverse sweep); the HBM fraction is context"},
           "gpu_launches": launches * steps, "clocks": clk.summary(), "tile_state_reuse": reuse}
    del inp, dy, ws, out
    return res


def bench_tile_state_reuse(ops, inp, dy, out, ws, n_chunks_req, stream, steps, warmup, dev):
    """A training step's two scan calls when the forward stores its tile
    states and the backward reuses them (no recomputed forward inside the
    backward): each call timed alone, in ms per call (CUDA events, the same
    workload and plan as the backward above)."""
    x = inp["x"]
    B, L, D = x.shape
    ts = torch.empty(ops.tile_states_shape(B, L, D), device=dev)
    y = torch.empty_like(x)
    nbytes = ops.mamba_scan_workspace_size(B, L, D, n_chunks_req)
    fws = torch.empty(max(nbytes, 256), device=dev, dtype=torch.uint8)
    args = (x, inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"], inp["Dskip"], inp["conv_w"],
            inp["conv_b"])

    def fwd(tiles):
        ops.mamba_scan_fwd(*args, y=y, workspace=fws, n_chunks=n_chunks_req, return_state=False,
                           tile_states=tiles, stream=stream)

    def bwd():
        ops.mamba_scan_bwd(*args, dy=dy, out=out, workspace=ws, n_chunks=n_chunks_req, tile_states=ts,
                           stream=stream)

    def per_call(fn):
        for _ in range(warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        assert ops.mamba_last_error(stream) == ops.MAMBA_OK
        return e0.elapsed_time(e1) / steps

    fwd_plain = per_call(lambda: fwd(None))
    fwd_tiles = per_call(lambda: fwd(ts))
    bwd_given = per_call(bwd)
    del ts, y, fws
    return {"fwd_ms": fwd_plain, "fwd_storing_tile_states_ms": fwd_tiles,
            "bwd_given_tile_states_ms": bwd_given,
            "note": "tile states (B, L/16, D, 16) fp32 written by the forward and read by the backward, "
                    "which then skips its states-only forward pass"}


def oracle_bwd_sample_rate(w, target_s: float):
    """The fp64 backward oracle on a few channels of the workload (every token
    and batch row): elements/s, extrapolated per channel."""
    import oracle
    oracle.build()
    L = w.seqlen

    def run(ch):
        sub = inputs.ScanWorkload(w.name, w.batch, L, ch, w.io, w.seed, w.bc_std)
        inp = inputs.workload_inputs(sub, device="cpu")
        dy = torch.randn(inp["x"].shape, generator=torch.Generator().manual_seed(1)).to(inp["x"].dtype)
        t0 = time.perf_counter()
        oracle.scan_bwd(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"],
                        inp["Dskip"], inp["conv_w"], inp["conv_b"], dy=dy)
        return time.perf_counter() - t0

    t1 = max(run(1), 1e-3)
    ch = int(max(1, min(w.d_inner, target_s / t1)))
    t = run(ch)
    elems = w.batch * L * ch
    return elems / t, {"kind": "oracle", "cores": 1,
                       "sample": f"{ch} of {w.d_inner} channels x all {L} tokens x batch {w.batch} "
                                 f"({elems} elements, {t:.1f} s, one thread: dB and dC sum over channels)"}


def bf16_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1800.0, 1400.0, "fallback"


def layer_weights(B, L, H, D, R, dev, seed):
    """Seeded layer weights and input: N(0, 1/fan_in) projections (bf16),
    the scan's parameters as in the workload recipe, dt_proj's bias chosen
    so that softplus(bias) is log-uniform in [1e-3, 1e-1]."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    bf = torch.bfloat16

    def n(shape, std):
        return (torch.randn(shape, generator=g, device=dev) * std).to(bf)
    dt = torch.exp(math.log(1e-3) + torch.rand(D, generator=g, device=dev) * (math.log(1e-1) - math.log(1e-3)))
    return dict(hidden=n((B, L, H), 1.0), W_in=n((2 * D, H), H ** -0.5),
                conv_w=torch.rand((D, D_CONV), generator=g, device=dev) - 0.5,
                conv_b=torch.zeros(D, device=dev), W_x=n((R + 32, D), D ** -0.5), W_dt=n((D, R), R ** -0.5),
                b_dt=torch.log(torch.expm1(dt)).to(bf),
                A_log=torch.log(torch.arange(1, D_STATE + 1, device=dev, dtype=torch.float32)).expand(D, D_STATE)
                .contiguous(),
                Dskip=torch.ones(D, device=dev), W_out=n((H, D), D ** -0.5))


def bench_layer(w, steps, warmup, local, n_chunks_req=0, d_model=4096, dt_rank=256):
    """The whole Mamba layer (mamba_layer_fwd): in_proj, conv + SiLU, x_proj,
    dt_proj, the scan and out_proj, at the workload's batch, length and
    d_inner with d_model = d_inner / 2 (expand 2) and dt_rank = d_model / 16."""
    from selective_state_space_118_b300 import ops
    dev = torch.device("cuda", local)
    B, L, D, H, R = w.batch, w.seqlen, w.d_inner, d_model, dt_rank
    p = layer_weights(B, L, H, D, R, dev, w.seed + 2000)
    ws = torch.empty(ops.mamba_layer_workspace_size(B, L, H, D, R, n_chunks_req), device=dev, dtype=torch.uint8)
    out = torch.empty(B, L, H, device=dev, dtype=torch.bfloat16)
    stream = torch.cuda.current_stream(dev)

    def call():
        ops.mamba_layer_fwd(p["hidden"], p["W_in"], p["conv_w"], p["conv_b"], p["W_x"], p["W_dt"], p["b_dt"],
                            p["A_log"], p["Dskip"], p["W_out"], out=out, workspace=ws, n_chunks=n_chunks_req,
                            stream=stream)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    assert ops.mamba_last_error(stream) == ops.MAMBA_OK
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(dev.index) as clk:
        ev[0].record(stream)
        for i in range(steps):
            call()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    t = ev[0].elapsed_time(ev[steps]) / 1e3 / steps
    flops = 2 * B * L * (H * 2 * D + D * (R + 32) + R * D + D * H)
    burst, sustained, src = bf16_peaks()
    n_chunks = ops.mamba_scan_plan(B, L, D, n_chunks_req)["n_chunks"]
    res = {"metric": "layer tokens/s", "value": B * L / t, "unit": "tokens/s",
           "config": {"workload": f"mamba_layer_bf16_b{B}_l{L}_h{H}_d{D}_r{R}", "batch": B, "seqlen": L,
                      "d_model": H, "d_inner": D, "dt_rank": R, "n_chunks": n_chunks,
                      "weights": "seeded N(0, 1/fan_in), bf16"},
           "ms_per_call": t * 1e3, "ms_per_call_min": min(per),
           "roofline": {"bound": "tensor", "achieved": flops / t / 1e12, "peak": sustained, "unit": "TFLOP/s",
                        "frac": flops / t / 1e12 / sustained, "peak_source": f"{src} (sustained: a long step)",
                        "flops_per_call": flops,
                        "note": "projection FLOPs over the whole layer call (the scan and conv included in "
                                "the time); the GEMMs are cuBLASLt"},
           "gpu_launches": (2 if n_chunks == 1 else 3) + 1, "library_gemms_per_call": 5, "clocks": clk.summary()}
    del p, ws, out
    return res


def ssd_algorithmic_bytes(B, L, H, G):
    """Minimum HBM bytes of one Mamba-2 scan call (bf16): x and z read and y
    written once, dt per (token, head), B and C rows per (token, group)."""
    return 3 * B * L * H * 64 * 2 + B * L * H * 2 + 2 * B * L * G * D_STATE * 2


def bench_ssd(w, steps, warmup, local, heads=None, groups=1):
    """Mamba-2's chunked scan (mamba2_scan_fwd) on the workload's batch and
    length, its d_inner cut into heads of 64 channels (Jamba shape: 128
    heads), one group of B and C rows, with the gate; seeded inputs of the
    scan workload's distributions (dt log-uniform per (token, head))."""
    from selective_state_space_118_b300 import ops
    dev = torch.device("cuda", local)
    B, L = w.batch, w.seqlen
    H = heads or w.d_inner // 64
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 3000)
    bf = torch.bfloat16
    x = torch.randn((B, L, H, 64), generator=g, device=dev).to(bf)
    z = torch.randn((B, L, H, 64), generator=g, device=dev).to(bf)
    u = torch.rand((B, L, H), generator=g, device=dev)
    dt_raw = torch.log(torch.expm1(torch.exp(math.log(1e-3) + u * (math.log(1e-1) - math.log(1e-3))))).to(bf)
    Bm = (torch.randn((B, L, groups, D_STATE), generator=g, device=dev) * w.bc_std).to(bf)
    Cm = (torch.randn((B, L, groups, D_STATE), generator=g, device=dev) * w.bc_std).to(bf)
    A_log = torch.log(torch.arange(H, device=dev, dtype=torch.float32) % 16 + 1)
    Dskip = torch.ones(H, device=dev)
    y = torch.empty_like(x)
    fs = torch.empty((B, H, D_STATE, 64), device=dev)
    ws = torch.empty(ops.mamba2_scan_workspace_size(B, L, H), device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)

    def call():
        ops.mamba2_scan_fwd(x, dt_raw, A_log, Bm, Cm, Dskip, z, None, y=y, final_state=fs, workspace=ws,
                            stream=stream)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(dev.index) as clk:
        ev[0].record(stream)
        for i in range(steps):
            call()
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    t = ev[0].elapsed_time(ev[steps]) / 1e3 / steps
    alg = ssd_algorithmic_bytes(B, L, H, groups)
    hbm, src = peaks()
    res = {"metric": "mamba2 scan elements/s", "value": B * L * H * 64 / t, "unit": UNIT,
           "config": {"workload": f"mamba2_scan_bf16_b{B}_l{L}_h{H}_p64_g{groups}_n16", "batch": B, "seqlen": L,
                      "heads": H, "head_dim": 64, "groups": groups, "d_state": D_STATE, "chunk": 64},
           "ms_per_call": t * 1e3, "ms_per_call_min": min(per),
           "roofline": {"bound": "hbm", "achieved": alg / t / 1e9, "peak": hbm, "unit": "GB/s",
                        "frac": alg / t / 1e9 / hbm, "peak_source": src, "algorithmic_bytes_per_call": alg,
                        "note": "whole call (3 kernels); the per-chunk states it writes and reads back are "
                                "not algorithmic bytes"},
           "gpu_launches": 3 * steps, "clocks": clk.summary()}
    del x, z, y, ws
    return res


def bench_decode(w, local, replays=3, layers=None, tokens=None):
    """28 layers x 256 tokens, one mamba_step per layer and token, replayed
    from one CUDA graph.  decode steps/s = tokens (for all 64 sequences
    through all layers) per second."""
    from selective_state_space_118_b300 import ops
    import dataclasses
    if layers or tokens:  # a smaller block of the same workload (profiling)
        w = dataclasses.replace(w, name=f"{w.name}@{layers or w.layers}x{tokens or w.steps}",
                                layers=layers or w.layers, steps=tokens or w.steps)
    dev = torch.device("cuda", local)
    states = [inputs.decode_layer_state(w, l, device=dev) for l in range(w.layers)]
    toks = [inputs.decode_token_inputs(w, l, w.steps, device=dev) for l in range(w.layers)]
    ys = [torch.empty(w.batch, w.d_inner, device=dev, dtype=inputs.torch_dtype(w.io))
          for _ in range(w.layers)]
    stream = torch.cuda.Stream(dev)

    def run_all():
        for t in range(w.steps):
            for l in range(w.layers):
                st, tk = states[l], toks[l]
                ops.mamba_step(st["h"], st["conv_state"], tk["x_t"][t], tk["z_t"][t],
                               tk["dt_raw_t"][t], tk["B_t"][t], tk["C_t"][t], st["A_log"],
                               st["Dskip"], st["conv_w"], st["conv_b"], y_t=ys[l], stream=stream)

    with torch.cuda.stream(stream):
        run_all()  # warm-up, outside the graph
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run_all()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk, torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(replays):
            g.replay()  # replays on the current stream, i.e. `stream`
        e1.record(stream)
        torch.cuda.synchronize(dev)
    t = e0.elapsed_time(e1) / 1e3 / replays
    launches = w.layers * w.steps
    es = 2 if w.io == "bf16" else 4
    alg = decode_algorithmic_bytes(w.batch, w.d_inner, es)
    hbm, src = peaks()
    per_launch = t / launches
    return {"metric": "decode steps/s", "value": w.steps / t, "unit": "steps/s",
            "config": {"workload": w.name, "layers": w.layers, "batch": w.batch,
                       "d_inner": w.d_inner, "tokens": w.steps, "cuda_graph": True},
            "ms_per_token": t * 1e3 / w.steps,
            "roofline": {"bound": "hbm", "achieved": alg / per_launch / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": alg / per_launch / 1e9 / hbm,
                         "traffic": measured_traffic(w.name), "peak_source": src,
                         "note": "per-launch time = graph replay time / launches (gaps included); "
                                 "traffic: ncu DRAM bytes of one step_kernel launch"},
            "gpu_launches": launches * replays, "clocks": clk.summary()}


# ---------------------------------------------------------------- oracle arm
def oracle_sample_rate(w, target_s: float, max_channels: int = 2048):
    """Times the fp64 oracle on an evenly strided subset of channels of the
    workload (exact per channel: channels are independent) for about
    target_s seconds of CPU work; returns elements/s and a description."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    L = w.seqlen
    inp = inputs.workload_inputs(inputs.ScanWorkload(w.name, w.batch, L, 16, w.io, w.seed, w.bc_std),
                                 device="cpu")
    t0 = time.perf_counter()
    oracle.scan(inp["x"][:, :, :1], inp["z"][:, :, :1], inp["dt_raw"][:, :, :1], inp["Bm"],
                inp["Cm"], inp["A_log"][:1], inp["Dskip"][:1], inp["conv_w"][:1], inp["conv_b"][:1],
                n_threads=1)
    per_row = max(time.perf_counter() - t0, 1e-4)
    rows = int(target_s * threads / per_row)
    ch = int(min(max(rows // w.batch, min(threads, w.d_inner)), w.d_inner, max_channels))
    ch = max(ch, 1)
    inp = inputs.workload_inputs(inputs.ScanWorkload(w.name, w.batch, L, ch, w.io, w.seed, w.bc_std),
                                 device="cpu")
    t0 = time.perf_counter()
    oracle.scan(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"],
                inp["Dskip"], inp["conv_w"], inp["conv_b"], n_threads=threads)
    t = time.perf_counter() - t0
    elems = w.batch * L * ch
    return elems / t, {"kind": "oracle", "cores": threads,
                       "sample": f"{ch} of {w.d_inner} channels x all {L} tokens x batch {w.batch} "
                                 f"({elems} elements, {t:.1f} s); elements/s extrapolate exactly "
                                 f"since channels are independent"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    w = workload_of(args)
    vals = []
    desc = None
    for i in range(args.warmup + args.steps):
        v, desc = oracle_sample_rate(w, target_s=2.0, max_channels=256)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": w.batch * w.seqlen * w.d_inner / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, None),
            "cpu_baseline": dict(desc, value=value, unit=UNIT),
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_of(args):
    w = inputs.SCAN_WORKLOADS[args.workload]
    if args.seqlen:
        w = inputs.ScanWorkload(f"{w.name}@L{args.seqlen}", w.batch, args.seqlen, w.d_inner, w.io,
                                w.seed, w.bc_std)
    return w


def config_of(w, n_chunks):
    return {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "d_inner": w.d_inner,
            "d_state": D_STATE, "d_conv": D_CONV, "io": w.io, "n_chunks": n_chunks,
            "l2": "inputs larger than L2 (no flush needed)", "parallelism": "replicas"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=inputs.JAMBA_PREFILL.name, choices=list(inputs.SCAN_WORKLOADS))
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="decode block only (profiling)")
    ap.add_argument("--decode-layers", type=int, default=0, help="fewer decode layers (profiling)")
    ap.add_argument("--decode-tokens", type=int, default=0, help="fewer decode tokens (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--backward-only", action="store_true", help="the backward block alone (profiling)")
    ap.add_argument("--no-layer", action="store_true")
    ap.add_argument("--no-ssd", action="store_true")
    ap.add_argument("--ssd-only", action="store_true", help="the Mamba-2 scan block alone (profiling)")
    ap.add_argument("--layer-only", action="store_true", help="the layer block alone (profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--n-chunks", type=int, default=0,
                    help="chunk count passed to the library (0: its own plan)")
    ap.add_argument("--seqlen", type=int, default=0,
                    help="override the workload's sequence length (smaller cases for profiling)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    from selective_state_space_118_b300 import build, ops
    if rank == 0 and not os.path.exists(ops.LIB_PATH):
        build.build()
    barrier(world)
    if args.no_prefill:
        d = bench_decode(inputs.DECODE, local, layers=args.decode_layers, tokens=args.decode_tokens)
        if rank == 0:
            print(json.dumps(d), flush=True)
        return
    w = workload_of(args)
    if args.backward_only:
        b = bench_backward(w, args.steps, args.warmup, local, args.n_chunks)
        if rank == 0:
            print(json.dumps(b), flush=True)
        return
    if args.ssd_only:
        b = bench_ssd(w, args.steps, args.warmup, local)
        if rank == 0:
            print(json.dumps(b), flush=True)
        return
    if args.layer_only:
        b = bench_layer(w, args.steps, args.warmup, local, args.n_chunks)
        if rank == 0:
            print(json.dumps(b), flush=True)
        return
    res, inp, out, ws = bench_prefill(w, args.steps, args.warmup, world, local, args.n_chunks)
    value = job_value(res["elems"], args.steps, world, res["t_ms"])
    hbm, src = peaks()
    achieved = res["alg_bytes"] / (res["per_launch_ms"] / 1e3) / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["t_ms"] / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.io,
            "data": "synthetic", "config": dict(config_of(w, res["n_chunks"]), plan=res["plan"]),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": measured_traffic(w.name), "peak_source": src,
                         "kernel": "mamba_scan_fwd: bc_widen + scan_carry + scan_fwd (one call)",
                         "algorithmic_bytes_per_launch": res["alg_bytes"]},
            "gpu_launches": res["launches_per_step"] * args.steps,
            "clocks": res["clocks"]}
    if not args.no_e2e:
        e2e = bench_e2e(w, inp, out, ws, max(4, min(args.steps, 8)), local)
        t = max_over_ranks(e2e.pop("t"), world)
        e2e = dict(value=res["elems"] * e2e["steps"] * world / t, **e2e)
        line["e2e"] = e2e
    del inp, out, ws
    torch.cuda.empty_cache()
    if not args.no_decode:
        line["decode"] = bench_decode(inputs.DECODE, local, layers=args.decode_layers,
                                      tokens=args.decode_tokens)
        torch.cuda.empty_cache()
    if not args.no_ssd:
        line["mamba2"] = bench_ssd(w, max(3, min(args.steps, 20)), 3, local)
        torch.cuda.empty_cache()
    if not args.no_layer:
        line["layer"] = bench_layer(w, max(3, min(args.steps, 20)), 3, local, args.n_chunks)
        torch.cuda.empty_cache()
    if not args.no_backward:
        line["backward"] = bench_backward(w, max(3, min(args.steps, 20)), 3, local, args.n_chunks)
        torch.cuda.empty_cache()
        if rank == 0 and not args.no_cpu_baseline and world == 1:
            v, desc = oracle_bwd_sample_rate(w, target_s=4.0)
            line["backward"]["cpu_baseline"] = dict(desc, value=v, unit=UNIT)
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        v, desc = oracle_sample_rate(w, target_s=10.0, max_channels=w.d_inner)
        line["cpu_baseline"] = dict(desc, value=v, unit=UNIT)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
