#!/usr/bin/env python
"""Benchmark of the selective-scan library on synthetic Jamba-shaped inputs.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--seqlen L] [--n-chunks K]
                [--no-e2e] [--no-cpu-baseline] [--no-decode] [--no-ssd]
                [--no-layer] [--no-backward] [--no-complex] [--no-extra-prefill]
                [--no-prefill | --prefill-only | --backward-only | --layer-only | --ssd-only |
                 --complex-only]

A step is one prefill of the layer's scan (conv, SiLU, softplus, discretised
scan, D skip, SiLU(z) gate; final h and conv state) over the workload's whole
sequence, through the C ABI, inputs resident in HBM (larger than L2).  The
default workload is the 256k-token context (1 x 262,144 tokens x 8,192
channels, bf16) fed as 64 consecutive calls of 4,096 tokens, each carrying
the state of the one before.  Prints one JSON line on rank 0.  Under torchrun every rank runs an independent
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
def prefill_slices(w):
    """The calls of one step: the workload's sequence cut into host_chunks
    consecutive calls ((t0, t1) token ranges), or one call."""
    n = max(1, w.host_chunks)
    step = (w.seqlen + n - 1) // n
    return [(t0, min(t0 + step, w.seqlen)) for t0 in range(0, w.seqlen, step)]


def prefill_step(ops, inp, out, ws, stream, slices, n_chunks=0):
    """One step: one mamba_scan_fwd per slice, each carrying the previous
    call's final state and conv state in as its initial ones (final_h and
    final_conv_state alias h0 and conv_state0); the first call starts from
    zero.  Slices of a batch-1 tensor along the sequence are contiguous."""
    one = len(slices) == 1
    for i, (t0, t1) in enumerate(slices):
        def part(k):
            return inp[k] if one else inp[k][:, t0:t1]
        ops.mamba_scan_fwd(part("x"), part("z"), part("dt_raw"), part("Bm"), part("Cm"), inp["A_log"],
                           inp["Dskip"], inp["conv_w"], inp["conv_b"], out["fh"] if i else None,
                           out["fcs"] if i else None, y=out["y"] if one else out["y"][:, t0:t1],
                           final_h=out["fh"], final_conv_state=out["fcs"], workspace=ws, n_chunks=n_chunks,
                           stream=stream)


def scan_launches(ops, B, L, D, n_chunks_req):
    """Kernels one mamba_scan_fwd launches: B/C widening, then the main pass
    (one chunk) or the chunk carries and the main pass in one launch."""
    return 2


def mufu_peak():
    """MUFU slots per second of the whole GPU: 32 ex2 results per clock per SM
    (measured by a throughput probe on this B300) at the maximum SM clock."""
    mhz = 2032.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    except Exception:
        pass
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148
    return 32.0 * sms * mhz * 1e6, f"32 ex2/clk/SM x {sms} SMs x {mhz:.0f} MHz"


# MUFU slots per prefill element (b, t, c): 16 state decays 2^(dt A2), the
# exponentials of the two SiLUs and of softplus (ex2, one slot each) and the
# SiLUs' two reciprocals (rcp, two slots each: 16 results per clock per SM).
MUFU_SLOTS_PER_ELEMENT = 16 + 3 + 2 * 2


# The complex scan's: per mode (8 of them) the decay's ex2 and the turn's sin
# and cos, plus the SiLUs' and softplus' three ex2 and two reciprocals.
COMPLEX_MUFU_SLOTS_PER_ELEMENT = 8 * 3 + 3 + 2 * 2


def compute_roofline(elems_per_s, elems_per_step, t_step_s, slots=MUFU_SLOTS_PER_ELEMENT,
                     note="the exponentials alone bound the scan below the HBM roofline: "
                          "16 decays per element need 16 MUFU slots for 8 bytes"):
    peak, how = mufu_peak()
    achieved = elems_per_s * slots
    return {"bound": "alu", "what": "MUFU (special-function unit)", "achieved": achieved, "peak": peak,
            "unit": "MUFU slots/s", "frac": achieved / peak, "peak_source": how,
            "slots_per_element": slots,
            "floor_ms_per_step": elems_per_step * slots / peak * 1e3,
            "note": note}


# The backward's instruction mix, measured by ncu on the reverse-sweep kernel
# (L = 4096, the Jamba width): warp-instructions per warp-token (one warp, its
# 32 channels, one token) and the MUFU share of them.
BWD_WARP_INSTR_PER_WARP_TOKEN = 457
BWD_MUFU_SHARE = 0.12


def bwd_compute_floor(elems, t_s):
    """Two floors of the backward at its measured instruction mix: issue (one
    warp-instruction per scheduler per clock, four schedulers per SM) and the
    MUFU's (its instructions at 16 per clock per SM, the reciprocal's rate;
    ex2 runs at twice that)."""
    sms, mhz = 148, 2032.0
    try:
        props = torch.cuda.get_device_properties(torch.cuda.current_device())
        sms = props.multi_processor_count
    except Exception:
        pass
    per_elem = BWD_WARP_INSTR_PER_WARP_TOKEN / 32.0  # warp-instructions per element
    issue_s = elems * per_elem / (4 * sms * mhz * 1e6)
    mufu_s = elems * per_elem * BWD_MUFU_SHARE * 32 / (16 * sms * mhz * 1e6)
    return {"what": "issue and MUFU floors at the measured instruction mix",
            "warp_instructions_per_warp_token": BWD_WARP_INSTR_PER_WARP_TOKEN, "mufu_share": BWD_MUFU_SHARE,
            "issue_floor_ms": issue_s * 1e3, "issue_frac": issue_s / t_s,
            "mufu_floor_ms": mufu_s * 1e3, "mufu_frac": mufu_s / t_s,
            "sm_clock_mhz_assumed": mhz}


def bench_prefill(w, steps, warmup, world, local, n_chunks_req=0, inp=None, slices=None):
    from selective_state_space_118_b300 import ops
    dev = torch.device("cuda", local)
    if inp is None:
        inp = inputs.workload_inputs(w, device=dev)
    B, L, D = w.batch, w.seqlen, w.d_inner
    slices = slices or prefill_slices(w)
    assert B == 1 or len(slices) == 1, "carried calls slice a batch-1 sequence"
    es = 2 if w.io == "bf16" else 4
    out = {"y": torch.empty_like(inp["x"]),
           "fh": torch.empty(B, D, D_STATE, device=dev),
           "fcs": torch.empty(B, D_CONV - 1, D, device=dev, dtype=inp["x"].dtype)}
    nbytes = max(ops.mamba_scan_workspace_size(B, t1 - t0, D, n_chunks_req) for t0, t1 in slices)
    ws = torch.empty(max(nbytes, 1), device=dev, dtype=torch.uint8) if nbytes else None
    plans = sorted({(t1 - t0) for t0, t1 in slices})
    plan = {str(l): ops.mamba_scan_plan(B, l, D, n_chunks_req) for l in plans}
    launches = sum(scan_launches(ops, B, t1 - t0, D, n_chunks_req) for t0, t1 in slices)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        prefill_step(ops, inp, out, ws, stream, slices, n_chunks_req)
    torch.cuda.synchronize(dev)
    assert ops.mamba_last_error(stream) == ops.MAMBA_OK
    barrier(world)
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with ClockSampler(dev.index) as clk:
        ev[0].record(stream)
        for i in range(steps):
            prefill_step(ops, inp, out, ws, stream, slices, n_chunks_req)
            ev[i + 1].record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    assert ops.mamba_last_error(stream) == ops.MAMBA_OK
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    t_total_ms = ev[0].elapsed_time(ev[steps])
    t_max_ms = max_over_ranks(t_total_ms, world)
    elems = B * L * D
    alg = scan_algorithmic_bytes(B, L, D, es)
    res = dict(elems=elems, t_ms=t_max_ms, per_step_ms=statistics.mean(per),
               per_step_min_ms=min(per), alg_bytes=alg, plan=plan, calls_per_step=len(slices),
               launches_per_step=launches, clocks=clk.summary(),
               in_bytes=sum(inp[k].numel() * inp[k].element_size()
                            for k in ("x", "z", "dt_raw", "Bm", "Cm")),
               out_bytes=out["y"].numel() * out["y"].element_size())
    return res, inp, out, ws


def prefill_block(w, steps, warmup, local, n_chunks_req=0, slices=None):
    """A secondary prefill measurement (its own inputs and timing) as a JSON
    object: elements/s, ms per step and the two rooflines."""
    res, inp, out, ws = bench_prefill(w, steps, warmup, 1, local, n_chunks_req, slices=slices)
    del inp, out, ws
    t = res["per_step_ms"] / 1e3
    hbm, src = peaks()
    achieved = res["alg_bytes"] / t / 1e9
    return {"metric": "prefill elements/s", "value": res["elems"] / t, "unit": UNIT,
            "config": dict(config_of(w, None), calls_per_step=res["calls_per_step"], plan=res["plan"]),
            "ms_per_step": res["per_step_ms"], "ms_per_step_min": res["per_step_min_ms"],
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_source": src,
                         "algorithmic_bytes_per_step": res["alg_bytes"],
                         "compute": compute_roofline(res["elems"] / t, res["elems"], t)},
            "gpu_launches": res["launches_per_step"] * steps, "clocks": res["clocks"]}


def bench_e2e(w, inp, out, ws, steps, local, slices):
    """Same metric through the C ABI with the inputs in pinned HOST memory:
    every step copies x, z, dt_raw, B, C host->device, scans, and copies y
    device->host, all inside the timed region.  The copies and the scans are
    pipelined over the step's calls (one per slice of the sequence, state
    carried from call to call), the way a serving loop would stream a long
    prompt: uploads on one stream, the scans on another, downloads on a
    third, with two device buffer sets, so that slice i+1's upload and slice
    i-1's download overlap slice i's scan (the host link's two directions
    work at the same time).  With one slice per step, consecutive steps are
    independent requests pipelined the same way."""
    from selective_state_space_118_b300 import ops
    dev = torch.device("cuda", local)
    names = ("x", "z", "dt_raw", "Bm", "Cm")
    host = {k: torch.empty(inp[k].shape, dtype=inp[k].dtype, pin_memory=True) for k in names}
    for k in host:
        host[k].copy_(inp[k])
    y_host = torch.empty(out["y"].shape, dtype=out["y"].dtype, pin_memory=True)
    one = len(slices) == 1
    n_sets = 2
    lmax = max(t1 - t0 for t0, t1 in slices)

    def dev_slice(t, l):
        return t if one else t[:, :l]
    bufs = [{k: torch.empty((inp[k].shape[0], lmax) + tuple(inp[k].shape[2:]), dtype=inp[k].dtype, device=dev)
             for k in names} for _ in range(n_sets)]
    ybufs = [torch.empty((out["y"].shape[0], lmax, out["y"].shape[2]), dtype=out["y"].dtype, device=dev)
             for _ in range(n_sets)]
    up, comp, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    uploaded = [torch.cuda.Event() for _ in range(n_sets)]
    scanned = [torch.cuda.Event() for _ in range(n_sets)]
    downloaded = [torch.cuda.Event() for _ in range(n_sets)]
    for e in scanned:
        e.record(comp)
    for e in downloaded:
        e.record(down)
    seq = [0]

    def step():
        for i, (t0, t1) in enumerate(slices):
            s = seq[0] % n_sets
            seq[0] += 1
            l = t1 - t0
            up.wait_event(scanned[s])  # input set s is free once the scan that read it is done
            with torch.cuda.stream(up):
                for k in names:
                    src = host[k] if one else host[k][:, t0:t1]
                    dev_slice(bufs[s][k], l).copy_(src, non_blocking=True)
            uploaded[s].record(up)
            comp.wait_event(uploaded[s])
            comp.wait_event(downloaded[s])  # y set s is free once its last slice left
            sl = {k: dev_slice(bufs[s][k], l) for k in names}
            ys = dev_slice(ybufs[s], l)
            ops.mamba_scan_fwd(sl["x"], sl["z"], sl["dt_raw"], sl["Bm"], sl["Cm"], inp["A_log"], inp["Dskip"],
                               inp["conv_w"], inp["conv_b"], out["fh"] if i else None, out["fcs"] if i else None,
                               y=ys, final_h=out["fh"], final_conv_state=out["fcs"], workspace=ws, stream=comp)
            scanned[s].record(comp)
            down.wait_event(scanned[s])
            with torch.cuda.stream(down):
                (y_host if one else y_host[:, t0:t1]).copy_(ys, non_blocking=True)
            downloaded[s].record(down)

    step()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize(dev)
    t = time.perf_counter() - t0
    bi = sum(h.numel() * h.element_size() for h in host.values())
    bo = y_host.numel() * y_host.element_size()

    # the host link alone, outside the timed region: one step's uploads, its
    # downloads, and both at once (on their two streams), as the same copies
    # with nothing else running
    def link(directions):
        torch.cuda.synchronize(dev)
        t0_wall = time.perf_counter()
        for i, (t0_, t1_) in enumerate(slices):
            s = i % n_sets
            l = t1_ - t0_
            if "h2d" in directions:
                with torch.cuda.stream(up):
                    for k in names:
                        dev_slice(bufs[s][k], l).copy_(host[k] if one else host[k][:, t0_:t1_], non_blocking=True)
            if "d2h" in directions:
                with torch.cuda.stream(down):
                    (y_host if one else y_host[:, t0_:t1_]).copy_(dev_slice(ybufs[s], l), non_blocking=True)
        torch.cuda.synchronize(dev)
        moved = (bi if "h2d" in directions else 0) + (bo if "d2h" in directions else 0)
        return moved / (time.perf_counter() - t0_wall) / 1e9
    h2d, d2h, both = link(("h2d",)), link(("d2h",)), link(("h2d", "d2h"))
    res = {"t": t, "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
           "steps": steps, "ms_per_step": t * 1e3 / steps,
           "pipelining": f"uploads / scans / downloads on three streams, two buffer sets, "
                         f"{len(slices)} call(s) per step",
           "host_link": {"h2d_gbs": h2d, "d2h_gbs": d2h, "both_gbs": both,
                         "floor_ms_per_step": (bi + bo) / both / 1e6,
                         "note": "one step's copies alone (the same pinned buffers and calls), "
                                 "each direction by itself and both at once; the two directions "
                                 "share the link, so a step moving both cannot beat floor_ms_per_step"}}
    del host, y_host, bufs, ybufs
    return res


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
                        "compute": bwd_compute_floor(B * L * D, t),
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
    gemms = compare_gemms(ops, B * L, H, D, R, dev, stream, max(3, steps))
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
                                "the time); the GEMMs are the library's tcgen05 GEMM"},
           "gemms": gemms,
           "gpu_launches": ((2 if n_chunks == 1 else 3) + 1 + 5) * steps, "clocks": clk.summary()}
    del p, ws, out
    return res


def compare_gemms(ops, M, H, D, R, dev, stream, reps):
    """The layer's five projection shapes timed alone through the library's
    tcgen05 GEMM (mamba_linear_fwd) and through cuBLAS (torch's linear, for
    comparison only), ms per GEMM and TFLOP/s, on seeded operands."""
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    bf = torch.bfloat16
    out = {}
    # (name, M, N, K, bias)
    for name, N, K, bias in (("in_proj_x", D, H, False), ("in_proj_z", D, H, False), ("x_proj", R + 32, D, False),
                             ("dt_proj", D, R, True), ("out_proj", H, D, False)):
        A = torch.randn((M, K), generator=g, device=dev).to(bf)
        W = (torch.randn((N, K), generator=g, device=dev) * K ** -0.5).to(bf)
        b = torch.randn((N,), generator=g, device=dev).to(bf) if bias else None
        C = torch.empty((M, N), device=dev, dtype=bf)
        res = {}
        for impl, fn in (("tcgen05", lambda: ops.mamba_linear_fwd(A, W, b, out=C, stream=stream)),
                         ("cublas", lambda: torch.nn.functional.linear(A, W, b, out=C))):
            for _ in range(3):
                fn()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(torch.cuda.current_stream(dev))
            for _ in range(reps):
                fn()
            e1.record(torch.cuda.current_stream(dev))
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1) / reps
            res[impl] = {"ms": ms, "tflops": 2 * M * N * K / ms / 1e9}
        res["shape"] = [M, N, K]
        res["tcgen05_vs_cublas_time"] = res["cublas"]["ms"] / res["tcgen05"]["ms"]
        out[name] = res
        del A, W, C
    return out


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
                      "heads": H, "head_dim": 64, "groups": groups, "d_state": D_STATE, "chunk": 128},
           "ms_per_call": t * 1e3, "ms_per_call_min": min(per),
           "roofline": {"bound": "hbm", "achieved": alg / t / 1e9, "peak": hbm, "unit": "GB/s",
                        "frac": alg / t / 1e9 / hbm, "peak_source": src, "algorithmic_bytes_per_call": alg,
                        "note": "whole call (3 kernels); the per-chunk states it writes and reads back are "
                                "not algorithmic bytes"},
           "gpu_launches": 3 * steps, "clocks": clk.summary()}
    del x, z, y, ws
    return res


def bench_complex(w, steps, warmup, local, trapezoidal, n_chunks_req=0):
    """The complex-valued scan (mamba3_scan_fwd, Mamba-3's state update) on the
    workload's shapes and distributions (8 complex modes per channel, A_log =
    log(n+1), theta = pi n): elements/s and its HBM roofline."""
    from selective_state_space_118_b300 import ops
    dev = torch.device("cuda", local)
    inp = inputs.complex_scan_inputs(w.batch, w.seqlen, w.d_inner, w.io, w.seed, w.bc_std, device=dev)
    B, L, D = w.batch, w.seqlen, w.d_inner
    es = 2 if w.io == "bf16" else 4
    y = torch.empty_like(inp["x"])
    fh = torch.empty(B, D, D_STATE, device=dev)
    fv = torch.empty(B, D, D_STATE, device=dev)
    fcs = torch.empty(B, D_CONV - 1, D, device=dev, dtype=inp["x"].dtype)
    ws = torch.empty(max(ops.mamba3_scan_workspace_size(B, L, D, n_chunks_req), 256), device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)

    def call():
        ops.mamba3_scan_fwd(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"], inp["theta"],
                            inp["Dskip"], inp["conv_w"], inp["conv_b"], trapezoidal=trapezoidal, y=y, final_h=fh,
                            final_conv_state=fcs, final_v=fv, workspace=ws, n_chunks=n_chunks_req, stream=stream)

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
    # the real scan's minimum bytes plus theta and the state input out (fp32)
    alg = scan_algorithmic_bytes(B, L, D, es) + D * 8 * 4 + B * D * D_STATE * 4
    hbm, src = peaks()
    ws_big = ops.mamba3_scan_workspace_size(B, L, D, n_chunks_req) > ops.mamba3_scan_workspace_size(B, L, D, 1)
    res = {"metric": "complex scan elements/s", "value": B * L * D / t, "unit": UNIT,
           "config": {"workload": f"{w.name}_complex8", "batch": B, "seqlen": L, "d_inner": D, "modes": 8,
                      "discretization": "trapezoidal" if trapezoidal else "euler", "chunked": ws_big,
                      "theta": "pi * n", "A_log": "log(n + 1)"},
           "ms_per_call": t * 1e3, "ms_per_call_min": min(per),
           "roofline": {"bound": "hbm", "achieved": alg / t / 1e9, "peak": hbm, "unit": "GB/s",
                        "frac": alg / t / 1e9 / hbm, "peak_source": src, "algorithmic_bytes_per_call": alg,
                        "compute": compute_roofline(
                            B * L * D / t, B * L * D, t, COMPLEX_MUFU_SLOTS_PER_ELEMENT,
                            "per element 8 ex2 + 8 sin + 8 cos for the modes' decays and turns, plus the "
                            "SiLUs and softplus; the kernel is issue- and latency-bound below this floor"),
                        "note": "compute: the MUFU floor; bytes: far below the HBM roofline"},
           "gpu_launches": (4 if ws_big else 2) * steps, "clocks": clk.summary()}
    del inp, y, ws
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
def sample_channels(D: int, n: int) -> list:
    """n channels evenly strided over [0, D)."""
    n = max(1, min(n, D))
    return sorted({int(round(i * (D - 1) / max(n - 1, 1))) for i in range(n)})


def host_sample(inp, channels):
    """The inputs of some channels (B, C rows whole: they are per token), on the host."""
    idx = torch.as_tensor(channels, device=inp["x"].device)
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        elif k in ("Bm", "Cm"):
            out[k] = v.cpu()
        elif k in ("x", "z", "dt_raw"):
            out[k] = v.index_select(2, idx).cpu()
        else:
            out[k] = v.index_select(0, idx).cpu()
    return out


def oracle_seconds_per_channel(w, threads: int) -> float:
    """Wall time of the fp64 oracle per channel of the workload (every token
    and batch row) with `threads` host threads, from a short timed run."""
    import oracle
    oracle.build()
    n = max(1, threads)
    inp = inputs.workload_inputs(inputs.ScanWorkload(w.name, w.batch, w.seqlen, n, w.io, w.seed, w.bc_std),
                                 device="cpu")
    t0 = time.perf_counter()
    oracle.scan(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"], inp["Dskip"],
                inp["conv_w"], inp["conv_b"], n_threads=threads)
    return max(time.perf_counter() - t0, 1e-4) / n


def rel_errors(gpu, ref, rounded_bf16: bool):
    """(plain, after the half-ulp allowance of a bf16 output) max|gpu - oracle| / rms(oracle)."""
    g = gpu.double().numpy()
    err = np.abs(g - ref)
    rms = float(np.sqrt(np.mean(ref * ref))) or 1.0
    plain = float(err.max()) / rms
    arith = float(np.maximum(err - 2.0 ** -8 * np.abs(ref), 0.0).max()) / rms if rounded_bf16 else plain
    return plain, arith


def oracle_baseline(w, target_s: float, sample=None, gpu_out=None):
    """The fp64 oracle on all host threads, on an evenly strided subset of the
    workload's channels (every token and batch row; exact per channel since
    channels are independent), sized for about target_s seconds: elements/s
    and a description.  Given the GPU's inputs and outputs (`sample`: the
    device inputs, `gpu_out`: y and final_h of the timed run), the sample is
    those channels of the very inputs the GPU scanned, and the GPU's outputs
    on them are compared with the oracle's (plain and after the bf16
    allowance: max |gpu - oracle| / rms(oracle))."""
    import oracle
    threads = os.cpu_count() or 1
    per_ch = oracle_seconds_per_channel(w, threads)
    ch = int(min(w.d_inner, max(threads, target_s / per_ch)))
    chans = sample_channels(w.d_inner, ch)
    if sample is not None:
        inp = host_sample(sample, chans)
    else:
        inp = inputs.workload_inputs(inputs.ScanWorkload(w.name, w.batch, w.seqlen, len(chans), w.io, w.seed,
                                                         w.bc_std), device="cpu")
    t0 = time.perf_counter()
    yr, fhr, _ = oracle.scan(inp["x"], inp["z"], inp["dt_raw"], inp["Bm"], inp["Cm"], inp["A_log"],
                             inp["Dskip"], inp["conv_w"], inp["conv_b"], n_threads=threads)
    t = time.perf_counter() - t0
    elems = w.batch * w.seqlen * len(chans)
    desc = {"kind": "oracle", "cores": threads,
            "sample": f"{len(chans)} of {w.d_inner} channels (evenly strided) x all {w.seqlen} tokens x batch "
                      f"{w.batch} ({elems} elements, {t:.1f} s, {threads} threads); elements/s extrapolate "
                      f"exactly since channels are independent",
            "sample_elements": elems, "sample_seconds": t}
    if gpu_out is not None:
        idx = torch.as_tensor(chans, device=gpu_out["y"].device)
        yp, ya = rel_errors(gpu_out["y"].index_select(2, idx).cpu(), yr, w.io == "bf16")
        hp, _ = rel_errors(gpu_out["fh"].index_select(1, idx).cpu(), fhr, False)
        desc["parity"] = {"channels": len(chans), "y_plain": yp, "y_after_bf16_allowance": ya,
                          "final_h_plain": hp, "tolerance": 1e-2 if w.io == "bf16" else 1e-4,
                          "metric": "max|gpu - oracle| / rms(oracle) on the sampled channels; the "
                                    "allowance subtracts each bf16 output's own half-ulp rounding first"}
    return elems / t, desc


def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle, as it stands, on the host cores.
    Each step times the oracle on one bounded sample of the workload (a few
    channels, every token); ms_per_step and the elements of a step describe
    that sample, value is its rate (exact per channel)."""
    if rank != 0:
        return
    import oracle
    w = workload_of(args)
    threads = os.cpu_count() or 1
    per_ch = oracle_seconds_per_channel(w, threads)
    ch = int(min(w.d_inner, max(threads, 2.0 / per_ch)))
    chans = sample_channels(w.d_inner, ch)
    inp = inputs.workload_inputs(inputs.ScanWorkload(w.name, w.batch, w.seqlen, len(chans), w.io, w.seed,
                                                     w.bc_std), device="cpu")
    slices = prefill_slices(w)

    def step():
        # the workload's own calls: consecutive slices carrying the state
        h = cs = None
        for t0, t1 in slices:
            sub = {k: inp[k][:, t0:t1] for k in ("x", "z", "dt_raw", "Bm", "Cm")}
            _, h, cs = oracle.scan(sub["x"], sub["z"], sub["dt_raw"], sub["Bm"], sub["Cm"], inp["A_log"],
                                   inp["Dskip"], inp["conv_w"], inp["conv_b"], h, cs, n_threads=threads)

    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        step()
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    elems = w.batch * w.seqlen * len(chans)
    t = statistics.mean(times)
    value = elems / t
    desc = {"kind": "oracle", "cores": threads,
            "sample": f"each step: {len(chans)} of {w.d_inner} channels (evenly strided) x all {w.seqlen} "
                      f"tokens x batch {w.batch} in the workload's {len(slices)} carried call(s) "
                      f"({elems} elements, {threads} threads); elements/s extrapolate exactly since channels "
                      f"are independent"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "elements_per_step": elems,
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
    cfg = {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "d_inner": w.d_inner,
           "d_state": D_STATE, "d_conv": D_CONV, "io": w.io, "n_chunks": n_chunks,
           "l2": "inputs larger than L2 (no flush needed)", "parallelism": "replicas"}
    if w.host_chunks > 1:
        cfg["calls_per_step"] = w.host_chunks
        cfg["tokens_per_call"] = (w.seqlen + w.host_chunks - 1) // w.host_chunks
        cfg["carry"] = "each call's final_h / final_conv_state are the next call's h0 / conv_state0"
    return cfg


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=inputs.PREFILL_256K.name, choices=list(inputs.SCAN_WORKLOADS))
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="decode block only (profiling)")
    ap.add_argument("--decode-layers", type=int, default=0, help="fewer decode layers (profiling)")
    ap.add_argument("--decode-tokens", type=int, default=0, help="fewer decode tokens (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--backward-only", action="store_true", help="the backward block alone (profiling)")
    ap.add_argument("--no-layer", action="store_true")
    ap.add_argument("--no-ssd", action="store_true")
    ap.add_argument("--no-complex", action="store_true")
    ap.add_argument("--complex-only", action="store_true",
                    help="the complex-valued scan blocks alone (profiling)")
    ap.add_argument("--no-extra-prefill", action="store_true",
                    help="skip the secondary prefill blocks (one-call 256k, 32k workload)")
    ap.add_argument("--ssd-only", action="store_true", help="the Mamba-2 scan block alone (profiling)")
    ap.add_argument("--layer-only", action="store_true", help="the layer block alone (profiling)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="the headline prefill alone, no e2e or other blocks (profiling)")
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
    # the per-token rows of the secondary blocks: the Jamba-shaped 32k layer
    w32 = inputs.JAMBA_PREFILL if args.seqlen == 0 else w
    if args.backward_only:
        b = bench_backward(w32, args.steps, args.warmup, local, args.n_chunks)
        if rank == 0:
            print(json.dumps(b), flush=True)
        return
    if args.ssd_only:
        b = bench_ssd(w32, args.steps, args.warmup, local)
        if rank == 0:
            print(json.dumps(b), flush=True)
        return
    if args.complex_only:
        b = {rule: bench_complex(w32, args.steps, args.warmup, local, rule == "trapezoidal", args.n_chunks)
             for rule in ("euler", "trapezoidal")}
        if rank == 0:
            print(json.dumps(b), flush=True)
        return
    if args.layer_only:
        b = bench_layer(w32, args.steps, args.warmup, local, args.n_chunks)
        if rank == 0:
            print(json.dumps(b), flush=True)
        return
    slices = prefill_slices(w)
    res, inp, out, ws = bench_prefill(w, args.steps, args.warmup, world, local, args.n_chunks, slices=slices)
    value = job_value(res["elems"], args.steps, world, res["t_ms"])
    hbm, src = peaks()
    t_step = res["per_step_ms"] / 1e3
    achieved = res["alg_bytes"] / t_step / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["t_ms"] / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.io,
            "data": "synthetic", "config": dict(config_of(w, None), plan=res["plan"]),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "traffic": measured_traffic(w.name), "peak_source": src,
                         "kernel": f"mamba_scan_fwd x {res['calls_per_step']} calls per step "
                                   f"(bc_widen + scan_fused each), CUDA events around the step",
                         "algorithmic_bytes_per_step": res["alg_bytes"],
                         "compute": compute_roofline(res["elems"] / t_step, res["elems"], t_step)},
            "gpu_launches": res["launches_per_step"] * args.steps,
            "clocks": res["clocks"]}
    if not args.no_e2e and not args.prefill_only:
        try:
            e2e = bench_e2e(w, inp, out, ws, 3 if w.host_chunks > 1 else max(4, min(args.steps, 8)), local,
                            slices)
            t = max_over_ranks(e2e.pop("t"), world)
            line["e2e"] = dict(value=res["elems"] * e2e["steps"] * world / t, **e2e)
        except RuntimeError as e:  # pinned host memory refused: say so, do not guess
            line["e2e"] = {"value": None, "unit": UNIT, "error": f"{type(e).__name__}: {e}"[:300]}
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline and world == 1 and not args.prefill_only:
        v, desc = oracle_baseline(w, target_s=10.0, sample=inp, gpu_out=out)
        line["cpu_baseline"] = dict(desc, value=v, unit=UNIT)
    del inp, out, ws
    torch.cuda.empty_cache()
    if args.prefill_only:
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if not args.no_extra_prefill and args.seqlen == 0:
        if w.host_chunks > 1:
            one = inputs.ScanWorkload(w.name + "_one_call", w.batch, w.seqlen, w.d_inner, w.io, w.seed, w.bc_std)
            line["prefill_one_call"] = prefill_block(one, max(3, min(args.steps, 5)), 3, local, args.n_chunks)
            torch.cuda.empty_cache()
        if w.name != inputs.JAMBA_PREFILL.name:
            line["prefill_32k"] = prefill_block(inputs.JAMBA_PREFILL, max(3, min(args.steps, 20)), 3, local,
                                                args.n_chunks)
            torch.cuda.empty_cache()
    if not args.no_decode:
        line["decode"] = bench_decode(inputs.DECODE, local, layers=args.decode_layers,
                                      tokens=args.decode_tokens)
        torch.cuda.empty_cache()
    if not args.no_ssd:
        line["mamba2"] = bench_ssd(w32, max(3, min(args.steps, 20)), 3, local)
        torch.cuda.empty_cache()
    if not args.no_complex:
        line["complex"] = {rule: bench_complex(w32, max(3, min(args.steps, 20)), 3, local, rule == "trapezoidal")
                           for rule in ("euler", "trapezoidal")}
        torch.cuda.empty_cache()
    if not args.no_layer:
        line["layer"] = bench_layer(w32, max(3, min(args.steps, 20)), 3, local, args.n_chunks)
        torch.cuda.empty_cache()
    if not args.no_backward:
        line["backward"] = bench_backward(w32, max(3, min(args.steps, 20)), 3, local, args.n_chunks)
        torch.cuda.empty_cache()
        if rank == 0 and not args.no_cpu_baseline and world == 1:
            v, desc = oracle_bwd_sample_rate(w32, target_s=4.0)
            line["backward"]["cpu_baseline"] = dict(desc, value=v, unit=UNIT)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
