"""fp64 CPU oracle of the Mamba selective-scan layer -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg and
reference arm of ``bench.py`` may import this package.  The library under
``selective_state_space_118_b300`` never imports it, and it imports nothing
from the library: the two share no code.

The arithmetic lives in ``mamba_oracle.c`` (plain sequential fp64 loops; see
its header for the definition and the page sections it follows).  This module
only compiles that file with gcc, converts arrays to contiguous fp64 and calls
it through ctypes.

Functions
---------
scan(...)          sequential scan over a whole sequence (prefill)
scan_chunked(...)  the same scan evaluated chunk by chunk with a carried,
                   decayed chunk state (checks the chunked decomposition)
step(...)          one decode token, state updated in place
scan_bwd(...)      gradients of sum(y*dy) (+ final-state terms) w.r.t. every
                   input of scan(...)
ssd(...)           Mamba-2's scan: heads of P channels sharing one scalar
                   decay per token, an N x P state per head
layer(...)         the whole Mamba layer: the projections (numpy matmuls in
                   fp64) around scan(...), with every stored intermediate
                   rounded to bf16 where the library stores it
m3_scan(...)       the complex-valued scan (Mamba-3's state update, Euler or
                   exponential-trapezoidal; ``mamba3_oracle.c``)
m3_core(...)       its bare recurrence on one row, given u and dt directly
build()            compile ``liboracle.so`` and ``liboracle_m3.so`` next to
                   this file
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mamba_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_SRC_M3 = os.path.join(_HERE, "mamba3_oracle.c")
_LIB_M3_PATH = os.path.join(_HERE, "liboracle_m3.so")
_lib = None
_lib_m3 = None
_lock = threading.Lock()

_P = ctypes.POINTER(ctypes.c_double)


def _compile(src: str, lib: str, force: bool) -> str:
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= os.path.getmtime(src):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
           "-Wall", "-Wextra", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def build(force: bool = False) -> str:
    """Compile mamba_oracle.c into liboracle.so and mamba3_oracle.c into
    liboracle_m3.so (gcc, -O2, OpenMP)."""
    _compile(_SRC_M3, _LIB_M3_PATH, force)
    return _compile(_SRC, _LIB_PATH, force)


def _bind(path: str):
    lib = ctypes.CDLL(path)
    i = ctypes.c_int
    lib.oracle_scan_f64.argtypes = [i, i, i, i, i] + [_P] * 14 + [i]
    lib.oracle_scan_f64.restype = None
    lib.oracle_scan_chunked_f64.argtypes = [i, i, i, i, i, i] + [_P] * 14
    lib.oracle_scan_chunked_f64.restype = None
    lib.oracle_step_f64.argtypes = [i, i, i, i] + [_P] * 12
    lib.oracle_step_f64.restype = None
    lib.oracle_scan_bwd_f64.argtypes = [i, i, i, i, i] + [_P] * 25
    lib.oracle_scan_bwd_f64.restype = None
    lib.oracle_ssd_f64.argtypes = [i] * 6 + [_P] * 10
    lib.oracle_ssd_f64.restype = None
    return lib


def _load(lib=None):
    """The default oracle library, or `lib` when given (a path or a handle):
    the tests load deliberately mutated copies this way."""
    global _lib
    if lib is not None:
        return _bind(lib) if isinstance(lib, str) else lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile C source text (e.g. a mutated copy of mamba_oracle.c, for the
    tests that check the pins catch planted mistakes) into out_path."""
    c_path = out_path + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o",
                    out_path, c_path, "-lm"], check=True)
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def f64(a) -> np.ndarray:
    """Contiguous fp64 numpy copy of a numpy array or a (CPU/CUDA) torch tensor.

    bf16 and fp32 values convert to fp64 exactly, so the oracle sees the very
    values the GPU receives.
    """
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(_P)


def scan(x, z, dt_raw, Bm, Cm, A_log, Dskip, conv_w, conv_b=None, h0=None,
         conv_state0=None, n_threads: int = 0, lib=None):
    """Sequential fp64 scan.  Shapes: x, z, dt_raw (B,L,D); Bm, Cm (B,L,N);
    A_log (D,N); Dskip (D,); conv_w (D,K); conv_b (D,) or None;
    h0 (B,D,N) or None; conv_state0 (B,K-1,D) or None.
    Returns (y (B,L,D), final_h (B,D,N), final_conv_state (B,K-1,D))."""
    lib = _load(lib)
    x, z, dt_raw, Bm, Cm = map(f64, (x, z, dt_raw, Bm, Cm))
    A_log, Dskip, conv_w, conv_b, h0, conv_state0 = map(
        f64, (A_log, Dskip, conv_w, conv_b, h0, conv_state0))
    B, L, D = x.shape
    N = A_log.shape[1]
    K = conv_w.shape[1]
    y = np.zeros((B, L, D))
    fh = np.zeros((B, D, N))
    fcs = np.zeros((B, max(K - 1, 0), D))
    lib.oracle_scan_f64(B, L, D, N, K, _ptr(x), _ptr(z), _ptr(dt_raw), _ptr(Bm),
                        _ptr(Cm), _ptr(A_log), _ptr(Dskip), _ptr(conv_w),
                        _ptr(conv_b), _ptr(h0), _ptr(conv_state0), _ptr(y),
                        _ptr(fh), _ptr(fcs), int(n_threads))
    return y, fh, fcs


def scan_chunked(x, z, dt_raw, Bm, Cm, A_log, Dskip, conv_w, conv_b=None,
                 h0=None, conv_state0=None, chunk: int = 64, lib=None):
    """The scan evaluated chunk by chunk (see mamba_oracle.c); same outputs."""
    lib = _load(lib)
    x, z, dt_raw, Bm, Cm = map(f64, (x, z, dt_raw, Bm, Cm))
    A_log, Dskip, conv_w, conv_b, h0, conv_state0 = map(
        f64, (A_log, Dskip, conv_w, conv_b, h0, conv_state0))
    B, L, D = x.shape
    N = A_log.shape[1]
    K = conv_w.shape[1]
    y = np.zeros((B, L, D))
    fh = np.zeros((B, D, N))
    fcs = np.zeros((B, max(K - 1, 0), D))
    lib.oracle_scan_chunked_f64(B, L, D, N, K, int(chunk), _ptr(x), _ptr(z),
                                _ptr(dt_raw), _ptr(Bm), _ptr(Cm), _ptr(A_log),
                                _ptr(Dskip), _ptr(conv_w), _ptr(conv_b),
                                _ptr(h0), _ptr(conv_state0), _ptr(y), _ptr(fh),
                                _ptr(fcs))
    return y, fh, fcs


def step(h, conv_state, x_t, z_t, dt_raw_t, B_t, C_t, A_log, Dskip, conv_w,
         conv_b=None, lib=None):
    """One fp64 decode token.  h (B,D,N) and conv_state (B,K-1,D) are taken
    as fp64 copies, updated and returned: (y_t (B,D), h, conv_state)."""
    lib = _load(lib)
    h = f64(h).copy()
    conv_state = f64(conv_state).copy()
    x_t, z_t, dt_raw_t, B_t, C_t = map(f64, (x_t, z_t, dt_raw_t, B_t, C_t))
    A_log, Dskip, conv_w, conv_b = map(f64, (A_log, Dskip, conv_w, conv_b))
    B, D = x_t.shape
    N = A_log.shape[1]
    K = conv_w.shape[1]
    y = np.zeros((B, D))
    lib.oracle_step_f64(B, D, N, K, _ptr(h), _ptr(conv_state), _ptr(x_t),
                        _ptr(z_t), _ptr(dt_raw_t), _ptr(B_t), _ptr(C_t),
                        _ptr(A_log), _ptr(Dskip), _ptr(conv_w), _ptr(conv_b),
                        _ptr(y))
    return y, h, conv_state


BWD_NAMES = ("dx", "dz", "ddt_raw", "dB", "dC", "dA_log", "dD", "dconv_w", "dconv_b", "dh0",
             "dconv_state0")


def scan_bwd(x, z, dt_raw, Bm, Cm, A_log, Dskip, conv_w, conv_b=None, h0=None,
             conv_state0=None, dy=None, dfinal_h=None, dfinal_conv_state=None, lib=None):
    """Gradients of loss = sum(y*dy) + sum(final_h*dfinal_h)
    + sum(final_conv_state*dfinal_conv_state) with respect to every input of
    scan(...).  Returns a dict keyed by BWD_NAMES (dconv_b is zero when conv_b
    is None; dh0 and dconv_state0 are returned whether or not h0 / conv_state0
    were given, as the gradients at those zero defaults)."""
    lib = _load(lib)
    x, z, dt_raw, Bm, Cm, dy = map(f64, (x, z, dt_raw, Bm, Cm, dy))
    A_log, Dskip, conv_w, conv_b, h0, conv_state0 = map(
        f64, (A_log, Dskip, conv_w, conv_b, h0, conv_state0))
    dfinal_h, dfinal_conv_state = f64(dfinal_h), f64(dfinal_conv_state)
    B, L, D = x.shape
    N = A_log.shape[1]
    K = conv_w.shape[1]
    out = {"dx": np.zeros((B, L, D)), "dz": np.zeros((B, L, D)), "ddt_raw": np.zeros((B, L, D)),
           "dB": np.zeros((B, L, N)), "dC": np.zeros((B, L, N)), "dA_log": np.zeros((D, N)),
           "dD": np.zeros(D), "dconv_w": np.zeros((D, K)), "dconv_b": np.zeros(D),
           "dh0": np.zeros((B, D, N)), "dconv_state0": np.zeros((B, max(K - 1, 0), D))}
    lib.oracle_scan_bwd_f64(B, L, D, N, K, _ptr(x), _ptr(z), _ptr(dt_raw), _ptr(Bm), _ptr(Cm),
                            _ptr(A_log), _ptr(Dskip), _ptr(conv_w), _ptr(conv_b), _ptr(h0),
                            _ptr(conv_state0), _ptr(dy), _ptr(dfinal_h), _ptr(dfinal_conv_state),
                            *[_ptr(out[k]) for k in BWD_NAMES])
    return out


def bf16_round(a) -> np.ndarray:
    """fp64 values rounded to bf16 the way the GPU stores an fp32 result: to
    fp32 (nearest), then to the upper 16 bits (nearest, ties to even);
    returned as fp64.  Finite values only."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float64).astype(np.float32))
    bits = f.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def layer(hidden, W_in, conv_w, conv_b, W_x, W_dt, b_dt, A_log, Dskip, W_out, lib=None):
    """The Mamba layer of "【大模型】- Jamba 混合 SSM-Transformer", section
    "实现 > Mamba 层" (MambaBlock.forward), in fp64:
      x | z = hidden W_in^T (in_proj, rows 0..D-1 then D..2D-1 of W_in)
      u = silu(conv(x)) (causal depthwise conv, zero inputs before t = 0)
      dt_in | B | C = u W_x^T (x_proj; per token dt_rank, 16 and 16 values:
                      the blog's x_proj omits C, the layer it describes has it)
      dt_raw = dt_in W_dt^T + b_dt (dt_proj with its bias)
      y = scan(x, z, dt_raw, B, C, ...) (the C oracle above)
      out = y W_out^T (out_proj)
    Every quantity the library stores in bf16 (x, z, u, the x_proj output,
    dt_raw, y, out) is rounded to bf16 here at the same point, so that both
    sides feed each stage the same kind of values.  Returns a dict with out
    and the intermediates."""
    h = f64(hidden)
    Bsz, L, _ = h.shape
    Win = f64(W_in)
    D = Win.shape[0] // 2
    x = bf16_round(h @ Win[:D].T)
    z = bf16_round(h @ Win[D:].T)
    cw = f64(conv_w)
    cb = np.zeros(D) if conv_b is None else f64(conv_b)
    xp = np.concatenate([np.zeros((Bsz, 3, D)), x], axis=1)
    pre = cb + cw[:, 0] * xp[:, 0:L] + cw[:, 1] * xp[:, 1:L + 1] + cw[:, 2] * xp[:, 2:L + 2] + cw[:, 3] * xp[:, 3:L + 3]
    u = bf16_round(pre / (1.0 + np.exp(-pre)))
    xdbl = bf16_round(u @ f64(W_x).T)
    R = f64(W_dt).shape[1]
    dt_in, Bm, Cm = xdbl[..., :R], xdbl[..., R:R + 16], xdbl[..., R + 16:R + 32]
    bias = 0.0 if b_dt is None else f64(b_dt)
    dt_raw = bf16_round(dt_in @ f64(W_dt).T + bias)
    y, fh, fcs = scan(x, z, dt_raw, np.ascontiguousarray(Bm), np.ascontiguousarray(Cm), A_log, Dskip, conv_w,
                      conv_b, lib=lib)
    y = bf16_round(y)
    out = bf16_round(y @ f64(W_out).T)
    return dict(out=out, x=x, z=z, u=u, xdbl=xdbl, dt_raw=dt_raw, y=y, final_h=fh, final_conv_state=fcs)


def ssd(x, dt_raw, A_log, Bm, Cm, Dskip, z=None, h0=None, lib=None):
    """Mamba-2's scan (mamba_oracle.c: oracle_ssd_f64, which states it and its
    page).  x, z (B,L,H,P); dt_raw (B,L,H); A_log, Dskip (H); Bm, Cm
    (B,L,G,N); h0 (B,H,N,P).  Returns (y (B,L,H,P), final_S (B,H,N,P))."""
    lib = _load(lib)
    x, z, dt_raw, A_log, Bm, Cm, Dskip, h0 = map(f64, (x, z, dt_raw, A_log, Bm, Cm, Dskip, h0))
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    y = np.zeros((B, L, H, P))
    fs = np.zeros((B, H, N, P))
    lib.oracle_ssd_f64(B, L, H, P, G, N, _ptr(x), _ptr(z), _ptr(dt_raw), _ptr(A_log), _ptr(Bm), _ptr(Cm),
                       _ptr(Dskip), _ptr(h0), _ptr(y), _ptr(fs))
    return y, fs


# ---------------------------------------------------------------- complex scan
def _bind_m3(path: str):
    lib = ctypes.CDLL(path)
    i = ctypes.c_int
    lib.oracle_m3_scan_f64.argtypes = [i] * 5 + [_P] * 13 + [i] + [_P] * 4 + [i]
    lib.oracle_m3_scan_f64.restype = None
    lib.oracle_m3_core_f64.argtypes = [i, i] + [_P] * 6 + [i] + [_P] * 3
    lib.oracle_m3_core_f64.restype = None
    return lib


def _load_m3(lib=None):
    global _lib_m3
    if lib is not None:
        return _bind_m3(lib) if isinstance(lib, str) else lib
    with _lock:
        if _lib_m3 is None:
            build()
            _lib_m3 = _bind_m3(_LIB_M3_PATH)
    return _lib_m3


def source_m3() -> str:
    with open(_SRC_M3) as f:
        return f.read()


def m3_scan(x, z, dt_raw, Bm, Cm, A_log, theta, Dskip, conv_w, conv_b=None, h0=None,
            conv_state0=None, v0=None, trapezoidal: bool = False, n_threads: int = 0, lib=None):
    """The complex-valued scan (mamba3_oracle.c).  Shapes: x, z, dt_raw (B,L,D);
    Bm, Cm (B,L,2M) as (re, im) pairs; A_log, theta (D,M); Dskip (D,);
    conv_w (D,K); conv_b (D,) or None; h0, v0 (B,D,2M) or None; conv_state0
    (B,K-1,D) or None.  Returns (y (B,L,D), final_h (B,D,2M),
    final_conv_state (B,K-1,D), final_v (B,D,2M))."""
    lib = _load_m3(lib)
    x, z, dt_raw, Bm, Cm = map(f64, (x, z, dt_raw, Bm, Cm))
    A_log, theta, Dskip, conv_w, conv_b, h0, conv_state0, v0 = map(
        f64, (A_log, theta, Dskip, conv_w, conv_b, h0, conv_state0, v0))
    B, L, D = x.shape
    M = A_log.shape[1]
    K = conv_w.shape[1]
    assert Bm.shape[-1] == 2 * M and theta.shape == A_log.shape
    y = np.zeros((B, L, D))
    fh = np.zeros((B, D, 2 * M))
    fv = np.zeros((B, D, 2 * M))
    fcs = np.zeros((B, max(K - 1, 0), D))
    lib.oracle_m3_scan_f64(B, L, D, M, K, _ptr(x), _ptr(z), _ptr(dt_raw), _ptr(Bm), _ptr(Cm),
                           _ptr(A_log), _ptr(theta), _ptr(Dskip), _ptr(conv_w), _ptr(conv_b),
                           _ptr(h0), _ptr(conv_state0), _ptr(v0), int(trapezoidal), _ptr(y),
                           _ptr(fh), _ptr(fcs), _ptr(fv), int(n_threads))
    return y, fh, fcs, fv


def m3_core(u, dt, Bm, Cm, A_log, theta, h0=None, v0=None, trapezoidal: bool = False, lib=None):
    """The bare complex recurrence of one row: u, dt (L,); Bm, Cm (L,2M);
    A_log, theta (M,); h0, v0 (2M,) or None.  Returns (ys (L,) = Re(C h)
    after each token, final h (2M,), final v (2M,))."""
    lib = _load_m3(lib)
    u, dt, Bm, Cm, A_log, theta = map(f64, (u, dt, Bm, Cm, A_log, theta))
    L, M = u.shape[0], A_log.shape[0]
    h = np.zeros(2 * M) if h0 is None else f64(h0).copy()
    v = np.zeros(2 * M) if v0 is None else f64(v0).copy()
    ys = np.zeros(L)
    lib.oracle_m3_core_f64(L, M, _ptr(u), _ptr(dt), _ptr(Bm), _ptr(Cm), _ptr(A_log), _ptr(theta),
                           int(trapezoidal), _ptr(h), _ptr(v), _ptr(ys))
    return ys, h, v
