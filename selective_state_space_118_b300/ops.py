"""ctypes binding of libmamba_ssm.so: argument marshalling only.

Every function here packs torch tensors' device pointers into the C structs
of ``include/mamba_ssm.h`` and calls the C ABI; all arithmetic runs in the
library's CUDA kernels.  Output and workspace tensors the caller does not
pass are allocated with torch (device memory is torch's job; the library
never allocates).  If the library is missing the first call raises -- there
is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmamba_ssm.so")

MAMBA_OK, MAMBA_ERR_INVALID_ARG, MAMBA_ERR_UNSUPPORTED, MAMBA_ERR_CUDA, MAMBA_ERR_TIMEOUT, \
    MAMBA_ERR_WORKSPACE = range(6)
MAMBA_F32, MAMBA_BF16 = 0, 1
MAMBA_FLAG_TEST_STALL_FIRST_LOAD = 0x1
MAMBA_FLAG_EXACT_CARRY = 0x2
D_STATE, D_CONV = 16, 4

# the functions the public header declares (checked by the tests)
EXPORTED = ("mamba_scan_workspace_size", "mamba_scan_default_chunks", "mamba_scan_plan", "mamba_scan_fwd",
            "mamba_step", "mamba_last_error", "mamba_status_string", "mamba_abi_version",
            "mamba_scan_fwd_noalloc", "mamba_scan_bwd_workspace_size", "mamba_scan_bwd",
            "mamba_layer_workspace_size", "mamba_layer_fwd", "mamba2_scan_workspace_size",
            "mamba2_scan_fwd", "mamba3_scan_workspace_size", "mamba3_scan_fwd", "mamba_linear_fwd")
MAMBA3_EULER, MAMBA3_TRAPEZOIDAL = 0, 1
MAMBA_NOALLOC_SCRATCH_BYTES = 32 << 20

_vp = ctypes.c_void_p


class ScanArgs(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("seqlen", ctypes.c_int), ("d_inner", ctypes.c_int),
                ("d_state", ctypes.c_int), ("d_conv", ctypes.c_int), ("io", ctypes.c_int),
                ("x", _vp), ("z", _vp), ("dt_raw", _vp), ("Bm", _vp), ("Cm", _vp),
                ("A_log", _vp), ("Dskip", _vp), ("conv_w", _vp), ("conv_b", _vp),
                ("h0", _vp), ("conv_state0", _vp), ("y", _vp), ("final_h", _vp),
                ("final_conv_state", _vp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t), ("n_chunks", ctypes.c_int),
                ("flags", ctypes.c_uint32), ("wait_timeout_ns", ctypes.c_uint64),
                ("tile_states", _vp)]


class BwdArgs(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("seqlen", ctypes.c_int), ("d_inner", ctypes.c_int),
                ("d_state", ctypes.c_int), ("d_conv", ctypes.c_int), ("io", ctypes.c_int),
                ("x", _vp), ("z", _vp), ("dt_raw", _vp), ("Bm", _vp), ("Cm", _vp),
                ("A_log", _vp), ("Dskip", _vp), ("conv_w", _vp), ("conv_b", _vp),
                ("h0", _vp), ("conv_state0", _vp), ("dy", _vp), ("dfinal_h", _vp),
                ("dfinal_conv_state", _vp), ("dx", _vp), ("dz", _vp), ("ddt_raw", _vp),
                ("dB", _vp), ("dC", _vp), ("dA_log", _vp), ("dDskip", _vp), ("dconv_w", _vp),
                ("dconv_b", _vp), ("dh0", _vp), ("dconv_state0", _vp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t), ("n_chunks", ctypes.c_int),
                ("flags", ctypes.c_uint32), ("wait_timeout_ns", ctypes.c_uint64),
                ("tile_states", _vp)]


class LayerArgs(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("seqlen", ctypes.c_int), ("d_model", ctypes.c_int),
                ("d_inner", ctypes.c_int), ("dt_rank", ctypes.c_int), ("d_state", ctypes.c_int),
                ("d_conv", ctypes.c_int), ("io", ctypes.c_int),
                ("hidden", _vp), ("W_in", _vp), ("conv_w", _vp), ("conv_b", _vp), ("W_x", _vp),
                ("W_dt", _vp), ("b_dt", _vp), ("A_log", _vp), ("Dskip", _vp), ("W_out", _vp),
                ("out", _vp), ("u_out", _vp), ("final_h", _vp), ("final_conv_state", _vp),
                ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t), ("n_chunks", ctypes.c_int)]


class Mamba2Args(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("seqlen", ctypes.c_int), ("heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("groups", ctypes.c_int), ("d_state", ctypes.c_int),
                ("io", ctypes.c_int), ("x", _vp), ("z", _vp), ("dt_raw", _vp), ("Bm", _vp), ("Cm", _vp),
                ("A_log", _vp), ("Dskip", _vp), ("h0", _vp), ("y", _vp), ("final_state", _vp),
                ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t)]


class Mamba3Args(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("seqlen", ctypes.c_int), ("d_inner", ctypes.c_int),
                ("d_state", ctypes.c_int), ("d_conv", ctypes.c_int), ("io", ctypes.c_int),
                ("x", _vp), ("z", _vp), ("dt_raw", _vp), ("Bm", _vp), ("Cm", _vp),
                ("A_log", _vp), ("theta", _vp), ("Dskip", _vp), ("conv_w", _vp), ("conv_b", _vp),
                ("h0", _vp), ("conv_state0", _vp), ("v0", _vp), ("y", _vp), ("final_h", _vp),
                ("final_conv_state", _vp), ("final_v", _vp), ("workspace", _vp),
                ("workspace_bytes", ctypes.c_size_t), ("n_chunks", ctypes.c_int),
                ("discretization", ctypes.c_int), ("wait_timeout_ns", ctypes.c_uint64), ("flags", ctypes.c_uint)]


class LinearArgs(ctypes.Structure):
    _fields_ = [("M", ctypes.c_long), ("N", ctypes.c_int), ("K", ctypes.c_int), ("A", _vp), ("lda", ctypes.c_int),
                ("W", _vp), ("bias", _vp), ("C", _vp), ("ldc", ctypes.c_int), ("wait_timeout_ns", ctypes.c_uint64)]


class StepArgs(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("d_inner", ctypes.c_int), ("d_state", ctypes.c_int),
                ("d_conv", ctypes.c_int), ("io", ctypes.c_int),
                ("h", _vp), ("conv_state", _vp), ("x_t", _vp), ("z_t", _vp), ("dt_raw_t", _vp),
                ("B_t", _vp), ("C_t", _vp), ("A_log", _vp), ("Dskip", _vp), ("conv_w", _vp),
                ("conv_b", _vp), ("y_t", _vp)]


class MambaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH):
    """Loads (once) and returns the C library with its signatures declared."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m selective_state_space_118_b300.build`")
        lib = ctypes.CDLL(path)
        lib.mamba_scan_workspace_size.argtypes = [ctypes.c_int] * 4
        lib.mamba_scan_workspace_size.restype = ctypes.c_size_t
        lib.mamba_scan_default_chunks.argtypes = [ctypes.c_int] * 3
        lib.mamba_scan_default_chunks.restype = ctypes.c_int
        lib.mamba_scan_plan.argtypes = [ctypes.c_int] * 4 + [ctypes.POINTER(ctypes.c_int)]
        lib.mamba_scan_plan.restype = ctypes.c_int
        lib.mamba_scan_fwd.argtypes = [ctypes.POINTER(ScanArgs), _vp]
        lib.mamba_scan_fwd.restype = ctypes.c_int
        lib.mamba_step.argtypes = [ctypes.POINTER(StepArgs), _vp]
        lib.mamba_step.restype = ctypes.c_int
        lib.mamba_last_error.argtypes = [_vp]
        lib.mamba_last_error.restype = ctypes.c_int
        lib.mamba_status_string.argtypes = [ctypes.c_int]
        lib.mamba_status_string.restype = ctypes.c_char_p
        lib.mamba_abi_version.argtypes = []
        lib.mamba_abi_version.restype = ctypes.c_int
        lib.mamba_scan_fwd_noalloc.argtypes = [ctypes.POINTER(ScanArgs), _vp]
        lib.mamba_scan_fwd_noalloc.restype = ctypes.c_int
        lib.mamba_scan_bwd_workspace_size.argtypes = [ctypes.c_int] * 4
        lib.mamba_scan_bwd_workspace_size.restype = ctypes.c_size_t
        lib.mamba_scan_bwd.argtypes = [ctypes.POINTER(BwdArgs), _vp]
        lib.mamba_scan_bwd.restype = ctypes.c_int
        lib.mamba_layer_workspace_size.argtypes = [ctypes.c_int] * 7
        lib.mamba_layer_workspace_size.restype = ctypes.c_size_t
        lib.mamba_layer_fwd.argtypes = [ctypes.POINTER(LayerArgs), _vp]
        lib.mamba_layer_fwd.restype = ctypes.c_int
        lib.mamba2_scan_workspace_size.argtypes = [ctypes.c_int] * 3
        lib.mamba2_scan_workspace_size.restype = ctypes.c_size_t
        lib.mamba2_scan_fwd.argtypes = [ctypes.POINTER(Mamba2Args), _vp]
        lib.mamba2_scan_fwd.restype = ctypes.c_int
        lib.mamba3_scan_workspace_size.argtypes = [ctypes.c_int] * 4
        lib.mamba3_scan_workspace_size.restype = ctypes.c_size_t
        lib.mamba3_scan_fwd.argtypes = [ctypes.POINTER(Mamba3Args), _vp]
        lib.mamba3_scan_fwd.restype = ctypes.c_int
        lib.mamba_linear_fwd.argtypes = [ctypes.POINTER(LinearArgs), _vp]
        lib.mamba_linear_fwd.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().mamba_status_string(int(status)).decode()


def _io_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MAMBA_BF16
    if t.dtype == torch.float32:
        return MAMBA_F32
    raise TypeError(f"I/O tensors must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _check_args(specs, check_shapes: bool = True) -> None:
    """Dtype, shape and device of every tensor argument given.  The C ABI
    takes bare pointers and cannot see a buffer's extent, so a tensor smaller
    than the sizes passed with it would be read or written out of bounds;
    this is checked here, before any device access.  specs: (name, tensor or
    None, expected shape, expected dtype).  check_shapes is False for sizes
    the library does not support: it refuses those itself before touching
    memory.  A missing required tensor is the library's to refuse too."""
    dev = None
    for name, t, shape, dtype in specs:
        if t is None:
            continue
        if t.dtype != dtype:
            raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
        if check_shapes and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the other tensors on {dev}")


def _scan_specs(x, z, dt_raw, Bm, Cm, A_log, Dskip, conv_w, conv_b, h0, conv_state0):
    """The inputs shared by the prefill scan and its backward."""
    B, L, D = x.shape
    io, f32 = x.dtype, torch.float32
    return [("x", x, (B, L, D), io), ("z", z, (B, L, D), io), ("dt_raw", dt_raw, (B, L, D), io),
            ("Bm", Bm, (B, L, D_STATE), io), ("Cm", Cm, (B, L, D_STATE), io),
            ("A_log", A_log, (D, D_STATE), f32), ("Dskip", Dskip, (D,), f32),
            ("conv_w", conv_w, (D, D_CONV), f32), ("conv_b", conv_b, (D,), f32),
            ("h0", h0, (B, D, D_STATE), f32), ("conv_state0", conv_state0, (B, D_CONV - 1, D), io)]


def _scan_sizes_supported(A_log, conv_w) -> bool:
    return A_log.shape[-1] == D_STATE and conv_w.shape[-1] == D_CONV


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _launch(fn, args, stream, dev: torch.device) -> int:
    """Calls the C entry point with `dev` (the tensors' device) as the current
    device: the library launches on the current device and takes its
    per-device resources from it.  A stream given must belong to `dev`."""
    if stream is not None and stream.device != dev:
        raise ValueError(f"stream is on {stream.device}, the tensors on {dev}")
    with torch.cuda.device(dev):
        s = torch.cuda.current_stream(dev) if stream is None else stream
        return fn(ctypes.byref(args), s.cuda_stream)


def mamba_scan_workspace_size(batch: int, seqlen: int, d_inner: int, n_chunks: int = 0) -> int:
    return int(load_library().mamba_scan_workspace_size(batch, seqlen, d_inner, n_chunks))


def mamba_scan_default_chunks(batch: int, seqlen: int, d_inner: int) -> int:
    return int(load_library().mamba_scan_default_chunks(batch, seqlen, d_inner))


def mamba_scan_plan(batch: int, seqlen: int, d_inner: int, n_chunks: int = 0) -> dict:
    """The work plan of mamba_scan_fwd for these sizes: chunks, tokens per
    chunk, summary pieces per chunk and tokens per piece (0, 0 for one pass)."""
    out = (ctypes.c_int * 4)()
    st = load_library().mamba_scan_plan(batch, seqlen, d_inner, n_chunks, out)
    if st != MAMBA_OK:
        raise MambaError(st, "mamba_scan_plan")
    return dict(n_chunks=out[0], chunk_len=out[1], pieces=out[2], piece_len=out[3])


def mamba_scan_fwd(x, z, dt_raw, Bm, Cm, A_log, Dskip, conv_w, conv_b=None, h0=None,
                   conv_state0=None, *, y=None, final_h=None, final_conv_state=None,
                   workspace=None, n_chunks: int = 0, flags: int = 0,
                   wait_timeout_ns: int = 0, return_state: bool = True, tile_states=None,
                   stream=None):
    """Prefill scan (C ABI ``mamba_scan_fwd``).  x, z, dt_raw (B,L,D) and
    Bm, Cm (B,L,16) in fp32 or bf16; A_log (D,16), Dskip (D), conv_w (D,4),
    conv_b (D) fp32; h0 (B,D,16) fp32; conv_state0 (B,3,D) in the I/O dtype.
    Returns (y, final_h, final_conv_state) (the last two None when
    return_state is False and they were not passed).  tile_states: an fp32
    tensor of tile_states_shape(B, L, D) that receives the state entering
    every 16-token tile, for mamba_scan_bwd."""
    lib = load_library()
    B, L, D = x.shape
    dev = x.device
    _check_tile_states(tile_states, B, L, D)
    _check_args(_scan_specs(x, z, dt_raw, Bm, Cm, A_log, Dskip, conv_w, conv_b, h0, conv_state0)
                + [("y", y, (B, L, D), x.dtype), ("final_h", final_h, (B, D, D_STATE), torch.float32),
                   ("final_conv_state", final_conv_state, (B, D_CONV - 1, D), x.dtype)],
                _scan_sizes_supported(A_log, conv_w))
    if y is None:
        y = torch.empty_like(x)
    if return_state:
        if final_h is None:
            final_h = torch.empty((B, D, D_STATE), device=dev, dtype=torch.float32)
        if final_conv_state is None:
            final_conv_state = torch.empty((B, D_CONV - 1, D), device=dev, dtype=x.dtype)
    ws_bytes = mamba_scan_workspace_size(B, L, D, n_chunks)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    a = ScanArgs(batch=B, seqlen=L, d_inner=D, d_state=A_log.shape[-1], d_conv=conv_w.shape[-1],
                 io=_io_code(x), x=_ptr(x), z=_ptr(z), dt_raw=_ptr(dt_raw), Bm=_ptr(Bm),
                 Cm=_ptr(Cm), A_log=_ptr(A_log), Dskip=_ptr(Dskip), conv_w=_ptr(conv_w),
                 conv_b=_ptr(conv_b), h0=_ptr(h0), conv_state0=_ptr(conv_state0), y=_ptr(y),
                 final_h=_ptr(final_h), final_conv_state=_ptr(final_conv_state),
                 workspace=_ptr(workspace),
                 workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
                 n_chunks=n_chunks, flags=flags, wait_timeout_ns=wait_timeout_ns,
                 tile_states=_ptr(tile_states))
    st = _launch(lib.mamba_scan_fwd, a, stream, dev)
    if st != MAMBA_OK:
        raise MambaError(st, "mamba_scan_fwd")
    return y, final_h, final_conv_state


def mamba_scan_bwd_workspace_size(batch: int, seqlen: int, d_inner: int, n_chunks: int = 0) -> int:
    return int(load_library().mamba_scan_bwd_workspace_size(batch, seqlen, d_inner, n_chunks))


BWD_OUTPUTS = ("dx", "dz", "ddt_raw", "dB", "dC", "dA_log", "dDskip", "dconv_w", "dconv_b", "dh0",
               "dconv_state0")


def tile_states_shape(batch: int, seqlen: int, d_inner: int) -> tuple:
    """Shape of the tile states mamba_scan_fwd can store for mamba_scan_bwd."""
    return (batch, (seqlen + 15) // 16, d_inner, D_STATE)


def _check_tile_states(t, batch: int, seqlen: int, d_inner: int) -> None:
    """The C ABI takes a bare pointer: the buffer's size is checked here."""
    if t is None:
        return
    shape = tile_states_shape(batch, seqlen, d_inner)
    if t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != shape:
        raise ValueError(f"tile_states must be a contiguous float32 tensor of shape {shape}")


def mamba_scan_bwd(x, z, dt_raw, Bm, Cm, A_log, Dskip, conv_w, conv_b=None, h0=None,
                   conv_state0=None, *, dy, dfinal_h=None, dfinal_conv_state=None,
                   out=None, workspace=None, n_chunks: int = 0, flags: int = 0, wait_timeout_ns: int = 0,
                   tile_states=None, stream=None) -> dict:
    """Backward of the prefill scan (C ABI ``mamba_scan_bwd``): the gradients
    of l given dy = dl/dy (B,L,D) and optionally dl/dfinal_h (B,D,16) fp32 and
    dl/dfinal_conv_state (B,3,D).  Returns a dict keyed by BWD_OUTPUTS: dx,
    dz, ddt_raw in the I/O dtype, everything else fp32 (dconv_b only when
    conv_b is given).  `out` may hold preallocated outputs by the same keys.
    tile_states: the tile states of a mamba_scan_fwd of the same inputs
    (skips the forward recomputation; with the same n_chunks as that call,
    the gradients are the same bits as without it)."""
    lib = load_library()
    B, L, D = x.shape
    dev = x.device
    _check_tile_states(tile_states, B, L, D)
    f32 = torch.float32
    shapes = {"dx": ((B, L, D), x.dtype), "dz": ((B, L, D), x.dtype), "ddt_raw": ((B, L, D), x.dtype),
              "dB": ((B, L, D_STATE), f32), "dC": ((B, L, D_STATE), f32),
              "dA_log": ((D, D_STATE), f32), "dDskip": ((D,), f32), "dconv_w": ((D, D_CONV), f32),
              "dconv_b": ((D,), f32), "dh0": ((B, D, D_STATE), f32),
              "dconv_state0": ((B, D_CONV - 1, D), f32)}
    g = dict(out or {})
    for k, (shape, dtype) in shapes.items():
        if k == "dconv_b" and conv_b is None:
            g.setdefault(k, None)
            continue
        if g.get(k) is None:
            g[k] = torch.empty(shape, device=dev, dtype=dtype)
    _check_args(_scan_specs(x, z, dt_raw, Bm, Cm, A_log, Dskip, conv_w, conv_b, h0, conv_state0)
                + [("dy", dy, (B, L, D), x.dtype), ("dfinal_h", dfinal_h, (B, D, D_STATE), f32),
                   ("dfinal_conv_state", dfinal_conv_state, (B, D_CONV - 1, D), x.dtype)]
                + [(k, g[k], shape, dtype) for k, (shape, dtype) in shapes.items()],
                _scan_sizes_supported(A_log, conv_w))
    ws_bytes = mamba_scan_bwd_workspace_size(B, L, D, n_chunks)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    a = BwdArgs(batch=B, seqlen=L, d_inner=D, d_state=A_log.shape[-1], d_conv=conv_w.shape[-1],
                io=_io_code(x), x=_ptr(x), z=_ptr(z), dt_raw=_ptr(dt_raw), Bm=_ptr(Bm), Cm=_ptr(Cm),
                A_log=_ptr(A_log), Dskip=_ptr(Dskip), conv_w=_ptr(conv_w), conv_b=_ptr(conv_b),
                h0=_ptr(h0), conv_state0=_ptr(conv_state0), dy=_ptr(dy), dfinal_h=_ptr(dfinal_h),
                dfinal_conv_state=_ptr(dfinal_conv_state),
                **{k: _ptr(g[k]) for k in BWD_OUTPUTS},
                workspace=_ptr(workspace),
                workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
                n_chunks=n_chunks, flags=flags, wait_timeout_ns=wait_timeout_ns,
                tile_states=_ptr(tile_states))
    st = _launch(lib.mamba_scan_bwd, a, stream, dev)
    if st != MAMBA_OK:
        raise MambaError(st, "mamba_scan_bwd")
    return g


def mamba_layer_workspace_size(batch: int, seqlen: int, d_model: int, d_inner: int, dt_rank: int,
                               n_chunks: int = 0, with_u_out: bool = False) -> int:
    return int(load_library().mamba_layer_workspace_size(batch, seqlen, d_model, d_inner, dt_rank, n_chunks,
                                                         int(with_u_out)))


def mamba_layer_fwd(hidden, W_in, conv_w, conv_b, W_x, W_dt, b_dt, A_log, Dskip, W_out, *, out=None,
                    u_out=None, final_h=None, final_conv_state=None, workspace=None, n_chunks: int = 0,
                    stream=None):
    """The whole Mamba layer (C ABI ``mamba_layer_fwd``): hidden (B,L,H) bf16;
    W_in (2D,H), W_x (R+32,D), W_dt (D,R), b_dt (D), W_out (H,D) bf16;
    conv_w (D,4), conv_b (D), A_log (D,16), Dskip (D) fp32.  Returns out
    (B,L,H) bf16 (u_out, final_h, final_conv_state are filled when given)."""
    lib = load_library()
    B, L, H = hidden.shape
    D = A_log.shape[0]
    R = W_dt.shape[1]
    bf, f32 = torch.bfloat16, torch.float32
    _check_args([("hidden", hidden, (B, L, H), bf), ("W_in", W_in, (2 * D, H), bf),
                 ("conv_w", conv_w, (D, D_CONV), f32), ("conv_b", conv_b, (D,), f32),
                 ("W_x", W_x, (R + 2 * D_STATE, D), bf), ("W_dt", W_dt, (D, R), bf), ("b_dt", b_dt, (D,), bf),
                 ("A_log", A_log, (D, D_STATE), f32), ("Dskip", Dskip, (D,), f32), ("W_out", W_out, (H, D), bf),
                 ("out", out, (B, L, H), bf), ("u_out", u_out, (B, L, D), bf),
                 ("final_h", final_h, (B, D, D_STATE), f32),
                 ("final_conv_state", final_conv_state, (B, D_CONV - 1, D), bf)],
                _scan_sizes_supported(A_log, conv_w) and R % 8 == 0)
    if out is None:
        out = torch.empty_like(hidden)
    ws_bytes = mamba_layer_workspace_size(B, L, H, D, R, n_chunks, u_out is not None)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, device=hidden.device, dtype=torch.uint8)
    a = LayerArgs(batch=B, seqlen=L, d_model=H, d_inner=D, dt_rank=R, d_state=A_log.shape[-1],
                  d_conv=conv_w.shape[-1], io=_io_code(hidden), hidden=_ptr(hidden), W_in=_ptr(W_in),
                  conv_w=_ptr(conv_w), conv_b=_ptr(conv_b), W_x=_ptr(W_x), W_dt=_ptr(W_dt), b_dt=_ptr(b_dt),
                  A_log=_ptr(A_log), Dskip=_ptr(Dskip), W_out=_ptr(W_out), out=_ptr(out), u_out=_ptr(u_out),
                  final_h=_ptr(final_h), final_conv_state=_ptr(final_conv_state), workspace=_ptr(workspace),
                  workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
                  n_chunks=n_chunks)
    st = _launch(lib.mamba_layer_fwd, a, stream, hidden.device)
    if st != MAMBA_OK:
        raise MambaError(st, "mamba_layer_fwd")
    return out


def mamba2_scan_workspace_size(batch: int, seqlen: int, heads: int) -> int:
    return int(load_library().mamba2_scan_workspace_size(batch, seqlen, heads))


def mamba2_scan_fwd(x, dt_raw, A_log, Bm, Cm, Dskip, z=None, h0=None, *, y=None, final_state=None,
                    workspace=None, stream=None):
    """Mamba-2's chunked scan (C ABI ``mamba2_scan_fwd``): x, z (B,L,H,64),
    dt_raw (B,L,H), Bm, Cm (B,L,G,16) bf16; A_log, Dskip (H) fp32; h0
    (B,H,16,64) fp32.  Returns (y, final_state)."""
    lib = load_library()
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    io, f32 = x.dtype, torch.float32
    _check_args([("x", x, (B, L, H, P), io), ("dt_raw", dt_raw, (B, L, H), io), ("A_log", A_log, (H,), f32),
                 ("Bm", Bm, (B, L, G, N), io), ("Cm", Cm, (B, L, G, N), io), ("Dskip", Dskip, (H,), f32),
                 ("z", z, (B, L, H, P), io), ("h0", h0, (B, H, N, P), f32), ("y", y, (B, L, H, P), io),
                 ("final_state", final_state, (B, H, N, P), f32)],
                P == 64 and N == D_STATE)
    if y is None:
        y = torch.empty_like(x)
    if final_state is None:
        final_state = torch.empty((B, H, N, P), device=x.device, dtype=torch.float32)
    ws_bytes = mamba2_scan_workspace_size(B, L, H)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, device=x.device, dtype=torch.uint8)
    a = Mamba2Args(batch=B, seqlen=L, heads=H, head_dim=P, groups=G, d_state=N, io=_io_code(x), x=_ptr(x),
                   z=_ptr(z), dt_raw=_ptr(dt_raw), Bm=_ptr(Bm), Cm=_ptr(Cm), A_log=_ptr(A_log),
                   Dskip=_ptr(Dskip), h0=_ptr(h0), y=_ptr(y), final_state=_ptr(final_state),
                   workspace=_ptr(workspace),
                   workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size())
    st = _launch(lib.mamba2_scan_fwd, a, stream, x.device)
    if st != MAMBA_OK:
        raise MambaError(st, "mamba2_scan_fwd")
    return y, final_state


def mamba3_scan_workspace_size(batch: int, seqlen: int, d_inner: int, n_chunks: int = 0) -> int:
    return int(load_library().mamba3_scan_workspace_size(batch, seqlen, d_inner, n_chunks))


def mamba3_scan_fwd(x, z, dt_raw, Bm, Cm, A_log, theta, Dskip, conv_w, conv_b=None, h0=None,
                    conv_state0=None, v0=None, *, trapezoidal: bool = False, y=None, final_h=None,
                    final_conv_state=None, final_v=None, workspace=None, n_chunks: int = 0,
                    wait_timeout_ns: int = 0, flags: int = 0, return_state: bool = True, stream=None):
    """The complex-valued scan (C ABI ``mamba3_scan_fwd``): x, z, dt_raw
    (B,L,D) and Bm, Cm (B,L,16: 8 complex numbers as (re, im) pairs) in fp32
    or bf16; A_log, theta (D,8), Dskip (D), conv_w (D,4), conv_b (D) fp32;
    h0, v0 (B,D,16) fp32; conv_state0 (B,3,D) in the I/O dtype.  Returns
    (y, final_h, final_conv_state, final_v) (the last three None when
    return_state is False and they were not passed)."""
    lib = load_library()
    B, L, D = x.shape
    dev = x.device
    f32 = torch.float32
    modes = D_STATE // 2
    specs = _scan_specs(x, z, dt_raw, Bm, Cm, None, Dskip, conv_w, conv_b, h0, conv_state0)
    specs += [("A_log", A_log, (D, modes), f32), ("theta", theta, (D, modes), f32),
              ("v0", v0, (B, D, D_STATE), f32), ("y", y, (B, L, D), x.dtype),
              ("final_h", final_h, (B, D, D_STATE), f32), ("final_v", final_v, (B, D, D_STATE), f32),
              ("final_conv_state", final_conv_state, (B, D_CONV - 1, D), x.dtype)]
    _check_args(specs, A_log.shape[-1] == modes and conv_w.shape[-1] == D_CONV)
    if y is None:
        y = torch.empty_like(x)
    if return_state:
        if final_h is None:
            final_h = torch.empty((B, D, D_STATE), device=dev, dtype=f32)
        if final_v is None:
            final_v = torch.empty((B, D, D_STATE), device=dev, dtype=f32)
        if final_conv_state is None:
            final_conv_state = torch.empty((B, D_CONV - 1, D), device=dev, dtype=x.dtype)
    ws_bytes = mamba3_scan_workspace_size(B, L, D, n_chunks)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, device=dev, dtype=torch.uint8)
    a = Mamba3Args(batch=B, seqlen=L, d_inner=D, d_state=2 * A_log.shape[-1], d_conv=conv_w.shape[-1],
                   io=_io_code(x), x=_ptr(x), z=_ptr(z), dt_raw=_ptr(dt_raw), Bm=_ptr(Bm), Cm=_ptr(Cm),
                   A_log=_ptr(A_log), theta=_ptr(theta), Dskip=_ptr(Dskip), conv_w=_ptr(conv_w),
                   conv_b=_ptr(conv_b), h0=_ptr(h0), conv_state0=_ptr(conv_state0), v0=_ptr(v0), y=_ptr(y),
                   final_h=_ptr(final_h), final_conv_state=_ptr(final_conv_state), final_v=_ptr(final_v),
                   workspace=_ptr(workspace),
                   workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
                   n_chunks=n_chunks, discretization=MAMBA3_TRAPEZOIDAL if trapezoidal else MAMBA3_EULER,
                   wait_timeout_ns=wait_timeout_ns, flags=flags)
    st = _launch(lib.mamba3_scan_fwd, a, stream, dev)
    if st != MAMBA_OK:
        raise MambaError(st, "mamba3_scan_fwd")
    return y, final_h, final_conv_state, final_v


def mamba_linear_fwd(A, W, bias=None, *, out=None, wait_timeout_ns: int = 0, stream=None):
    """C = A W^T (+ bias) on the tensor cores (C ABI ``mamba_linear_fwd``):
    A (..., K), W (N, K), bias (N) bf16; returns C (..., N) bf16.  A's rows
    may be a strided view (rows lda apart) of a wider matrix."""
    lib = load_library()
    K = A.shape[-1]
    N = W.shape[0]
    bf = torch.bfloat16
    A2 = A.reshape(-1, K) if A.is_contiguous() else A
    if A2.dim() != 2 or A2.stride(1) != 1:
        raise ValueError("A must be a row-major matrix (rows may be strided)")
    M = A2.shape[0]
    _check_args([("A", A2, (M, K), bf), ("W", W, (N, K), bf), ("bias", bias, (N,), bf)])
    if out is None:
        out = torch.empty(A.shape[:-1] + (N,), device=A.device, dtype=bf)
    C2 = out.reshape(-1, N) if out.is_contiguous() else out
    _check_args([("out", C2, (M, N), bf)])
    if not (A2.is_cuda and W.is_cuda and C2.is_cuda) or not W.is_contiguous():
        raise ValueError("tensors must be on a CUDA device and W contiguous")
    a = LinearArgs(M=M, N=N, K=K, A=A2.data_ptr(), lda=A2.stride(0), W=W.data_ptr(), bias=_ptr(bias),
                   C=C2.data_ptr(), ldc=C2.stride(0), wait_timeout_ns=wait_timeout_ns)
    st = _launch(lib.mamba_linear_fwd, a, stream, A.device)
    if st != MAMBA_OK:
        raise MambaError(st, "mamba_linear_fwd")
    return out


def mamba_step(h, conv_state, x_t, z_t, dt_raw_t, B_t, C_t, A_log, Dskip, conv_w, conv_b=None,
               *, y_t=None, stream=None):
    """One decode token (C ABI ``mamba_step``): h (B,D,16) fp32 and
    conv_state (B,3,D) are updated in place; returns y_t (B,D)."""
    lib = load_library()
    B, D = x_t.shape
    io, f32 = x_t.dtype, torch.float32
    _check_args([("h", h, (B, D, D_STATE), f32), ("conv_state", conv_state, (B, D_CONV - 1, D), io),
                 ("x_t", x_t, (B, D), io), ("z_t", z_t, (B, D), io), ("dt_raw_t", dt_raw_t, (B, D), io),
                 ("B_t", B_t, (B, D_STATE), io), ("C_t", C_t, (B, D_STATE), io),
                 ("A_log", A_log, (D, D_STATE), f32), ("Dskip", Dskip, (D,), f32),
                 ("conv_w", conv_w, (D, D_CONV), f32), ("conv_b", conv_b, (D,), f32), ("y_t", y_t, (B, D), io)],
                _scan_sizes_supported(A_log, conv_w))
    if y_t is None:
        y_t = torch.empty_like(x_t)
    a = StepArgs(batch=B, d_inner=D, d_state=A_log.shape[-1], d_conv=conv_w.shape[-1],
                 io=_io_code(x_t), h=_ptr(h), conv_state=_ptr(conv_state), x_t=_ptr(x_t),
                 z_t=_ptr(z_t), dt_raw_t=_ptr(dt_raw_t), B_t=_ptr(B_t), C_t=_ptr(C_t),
                 A_log=_ptr(A_log), Dskip=_ptr(Dskip), conv_w=_ptr(conv_w), conv_b=_ptr(conv_b),
                 y_t=_ptr(y_t))
    st = _launch(lib.mamba_step, a, stream, x_t.device)
    if st != MAMBA_OK:
        raise MambaError(st, "mamba_step")
    return y_t


def mamba_last_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the sticky device
    error code: MAMBA_OK or MAMBA_ERR_TIMEOUT."""
    return int(load_library().mamba_last_error(_stream(stream)))


def mamba_abi_version() -> int:
    return int(load_library().mamba_abi_version())


def mamba_scan_fwd_noalloc(x, z, dt_raw, Bm, Cm, A_log, Dskip, conv_w, conv_b=None, h0=None,
                           conv_state0=None, *, y, final_h=None, final_conv_state=None,
                           n_chunks: int = 0, stream=None):
    """Prefill scan through ``mamba_scan_fwd_noalloc``: the same computation
    as mamba_scan_fwd for callers that cannot allocate device memory -- the
    library uses its own fixed scratch array (MAMBA_NOALLOC_SCRATCH_BYTES per
    GPU) instead of a workspace, so the caller passes only inputs and outputs
    (y, and optionally final_h / final_conv_state) and nothing here allocates.
    Calls that may overlap on the GPU share that scratch and race."""
    lib = load_library()
    B, L, D = x.shape
    _check_args(_scan_specs(x, z, dt_raw, Bm, Cm, A_log, Dskip, conv_w, conv_b, h0, conv_state0)
                + [("y", y, (B, L, D), x.dtype), ("final_h", final_h, (B, D, D_STATE), torch.float32),
                   ("final_conv_state", final_conv_state, (B, D_CONV - 1, D), x.dtype)],
                _scan_sizes_supported(A_log, conv_w))
    a = ScanArgs(batch=B, seqlen=L, d_inner=D, d_state=A_log.shape[-1], d_conv=conv_w.shape[-1],
                 io=_io_code(x), x=_ptr(x), z=_ptr(z), dt_raw=_ptr(dt_raw), Bm=_ptr(Bm),
                 Cm=_ptr(Cm), A_log=_ptr(A_log), Dskip=_ptr(Dskip), conv_w=_ptr(conv_w),
                 conv_b=_ptr(conv_b), h0=_ptr(h0), conv_state0=_ptr(conv_state0), y=_ptr(y),
                 final_h=_ptr(final_h), final_conv_state=_ptr(final_conv_state),
                 workspace=None, workspace_bytes=0, n_chunks=n_chunks, flags=0, wait_timeout_ns=0)
    st = _launch(lib.mamba_scan_fwd_noalloc, a, stream, x.device)
    if st != MAMBA_OK:
        raise MambaError(st, "mamba_scan_fwd_noalloc")
    return y, final_h, final_conv_state
