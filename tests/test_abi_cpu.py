"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/mamba_ssm.h declares, the ctypes structs match the C layout,
and host-side argument checks return the documented status codes without
launching anything."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from selective_state_space_118_b300 import build, ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mamba_ssm.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mamba[23]?_\w+)\s*\(", text)))


def test_header_declares_the_binding_functions():
    assert declared_functions() == sorted(ops.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", ops.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (mamba[23]?_\w+)$", out, flags=re.M))
    missing = set(declared_functions()) - exported
    assert not missing, f"declared but not exported: {missing}"
    for name in declared_functions():
        assert hasattr(lib, name)


def _c_layout(tmp_path, struct, fields):
    src = tmp_path / "layout.c"
    body = "\n".join(f'printf("{f} %zu\\n", offsetof({struct}, {f}));' for f in fields)
    src.write_text(f'#include <stdio.h>\n#include <stddef.h>\n#include "mamba_ssm.h"\n'
                   f'int main(void) {{ printf("sizeof %zu\\n", sizeof({struct}));\n{body}\nreturn 0; }}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), "-o", str(exe), str(src)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    return dict((k, int(v)) for k, v in (line.split() for line in out.splitlines()))


@pytest.mark.parametrize("struct,cls", [("mamba_scan_args", ops.ScanArgs),
                                        ("mamba_step_args", ops.StepArgs),
                                        ("mamba_scan_bwd_args", ops.BwdArgs),
                                        ("mamba_layer_args", ops.LayerArgs),
                                        ("mamba2_scan_args", ops.Mamba2Args),
                                        ("mamba3_scan_args", ops.Mamba3Args),
                                        ("mamba_linear_args", ops.LinearArgs)])
def test_ctypes_structs_match_c_layout(tmp_path, struct, cls):
    fields = [f for f, _ in cls._fields_]
    c = _c_layout(tmp_path, struct, fields)
    assert c["sizeof"] == ctypes.sizeof(cls)
    for f in fields:
        assert c[f] == getattr(cls, f).offset, f


def test_status_strings_and_version(lib):
    assert ops.mamba_abi_version() == 100
    for code in range(6):
        assert ops.status_string(code)
    assert "timed out" in ops.status_string(ops.MAMBA_ERR_TIMEOUT)


def _args(**kw):
    base = dict(batch=1, seqlen=8, d_inner=16, d_state=16, d_conv=4, io=ops.MAMBA_BF16)
    base.update(kw)
    return ops.ScanArgs(**base)


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced: checks fail first


@pytest.mark.parametrize("kw,status", [
    (dict(d_state=8), ops.MAMBA_ERR_UNSUPPORTED),
    (dict(d_conv=3), ops.MAMBA_ERR_UNSUPPORTED),
    (dict(d_inner=20), ops.MAMBA_ERR_UNSUPPORTED),  # bf16 rows of 40 bytes: not a multiple of 16
    (dict(d_inner=6, io=ops.MAMBA_F32), ops.MAMBA_ERR_UNSUPPORTED),  # fp32 rows of 24 bytes
    (dict(io=7), ops.MAMBA_ERR_UNSUPPORTED),
    (dict(batch=0), ops.MAMBA_ERR_INVALID_ARG),
    (dict(seqlen=-1), ops.MAMBA_ERR_INVALID_ARG),
    (dict(), ops.MAMBA_ERR_INVALID_ARG),  # A_log, Dskip, conv_w missing
    (dict(A_log=FAKE, Dskip=FAKE, conv_w=FAKE), ops.MAMBA_ERR_INVALID_ARG),  # x... missing
    (dict(A_log=FAKE, Dskip=FAKE, conv_w=FAKE + 4, x=FAKE, z=FAKE, dt_raw=FAKE, Bm=FAKE, Cm=FAKE,
          y=FAKE), ops.MAMBA_ERR_INVALID_ARG),  # misaligned conv_w
    (dict(A_log=FAKE, Dskip=FAKE, conv_w=FAKE, x=FAKE + 2, z=FAKE, dt_raw=FAKE, Bm=FAKE, Cm=FAKE,
          y=FAKE), ops.MAMBA_ERR_INVALID_ARG),  # misaligned x
    (dict(batch=1, seqlen=4096, d_inner=16, n_chunks=4, A_log=FAKE, Dskip=FAKE, conv_w=FAKE, x=FAKE,
          z=FAKE, dt_raw=FAKE, Bm=FAKE, Cm=FAKE, y=FAKE), ops.MAMBA_ERR_WORKSPACE),
])
def test_scan_argument_checks(lib, kw, status):
    a = _args(**kw)
    assert lib.mamba_scan_fwd(ctypes.byref(a), None) == status
    assert lib.mamba_scan_fwd(None, None) == ops.MAMBA_ERR_INVALID_ARG


def test_step_argument_checks(lib):
    a = ops.StepArgs(batch=1, d_inner=16, d_state=16, d_conv=4, io=ops.MAMBA_BF16)
    assert lib.mamba_step(ctypes.byref(a), None) == ops.MAMBA_ERR_INVALID_ARG
    full = dict(batch=1, d_inner=16, d_state=16, d_conv=4, io=ops.MAMBA_BF16, h=FAKE, conv_state=FAKE,
                x_t=FAKE, z_t=FAKE, dt_raw_t=FAKE, B_t=FAKE, C_t=FAKE, A_log=FAKE, Dskip=FAKE,
                conv_w=FAKE, y_t=FAKE)
    for k, off in (("h", 16), ("B_t", 8), ("A_log", 4)):  # h needs 32 bytes, the others 16
        a = ops.StepArgs(**dict(full, **{k: FAKE + off}))
        assert lib.mamba_step(ctypes.byref(a), None) == ops.MAMBA_ERR_INVALID_ARG, k
    a.d_state = 32
    assert lib.mamba_step(ctypes.byref(a), None) == ops.MAMBA_ERR_UNSUPPORTED
    assert lib.mamba_step(None, None) == ops.MAMBA_ERR_INVALID_ARG


def test_bwd_argument_checks(lib):
    base = dict(batch=1, seqlen=8, d_inner=16, d_state=16, d_conv=4, io=ops.MAMBA_BF16)
    a = ops.BwdArgs(**base)
    assert lib.mamba_scan_bwd(ctypes.byref(a), None) == ops.MAMBA_ERR_INVALID_ARG  # params missing
    full = dict(base, A_log=FAKE, Dskip=FAKE, conv_w=FAKE, dA_log=FAKE, dDskip=FAKE, dconv_w=FAKE,
                x=FAKE, z=FAKE, dt_raw=FAKE, Bm=FAKE, Cm=FAKE, dy=FAKE, dx=FAKE, dz=FAKE, ddt_raw=FAKE,
                dB=FAKE, dC=FAKE)
    for k in ("dA_log", "dy", "dB"):
        assert lib.mamba_scan_bwd(ctypes.byref(ops.BwdArgs(**dict(full, **{k: 0}))), None) == \
            ops.MAMBA_ERR_INVALID_ARG, k
    for k in ("dconv_w", "dx", "dfinal_h"):
        assert lib.mamba_scan_bwd(ctypes.byref(ops.BwdArgs(**dict(full, **{k: FAKE + 4}))), None) == \
            ops.MAMBA_ERR_INVALID_ARG, k
    assert lib.mamba_scan_bwd(ctypes.byref(ops.BwdArgs(**dict(full, d_inner=20))), None) == \
        ops.MAMBA_ERR_UNSUPPORTED
    assert lib.mamba_scan_bwd(ctypes.byref(ops.BwdArgs(**full)), None) == ops.MAMBA_ERR_WORKSPACE
    assert lib.mamba_scan_bwd(None, None) == ops.MAMBA_ERR_INVALID_ARG


def test_layer_argument_checks(lib):
    base = dict(batch=1, seqlen=8, d_model=64, d_inner=32, dt_rank=8, d_state=16, d_conv=4, io=ops.MAMBA_BF16)
    assert lib.mamba_layer_fwd(ctypes.byref(ops.LayerArgs(**base)), None) == ops.MAMBA_ERR_INVALID_ARG
    full = dict(base, hidden=FAKE, W_in=FAKE, conv_w=FAKE, W_x=FAKE, W_dt=FAKE, A_log=FAKE, Dskip=FAKE,
                W_out=FAKE, out=FAKE)
    for kw, status in ((dict(io=ops.MAMBA_F32), ops.MAMBA_ERR_UNSUPPORTED),
                       (dict(dt_rank=12), ops.MAMBA_ERR_UNSUPPORTED),
                       (dict(d_model=60), ops.MAMBA_ERR_UNSUPPORTED),
                       (dict(d_inner=20), ops.MAMBA_ERR_UNSUPPORTED),
                       (dict(seqlen=0), ops.MAMBA_ERR_INVALID_ARG),
                       (dict(W_x=FAKE + 2), ops.MAMBA_ERR_INVALID_ARG),
                       (dict(), ops.MAMBA_ERR_WORKSPACE)):
        assert lib.mamba_layer_fwd(ctypes.byref(ops.LayerArgs(**dict(full, **kw))), None) == status, kw
    # intermediates (x, z, u, x_proj output, dt_raw, y) and the scan's workspace
    B, L, H, D, R = 1, 4096, 64, 32, 8
    r = lambda v: (v + 255) // 256 * 256  # noqa: E731
    scan = ops.mamba_scan_workspace_size(B, L, D, 1)
    assert ops.mamba_layer_workspace_size(B, L, H, D, R, 1, False) == \
        5 * r(B * L * D * 2) + r(B * L * (R + 32) * 2) + scan
    assert ops.mamba_layer_workspace_size(B, L, H, D, R, 1, True) == \
        4 * r(B * L * D * 2) + r(B * L * (R + 32) * 2) + scan


def test_bwd_workspace(lib):
    def r256(v):
        return (v + 255) // 256 * 256
    # one pass: the forward's B/C rows, the state entering every 16-token tile,
    # the per-group dB | dC sums and the per-chunk parameter partials
    B, L, D = 1, 32768, 8192
    assert ops.mamba_scan_bwd_workspace_size(B, L, D, 1) == (
        r256(B * L * 32 * 4) + r256(B * (L // 16) * D * 16 * 4) + r256((D // 32) * B * L * 32 * 4)
        + r256(B * D * 24 * 4))
    assert ops.mamba_scan_bwd_workspace_size(1, 0, 64, 1) == 0
    # chunked: plus the forward's carries, the adjoint carries, their counters
    # and the conv edge buffers
    B, L, D, n = 2, 4096, 64, 4
    ws = ops.mamba_scan_bwd_workspace_size(B, L, D, n)
    G = D // 32
    need = (B * L * 32 * 4 + B * n * D * 16 * 4 + (1 + B * G * n) * 4  # forward
            + B * (L // 16) * D * 16 * 4 + B * n * D * 16 * 4 + (1 + B * G * n) * 4
            + G * B * L * 32 * 4 + B * n * D * 24 * 4 + 2 * B * n * 3 * D * 4)
    assert need <= ws <= need + 9 * 256


def test_workspace_plan(lib):
    def r256(v):
        return (v + 255) // 256 * 256
    # one sequential pass: only B and C widened to fp32, (B, L, 32)
    assert ops.mamba_scan_workspace_size(1, 32768, 8192, 1) == r256(32768 * 32 * 4)
    assert ops.mamba_scan_workspace_size(2, 2048, 1024, 1) == r256(2 * 2048 * 32 * 4)
    assert ops.mamba_scan_workspace_size(2, 0, 1024, 1) == 0
    assert ops.mamba_scan_plan(2, 2048, 1024, 1) == dict(n_chunks=1, chunk_len=2048, pieces=0, piece_len=0)
    # chunked: plus the carries into every chunk, a ticket counter and one ready
    # flag per (batch row, group of 32 channels, chunk)
    B, L, D, n = 2, 4096, 64, 4
    pl = ops.mamba_scan_plan(B, L, D, n)
    assert pl["n_chunks"] == n and pl["chunk_len"] == L // n
    m = pl["pieces"]
    assert m >= 1 and pl["piece_len"] % 16 == 0 and (m - 1) * pl["piece_len"] < pl["chunk_len"] <= m * pl["piece_len"]
    ws = ops.mamba_scan_workspace_size(B, L, D, n)
    need = B * L * 32 * 4 + B * n * D * 16 * 4 + (1 + B * (D // 32) * n) * 4
    assert need <= ws <= need + 3 * 256
    # chunks are whole 16-token tiles; a chunk count above the tile count is clamped
    assert ops.mamba_scan_plan(1, 100, 16, 50)["n_chunks"] == 7
    p3 = ops.mamba_scan_plan(1, 100, 16, 3)
    assert p3["n_chunks"] == 3 and p3["chunk_len"] == 48
    p4 = ops.mamba_scan_plan(1, 100, 16, 4)
    assert p4["n_chunks"] == 4 and p4["chunk_len"] == 32
    assert ops.mamba_scan_default_chunks(1, 16, 16) == 1
    # batch 1 at the Jamba shape cannot fill the GPU with channel groups alone: chunked
    big = ops.mamba_scan_plan(1, 32768, 8192, 0)
    assert big["n_chunks"] > 1 and big["chunk_len"] * big["n_chunks"] >= 32768
    # many sequences fill it: one pass
    assert ops.mamba_scan_default_chunks(64, 4096, 8192) == 1


def test_tile_states_checks(lib):
    """A misaligned tile-state pointer is refused by both calls; the binding
    refuses a buffer of the wrong shape or dtype before calling the C ABI
    (which cannot see a pointer's extent)."""
    scan = dict(A_log=FAKE, Dskip=FAKE, conv_w=FAKE, x=FAKE, z=FAKE, dt_raw=FAKE, Bm=FAKE, Cm=FAKE, y=FAKE)
    a = _args(**dict(scan, tile_states=FAKE + 4))
    assert lib.mamba_scan_fwd(ctypes.byref(a), None) == ops.MAMBA_ERR_INVALID_ARG
    bwd = dict(batch=1, seqlen=8, d_inner=16, d_state=16, d_conv=4, io=ops.MAMBA_BF16, A_log=FAKE, Dskip=FAKE,
               conv_w=FAKE, dA_log=FAKE, dDskip=FAKE, dconv_w=FAKE, x=FAKE, z=FAKE, dt_raw=FAKE, Bm=FAKE,
               Cm=FAKE, dy=FAKE, dx=FAKE, dz=FAKE, ddt_raw=FAKE, dB=FAKE, dC=FAKE)
    assert lib.mamba_scan_bwd(ctypes.byref(ops.BwdArgs(**dict(bwd, tile_states=FAKE + 8))), None) == \
        ops.MAMBA_ERR_INVALID_ARG
    assert ops.tile_states_shape(2, 33, 64) == (2, 3, 64, 16)
    B, L, D = 1, 40, 32
    x = torch.zeros(B, L, D, dtype=torch.bfloat16)
    bc = torch.zeros(B, L, 16, dtype=torch.bfloat16)
    p = (torch.zeros(D, 16), torch.ones(D), torch.zeros(D, 4))
    for bad in (torch.zeros(B, 2, D, 16), torch.zeros(B, 3, D, 16, dtype=torch.float64),
                torch.zeros(B, D, 3, 16).transpose(1, 2)):
        with pytest.raises(ValueError):
            ops.mamba_scan_fwd(x, x, x, bc, bc, *p, tile_states=bad)
        with pytest.raises(ValueError):
            ops.mamba_scan_bwd(x, x, x, bc, bc, *p, dy=x, tile_states=bad)


CUDA_MSG = "must be on a CUDA device"  # what a CPU tensor meets once every check before it passed


def _scan_cpu(B=1, L=40, D=32, io=torch.bfloat16, N=16, K=4):
    a = dict(x=torch.zeros(B, L, D, dtype=io), z=torch.zeros(B, L, D, dtype=io), dt_raw=torch.zeros(B, L, D, dtype=io),
             Bm=torch.zeros(B, L, 16, dtype=io), Cm=torch.zeros(B, L, 16, dtype=io), A_log=torch.zeros(D, N),
             Dskip=torch.ones(D), conv_w=torch.zeros(D, K), conv_b=torch.zeros(D), h0=torch.zeros(B, D, 16),
             conv_state0=torch.zeros(B, 3, D, dtype=io))
    return a


@pytest.mark.parametrize("fn", ["fwd", "bwd", "noalloc"])
def test_scan_bindings_check_shapes_before_any_device_access(fn):
    """Every tensor's shape and dtype is checked against the sizes passed to
    the C ABI (which sees bare pointers), before any device access."""
    def call(**kw):
        a = dict(_scan_cpu(), **kw)
        args = [a[k] for k in ("x", "z", "dt_raw", "Bm", "Cm", "A_log", "Dskip", "conv_w", "conv_b", "h0",
                               "conv_state0")]
        extra = {k: a[k] for k in a if k not in ("x", "z", "dt_raw", "Bm", "Cm", "A_log", "Dskip", "conv_w",
                                                  "conv_b", "h0", "conv_state0")}
        if fn == "fwd":
            return ops.mamba_scan_fwd(*args, **extra)
        if fn == "bwd":
            extra.setdefault("dy", torch.zeros(1, 40, 32, dtype=torch.bfloat16))
            return ops.mamba_scan_bwd(*args, **extra)
        extra.setdefault("y", torch.zeros(1, 40, 32, dtype=torch.bfloat16))
        return ops.mamba_scan_fwd_noalloc(*args, **extra)

    with pytest.raises(ValueError, match=CUDA_MSG):
        call()  # consistent arguments pass every check
    bad = [dict(z=torch.zeros(1, 39, 32, dtype=torch.bfloat16)), dict(Bm=torch.zeros(1, 40, 8, dtype=torch.bfloat16)),
           dict(Dskip=torch.ones(16)), dict(conv_b=torch.zeros(31)), dict(h0=torch.zeros(1, 32, 8)),
           dict(conv_state0=torch.zeros(1, 4, 32, dtype=torch.bfloat16))]
    if fn == "bwd":
        bad += [dict(dy=torch.zeros(1, 40, 16, dtype=torch.bfloat16)), dict(dfinal_h=torch.zeros(1, 16, 16)),
                dict(out={"dB": torch.zeros(1, 40, 8)})]
    elif fn == "fwd":
        bad += [dict(y=torch.zeros(1, 20, 32, dtype=torch.bfloat16)), dict(final_h=torch.zeros(1, 32, 4))]
    else:
        bad += [dict(y=torch.zeros(1, 20, 32, dtype=torch.bfloat16))]
    for kw in bad:
        with pytest.raises(ValueError, match=next(iter(kw)) if "out" not in kw else "dB"):
            call(**kw)
    for kw in (dict(A_log=torch.zeros(32, 16, dtype=torch.bfloat16)), dict(z=torch.zeros(1, 40, 32))):
        with pytest.raises(TypeError):
            call(**kw)
    # an unsupported state size is the library's to refuse: no shape check
    with pytest.raises(ValueError, match=CUDA_MSG):
        call(A_log=torch.zeros(32, 8))


def test_step_layer_mamba2_bindings_check_shapes():
    B, D = 2, 32
    bf = torch.bfloat16
    st = dict(h=torch.zeros(B, D, 16), conv_state=torch.zeros(B, 3, D, dtype=bf), x_t=torch.zeros(B, D, dtype=bf),
              z_t=torch.zeros(B, D, dtype=bf), dt_raw_t=torch.zeros(B, D, dtype=bf), B_t=torch.zeros(B, 16, dtype=bf),
              C_t=torch.zeros(B, 16, dtype=bf), A_log=torch.zeros(D, 16), Dskip=torch.ones(D),
              conv_w=torch.zeros(D, 4))

    def step(**kw):
        return ops.mamba_step(**dict(st, **kw))

    with pytest.raises(ValueError, match=CUDA_MSG):
        step()
    for kw in (dict(h=torch.zeros(B, D, 8)), dict(conv_state=torch.zeros(B, 2, D, dtype=bf)),
               dict(C_t=torch.zeros(1, 16, dtype=bf)), dict(y_t=torch.zeros(B, D + 1, dtype=bf))):
        with pytest.raises(ValueError, match=next(iter(kw))):
            step(**kw)
    with pytest.raises(ValueError, match=CUDA_MSG):
        step(A_log=torch.zeros(D, 8))  # unsupported: left to the library

    Bt, L, H, Di, R = 1, 16, 64, 32, 8
    lw = dict(hidden=torch.zeros(Bt, L, H, dtype=bf), W_in=torch.zeros(2 * Di, H, dtype=bf), conv_w=torch.zeros(Di, 4),
              conv_b=torch.zeros(Di), W_x=torch.zeros(R + 32, Di, dtype=bf), W_dt=torch.zeros(Di, R, dtype=bf),
              b_dt=torch.zeros(Di, dtype=bf), A_log=torch.zeros(Di, 16), Dskip=torch.ones(Di),
              W_out=torch.zeros(H, Di, dtype=bf))

    def layer(**kw):
        return ops.mamba_layer_fwd(**dict(lw, **kw))

    with pytest.raises(ValueError, match=CUDA_MSG):
        layer()
    for kw in (dict(W_in=torch.zeros(Di, H, dtype=bf)), dict(W_x=torch.zeros(R + 16, Di, dtype=bf)),
               dict(W_out=torch.zeros(Di, H, dtype=bf)), dict(u_out=torch.zeros(Bt, L, H, dtype=bf))):
        with pytest.raises(ValueError, match=next(iter(kw))):
            layer(**kw)
    with pytest.raises(TypeError, match="b_dt"):
        layer(b_dt=torch.zeros(Di))
    with pytest.raises(ValueError, match=CUDA_MSG):
        layer(W_dt=torch.zeros(Di, 6, dtype=bf))  # dt_rank 6: unsupported, left to the library

    Hh, G = 4, 2
    m2 = dict(x=torch.zeros(Bt, L, Hh, 64, dtype=bf), dt_raw=torch.zeros(Bt, L, Hh, dtype=bf), A_log=torch.zeros(Hh),
              Bm=torch.zeros(Bt, L, G, 16, dtype=bf), Cm=torch.zeros(Bt, L, G, 16, dtype=bf), Dskip=torch.ones(Hh))

    def mamba2(**kw):
        return ops.mamba2_scan_fwd(**dict(m2, **kw))

    with pytest.raises(ValueError, match=CUDA_MSG):
        mamba2()
    for kw in (dict(dt_raw=torch.zeros(Bt, L, G, dtype=bf)), dict(Cm=torch.zeros(Bt, L, 1, 16, dtype=bf)),
               dict(h0=torch.zeros(Bt, Hh, 64, 16)), dict(z=torch.zeros(Bt, L, Hh, 32, dtype=bf))):
        with pytest.raises(ValueError, match=next(iter(kw))):
            mamba2(**kw)
    with pytest.raises(ValueError, match=CUDA_MSG):
        mamba2(x=torch.zeros(Bt, L, Hh, 32, dtype=bf))  # head_dim 32: unsupported, left to the library


def test_complex_scan_argument_checks(lib):
    """mamba3_scan_fwd refuses missing or misaligned pointers, an unknown
    discretization, unsupported sizes and a short workspace before anything
    runs (no GPU needed: the pointers are never dereferenced)."""
    full = dict(batch=1, seqlen=64, d_inner=32, d_state=16, d_conv=4, io=ops.MAMBA_BF16, x=FAKE, z=FAKE,
                dt_raw=FAKE, Bm=FAKE, Cm=FAKE, A_log=FAKE, theta=FAKE, Dskip=FAKE, conv_w=FAKE, y=FAKE)

    def call(**kw):
        return lib.mamba3_scan_fwd(ctypes.byref(ops.Mamba3Args(**dict(full, **kw))), None)
    assert lib.mamba3_scan_fwd(None, None) == ops.MAMBA_ERR_INVALID_ARG
    for k in ("x", "z", "dt_raw", "Bm", "Cm", "A_log", "theta", "Dskip", "conv_w", "y"):
        assert call(**{k: 0}) == ops.MAMBA_ERR_INVALID_ARG, k
        assert call(**{k: FAKE + 4}) == ops.MAMBA_ERR_INVALID_ARG, k
    for k in ("h0", "v0", "final_h", "final_v", "conv_b", "conv_state0", "final_conv_state"):
        assert call(**{k: FAKE + 8}) == ops.MAMBA_ERR_INVALID_ARG, k
    assert call(discretization=2) == ops.MAMBA_ERR_UNSUPPORTED
    assert call(d_state=8) == ops.MAMBA_ERR_UNSUPPORTED
    assert call(d_inner=20) == ops.MAMBA_ERR_UNSUPPORTED
    assert call(seqlen=-1) == ops.MAMBA_ERR_INVALID_ARG
    assert call() == ops.MAMBA_ERR_WORKSPACE
    need = ops.mamba3_scan_workspace_size(1, 64, 32, 0)
    assert call(workspace=FAKE, workspace_bytes=need - 1) == ops.MAMBA_ERR_WORKSPACE


def test_complex_scan_workspace(lib):
    def r256(v):
        return (v + 255) // 256 * 256
    # one pass: B and C widened to fp32 (B, L, 32)
    assert ops.mamba3_scan_workspace_size(2, 1000, 64, 1) == r256(2 * 1000 * 32 * 4)
    # chunked: plus the exact mode's chunk end states from zero and dt sums,
    # the entering states (B, n, D, 16), (B, n, D), (B, n, D, 16), and the
    # walked mode's ticket and flags (1 + B * groups * n words)
    B, L, D, n = 1, 4096, 64, 4
    need = B * L * 32 * 4 + B * n * D * 16 * 4 + B * n * D * 4 + B * n * D * 16 * 4 + (1 + B * (D // 32) * n) * 4
    ws = ops.mamba3_scan_workspace_size(B, L, D, n)
    assert need <= ws <= need + 5 * 256
    assert ops.mamba3_scan_workspace_size(1, 0, 64, 0) == 0
    assert ops.mamba3_scan_workspace_size(1, 64, 22, 0) == 0  # no I/O type takes rows of 22 channels
    assert ops.mamba3_scan_workspace_size(1, 64, 24, 0) > 0


def test_linear_argument_checks(lib):
    full = dict(M=256, N=256, K=128, A=FAKE, lda=128, W=FAKE, C=FAKE, ldc=256)

    def call(**kw):
        return lib.mamba_linear_fwd(ctypes.byref(ops.LinearArgs(**dict(full, **kw))), None)
    assert lib.mamba_linear_fwd(None, None) == ops.MAMBA_ERR_INVALID_ARG
    for k in ("A", "W", "C"):
        assert call(**{k: 0}) == ops.MAMBA_ERR_INVALID_ARG, k
        assert call(**{k: FAKE + 8}) == ops.MAMBA_ERR_INVALID_ARG, k
    assert call(bias=FAKE + 2) == ops.MAMBA_ERR_INVALID_ARG
    assert call(K=36, lda=40) == ops.MAMBA_ERR_UNSUPPORTED
    assert call(lda=132) == ops.MAMBA_ERR_UNSUPPORTED
    assert call(ldc=260) == ops.MAMBA_ERR_UNSUPPORTED
    assert call(lda=64) == ops.MAMBA_ERR_INVALID_ARG
    assert call(ldc=128) == ops.MAMBA_ERR_INVALID_ARG
    assert call(M=-1) == ops.MAMBA_ERR_INVALID_ARG
    assert call(M=0) == ops.MAMBA_OK  # nothing to do, nothing touched
