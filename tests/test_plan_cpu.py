"""The host-side work plan and workspace sizes of the prefill scan and its
backward, over many sizes (hypothesis), without a GPU: the plan covers the
sequence in whole 16-token tiles, its carry pieces cover a chunk, an explicit
chunk count is honoured as a bound, and the workspace sizes equal the
documented layouts summed here independently."""
import pytest
from hypothesis import given, settings, strategies as st

from selective_state_space_118_b300 import ops

T = 16  # tokens per tile


def r256(v):
    return (v + 255) // 256 * 256


def fwd_workspace(B, L, D, n):
    """B/C rows widened to fp32 (B, L, 32); in chunked mode the carries
    (B, n, D, 16) and the counters (a ticket and one flag per (row, group,
    chunk))."""
    total = r256(B * L * 32 * 4)
    if n <= 1:
        return total
    counters = r256(total + B * n * D * 16 * 4)
    return r256(counters + (1 + B * -(-D // 32) * n) * 4)  # groups of 32 channels, rounded up


def bwd_workspace(B, L, D, n):
    """The forward's workspace, the tile states (B, tiles, D, 16), chunked:
    the adjoint carries and their counters; the per-group dB | dC sums, the
    per-chunk parameter partials (B n, D, 24) and, chunked, the conv edge
    buffers (B, n, 3, D) twice."""
    G = -(-D // 32)
    o = fwd_workspace(B, L, D, n)
    o = r256(o + B * (-(-L // T)) * D * 16 * 4)
    if n > 1:
        o = r256(o + B * n * D * 16 * 4)
        o = r256(o + (1 + B * G * n) * 4)
    o = r256(o + G * B * L * 32 * 4)
    o = r256(o + B * n * D * 24 * 4)
    if n > 1:
        o = r256(o + B * n * 3 * D * 4)
        o = r256(o + B * n * 3 * D * 4)
    return o


sizes = st.tuples(st.integers(1, 4), st.integers(1, 300_000), st.integers(1, 4096).map(lambda k: 4 * k),
                  st.integers(0, 80))


@settings(max_examples=300, deadline=None, derandomize=True)
@given(sizes)
def test_plan_invariants(s):
    B, L, D, n_req = s
    pl = ops.mamba_scan_plan(B, L, D, n_req)
    n, C, m, P = pl["n_chunks"], pl["chunk_len"], pl["pieces"], pl["piece_len"]
    tiles = -(-L // T)
    assert n >= 1 and C % T == 0
    assert n * C >= tiles * T and (n - 1) * C < L  # every chunk holds tokens, the chunks cover L
    if n_req == 1 or tiles == 1:
        assert n == 1
    if n_req >= 1:
        assert n <= n_req
    else:
        assert n <= 64 and n == ops.mamba_scan_default_chunks(B, L, D)
    if n > 1:
        assert P % T == 0 and 0 < P <= 256
        assert m * P >= C > (m - 1) * P  # the carry pieces cover one chunk
    else:
        assert (m, P) == (0, 0) and C == tiles * T


@settings(max_examples=300, deadline=None, derandomize=True)
@given(sizes)
def test_workspace_sizes_follow_the_layouts(s):
    B, L, D, n_req = s
    n = ops.mamba_scan_plan(B, L, D, n_req)["n_chunks"]
    assert ops.mamba_scan_workspace_size(B, L, D, n_req) == fwd_workspace(B, L, D, n)
    assert ops.mamba_scan_bwd_workspace_size(B, L, D, n_req) == bwd_workspace(B, L, D, n)


@pytest.mark.parametrize("args", [(0, 10, 16, 0), (1, 0, 16, 0), (1, 10, 0, 0), (1, 10, 22, 0), (1, 10, 16, -1)])
def test_sizes_without_a_plan(args):
    assert ops.mamba_scan_workspace_size(*args) == 0
    assert ops.mamba_scan_bwd_workspace_size(*args) == 0


@settings(max_examples=200, deadline=None, derandomize=True)
@given(sizes, st.integers(1, 64).map(lambda k: 8 * k), st.booleans())
def test_layer_workspace_follows_its_layout(s, R, with_u_out):
    """x, z, u (unless the caller takes u), the x_proj output (rows, R + 32),
    dt_raw and y, all bf16; then the scan's workspace."""
    B, L, D, n_req = s
    H = 2 * D
    act = r256(B * L * D * 2)
    n = ops.mamba_scan_plan(B, L, D, n_req)["n_chunks"]
    want = (4 if with_u_out else 5) * act + r256(B * L * (R + 32) * 2) + fwd_workspace(B, L, D, n)
    assert ops.mamba_layer_workspace_size(B, L, H, D, R, n_req, with_u_out) == want


@settings(max_examples=200, deadline=None, derandomize=True)
@given(st.integers(1, 8), st.integers(1, 300_000), st.integers(1, 256))
def test_mamba2_workspace_follows_its_layout(B, L, H):
    """Per (row, head, 128-token chunk): the chunk's end state and entering
    state (16 x 64 fp32 each), its decay sum, and per token the dt and decay
    prefix (128 x 2 fp32)."""
    k = B * H * -(-L // 128)
    assert ops.mamba2_scan_workspace_size(B, L, H) == 2 * r256(k * 16 * 64 * 4) + r256(k * 4) + r256(k * 128 * 2 * 4)


@pytest.mark.parametrize("L,n_best", [(4096, 10), (32768, 9), (262144, 9)])
def test_default_plan_at_the_measured_shapes(L, n_best):
    """At 8,192 channels, batch 1, on a 148-SM B300 (16 one-warp tasks per
    SM), the default plan takes the chunk counts that measured fastest:
    4,096-token calls 10 chunks (8-12 chunks: 17.6, 16.1, 15.5, 16.9, 17.6 ms
    per 64 calls), 32k 9 (9-12: 1.28, 1.37-1.41, 1.32, 1.41 ms), 256k in
    one call 9."""
    import torch
    if torch.cuda.is_available() and torch.cuda.get_device_properties(0).multi_processor_count != 148:
        pytest.skip("the counts were measured on a 148-SM device")
    pl = ops.mamba_scan_plan(1, L, 8192, 0)
    assert pl["n_chunks"] == n_best
    assert pl["piece_len"] == 64
