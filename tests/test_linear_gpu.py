"""The tensor-core linear map (mamba_linear_fwd: hand-written tcgen05 GEMM)
through the C ABI, against its plain definition in fp64: C = A W^T + bias
from the same bf16 inputs (numpy matmul), rounded to bf16 the way the
library stores an fp32 result.  The fp32 accumulation order differs, so a
value close to a rounding boundary may land on the neighbouring bf16 value:
every element must be within one bf16 ulp of the rounded definition (2^-7 of
its magnitude bounds that) plus 1e-4 of the rms."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_118_b300 import ops

pytestmark = pytest.mark.gpu


def ulp_close(gpu, ref, what):
    g = oracle.f64(gpu)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    rms = float(np.sqrt(np.mean(ref * ref))) or 1.0
    excess = np.abs(g - ref) - (2.0 ** -7 * np.abs(ref) + 1e-4 * rms)
    assert excess.max() <= 0.0, f"{what}: {excess.max() / rms:.2e} of the rms beyond one ulp"


def case(M, N, K, seed, bias=True, lda=None, ldc=None):
    g = torch.Generator(device="cuda").manual_seed(seed)
    bf = torch.bfloat16
    lda = lda or K
    Abig = (torch.randn(M, lda, device="cuda", generator=g)).to(bf)
    A = Abig[:, :K]
    W = (torch.randn(N, K, device="cuda", generator=g) * K ** -0.5).to(bf)
    b = (torch.randn(N, device="cuda", generator=g)).to(bf) if bias else None
    out = None
    if ldc:
        out = torch.empty(M, ldc, device="cuda", dtype=bf)[:, :N]
    return A, W, b, out


def reference(A, W, b):
    r = oracle.f64(A) @ oracle.f64(W).T
    if b is not None:
        r = r + oracle.f64(b)
    return oracle.bf16_round(r)


SHAPES = [
    # (M, N, K, bias, lda, ldc)
    (128, 256, 64, False, None, None),     # one tile, one K block
    (256, 512, 128, True, None, None),
    (300, 288, 192, True, None, None),     # row and column tails (x_proj's width)
    (1000, 1000, 256, True, None, None),   # a column tail not a multiple of 32
    (517, 256, 320, False, 384, 264),      # strided A and C (views of wider matrices)
    (4096, 4096, 1024, True, None, None),  # many tiles per CTA: both accumulators, the stage ring wraps
    (700, 512, 96, True, None, None),      # K not a multiple of 64: the last K block is zero-filled
    (257, 320, 32, False, 288, None),      # K = 32 read from a wider row (dt_proj's input layout)
]


@pytest.mark.parametrize("M,N,K,bias,lda,ldc", SHAPES)
def test_linear_against_definition(M, N, K, bias, lda, ldc):
    A, W, b, out = case(M, N, K, seed=M + N + K, bias=bias, lda=lda, ldc=ldc)
    C = ops.mamba_linear_fwd(A, W, b, out=out)
    torch.cuda.synchronize()
    assert ops.mamba_last_error() == ops.MAMBA_OK
    ulp_close(C, reference(A, W, b), f"M{M} N{N} K{K}")


def test_linear_layer_shapes_sampled_rows():
    """The layer's projection shapes at the Jamba size (M = 32,768 tokens): the
    full product on the GPU, sampled rows against the definition."""
    rows = np.unique(np.linspace(0, 32767, 40).round().astype(np.int64))
    for N, K in ((8192, 4096), (4096, 8192), (288, 8192), (8192, 256)):
        A, W, b, _ = case(32768, N, K, seed=N + K, bias=(K == 256))
        C = ops.mamba_linear_fwd(A, W, b)
        torch.cuda.synchronize()
        idx = torch.as_tensor(rows, device="cuda")
        ulp_close(C.index_select(0, idx), reference(A.index_select(0, idx), W, b), f"N{N} K{K}")
        del A, W, C
    assert ops.mamba_last_error() == ops.MAMBA_OK


def test_linear_empty_and_refusals():
    A, W, b, _ = case(0, 256, 64, seed=1)
    C = ops.mamba_linear_fwd(A, W, b)
    assert C.shape == (0, 256)
    A, W, b, _ = case(64, 256, 36, seed=2)
    with pytest.raises(ops.MambaError) as e:
        ops.mamba_linear_fwd(A, W, b)
    assert e.value.status == ops.MAMBA_ERR_UNSUPPORTED
