"""msda_linear, the tensor-core projection (tcgen05.mma, bf16 operands, fp32
accumulation in tensor memory), against y = x w^T + bias in fp64 on the host.

Tolerance, derived from the arithmetic: the operands are exact bf16 values and
the products are summed in fp32 (relative rounding ~6e-8 per addition, K <= 256
terms), then rounded once to bf16 (relative error <= 2^-9): |err| <= 2^-8 |ref|
+ 1e-4 max|ref| element-wise (the second term covers results that cancel).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_05_b300 import binding
    return binding


def _check(B, rows, k, n, bias=True, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(n, k, generator=g) / np.sqrt(k)).to(torch.bfloat16)
    b = torch.randn(n, generator=g) if bias else None
    y = B.msda_linear(x.cuda(), w.cuda(), b.cuda() if bias else None)
    torch.cuda.synchronize()
    assert B.msda_last_device_error() == 0
    ref = x.double().numpy() @ w.double().numpy().T + (b.double().numpy() if bias else 0.0)
    got = y.float().cpu().double().numpy()
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-4 * np.abs(ref).max()
    assert (err <= bound).all(), f"max err {err.max():.3e}, worst excess {(err - bound).max():.3e}"


@pytest.mark.parametrize("rows,k,n", [
    (128, 256, 256),          # one full tile
    (300, 256, 256),          # a ragged last tile (decoder queries)
    (1, 64, 16),              # smallest shapes
    (1000, 256, 128),         # attention-weight projection width (M * L * P)
    (517, 192, 80),           # K of three swizzle atoms, N not a power of two
    (44446, 256, 256),        # encoder tokens x d_model: many tiles per CTA
])
def test_linear_matches_fp64(B, rows, k, n):
    _check(B, rows, k, n, seed=rows + k + n)


def test_linear_without_bias_and_batched_input(B):
    _check(B, 257, 128, 64, bias=False, seed=3)
    g = torch.Generator().manual_seed(4)
    x = torch.randn(2, 37, 256, generator=g).to(torch.bfloat16).cuda()
    w = torch.randn(256, 256, generator=g).to(torch.bfloat16).cuda()
    y = B.msda_linear(x, w)
    ref = (x.double() @ w.double().T).float()
    torch.cuda.synchronize()
    assert y.shape == (2, 37, 256)
    assert torch.allclose(y.float(), ref, rtol=2 ** -8, atol=1e-4 * ref.abs().max().item())


def test_linear_rejects_unsupported_shapes(B):
    x = torch.zeros(8, 32, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(16, 32, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.MsdaError) as e:
        B.msda_linear(x, w)                       # in_features not a multiple of 64
    assert e.value.status == 3
    x = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(24, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.MsdaError) as e:
        B.msda_linear(x, w)                       # out_features not a multiple of 16
    assert e.value.status == 3


def test_linear_bf16_bias(B):
    """The bias may be the bf16 parameter of a bf16 layer (widened in the kernel)."""
    g = torch.Generator().manual_seed(9)
    x = torch.randn(300, 256, generator=g).to(torch.bfloat16)
    w = (torch.randn(128, 256, generator=g) / 16).to(torch.bfloat16)
    b = torch.randn(128, generator=g).to(torch.bfloat16)
    y = B.msda_linear(x.cuda(), w.cuda(), b.cuda())
    torch.cuda.synchronize()
    ref = x.double().numpy() @ w.double().numpy().T + b.double().numpy()
    err = np.abs(y.float().cpu().double().numpy() - ref)
    assert (err <= 2.0 ** -8 * np.abs(ref) + 1e-4 * np.abs(ref).max()).all()
