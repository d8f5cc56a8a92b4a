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


# ----------------------------------------------------------------------------- fp32 (3 x TF32)
# msda_linear_f32 against the same fp64 product.  Bound, from the arithmetic:
# x = x_hi + x_lo exactly with |x_lo| <= 2^-11 |x| (TF32 keeps 10 explicit
# mantissa bits, rounded to nearest); the three products miss x_lo w_lo
# (<= 2^-22 |x||w|) and read the remainders as TF32 (<= 2^-10 of each, so
# <= 2^-21 |x||w| twice): <= 2^-19.4 |x||w| per term.  The fp32 accumulation
# of K <= 256 terms adds at most K u S with u = 2^-24 and S = sum |x||w|, but
# sums of signed random terms stay near u S; the test allows 2^-18 S, which a
# single TF32 product (about 2^-12 |x||w| per term) exceeds.

def _check_f32(B, rows, k, n, bias=True, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, k, generator=g)
    w = torch.randn(n, k, generator=g) / np.sqrt(k)
    b = torch.randn(n, generator=g) if bias else None
    y = B.msda_linear_f32(x.cuda(), w.cuda(), b.cuda() if bias else None)
    torch.cuda.synchronize()
    assert B.msda_last_device_error() == 0
    xd, wd = x.double().numpy(), w.double().numpy()
    ref = xd @ wd.T + (b.double().numpy() if bias else 0.0)
    s = np.abs(xd) @ np.abs(wd).T
    err = np.abs(y.cpu().double().numpy() - ref)
    bound = 2.0 ** -18 * s + (2.0 ** -23 * np.abs(b.double().numpy()) if bias else 0.0)
    assert (err <= bound).all(), f"max err {err.max():.3e}, worst excess {(err - bound).max():.3e}"
    return err, s


@pytest.mark.parametrize("rows,k,n", [
    (128, 256, 256),          # one full tile
    (300, 256, 256),          # a ragged last tile
    (1, 32, 16),              # smallest shapes
    (1000, 256, 128),         # attention-weight projection width
    (517, 96, 80),            # K of six 16-column stages, N not a power of two
    (300, 48, 144),           # K of three stages, N past one 128-column half
    (44446, 256, 256),        # encoder tokens x d_model: many tiles per CTA
])
def test_linear_f32_matches_fp64(B, rows, k, n):
    _check_f32(B, rows, k, n, seed=rows + k + n)


def test_linear_f32_is_more_accurate_than_one_tf32_product(B):
    """The split matters: the error stays far below what TF32 operands alone give."""
    err, s = _check_f32(B, 2048, 256, 256, bias=False, seed=11)
    g = torch.Generator().manual_seed(11)
    x = torch.randn(2048, 256, generator=g)
    w = torch.randn(256, 256, generator=g) / 16
    tf32 = lambda a: (a.view(torch.int32) + 0x1000 & ~0x1FFF).view(torch.float32)  # round to 10 bits
    one = tf32(x).double() @ tf32(w).double().T
    err1 = (one - x.double() @ w.double().T).abs().numpy()
    assert err.max() * 16 < err1.max()


def test_linear_f32_without_bias_batched_and_checks(B):
    _check_f32(B, 257, 128, 64, bias=False, seed=3)
    g = torch.Generator().manual_seed(5)
    x = torch.randn(2, 37, 256, generator=g).cuda()
    w = torch.randn(128, 256, generator=g).cuda()
    ws = torch.empty(B.msda_linear_workspace_bytes(74, 256, 128), dtype=torch.uint8, device="cuda")
    y = B.msda_linear_f32(x, w, workspace=ws)
    ref = x.double() @ w.double().T
    torch.cuda.synchronize()
    assert y.shape == (2, 37, 128)
    assert (y.double() - ref).abs().max().item() <= 2.0 ** -18 * (x.abs().double() @ w.abs().double().T).max().item()
    with pytest.raises(B.MsdaError) as e:
        B.msda_linear_f32(x, w, workspace=ws[:-16])           # workspace one chunk short
    assert e.value.status == 5
    with pytest.raises(B.MsdaError) as e:
        B.msda_linear_f32(torch.zeros(8, 40, device="cuda"), torch.zeros(16, 40, device="cuda"))
    assert e.value.status == 3                                 # in_features not a multiple of 16


# ------------------------------------------------------ fp32 weight gradient (3 x TF32)
# msda_linear_wgrad_f32 against grad_w = gy^T x and grad_b = sum gy in fp64.  The
# split contributes <= 2^-19.4 |gy||x| per term, as above; the partial sums of up
# to 148 CTAs (each over a contiguous range of rows) are added with fp32
# reductions, each rounding by <= 2^-24 of the running sum: allowed 2^-16 of
# S = |gy|^T |x| for grad_w, and 2^-16 of sum |gy| for grad_b (a thread's
# sequential sum over its rows, then the same reductions).

def _check_wgrad(B, rows, k, n, seed, accumulate=False):
    g = torch.Generator().manual_seed(seed)
    gy = torch.randn(rows, n, generator=g)
    x = torch.randn(rows, k, generator=g)
    w0 = torch.randn(n, k, generator=g) if accumulate else None
    b0 = torch.randn(n, generator=g) if accumulate else None
    if accumulate:
        gw, gb = B.msda_linear_wgrad_f32(gy.cuda(), x.cuda(), grad_w=w0.cuda(), grad_b=b0.cuda(),
                                         accumulate=True)
    else:
        gw, gb = B.msda_linear_wgrad_f32(gy.cuda(), x.cuda())
    torch.cuda.synchronize()
    assert B.msda_last_device_error() == 0
    gyd, xd = gy.double().numpy(), x.double().numpy()
    ref_w = gyd.T @ xd + (w0.double().numpy() if accumulate else 0.0)
    ref_b = gyd.sum(0) + (b0.double().numpy() if accumulate else 0.0)
    s = np.abs(gyd).T @ np.abs(xd) + (np.abs(w0.double().numpy()) if accumulate else 0.0)
    sb = np.abs(gyd).sum(0) + (np.abs(b0.double().numpy()) if accumulate else 0.0)
    err_w = np.abs(gw.cpu().double().numpy() - ref_w)
    err_b = np.abs(gb.cpu().double().numpy() - ref_b)
    assert (err_w <= 2.0 ** -16 * s).all(), f"grad_w max err {err_w.max():.3e}"
    assert (err_b <= 2.0 ** -16 * sb).all(), f"grad_b max err {err_b.max():.3e}"
    return err_w, s


@pytest.mark.parametrize("rows,k,n", [
    (16, 16, 16),             # one block of rows, smallest widths
    (300, 256, 256),          # two column tiles of grad_y, ragged last block
    (1000, 256, 128),         # one column tile (attention-weight projection width)
    (517, 96, 80),            # widths that are not powers of two
    (44446, 256, 256),        # encoder tokens: every CTA sums ~600 rows
])
def test_linear_wgrad_f32_matches_fp64(B, rows, k, n):
    _check_wgrad(B, rows, k, n, seed=rows + 3 * k + n)


def test_linear_wgrad_f32_accumulates_and_beats_one_tf32_product(B):
    _check_wgrad(B, 777, 128, 144, seed=21, accumulate=True)
    err, s = _check_wgrad(B, 64, 256, 256, seed=22)
    g = torch.Generator().manual_seed(22)
    gy, x = torch.randn(64, 256, generator=g), torch.randn(64, 256, generator=g)
    tf32 = lambda a: (a.view(torch.int32) + 0x1000 & ~0x1FFF).view(torch.float32)
    err1 = (tf32(gy).double().T @ tf32(x).double() - gy.double().T @ x.double()).abs().numpy()
    assert err.max() * 16 < err1.max()


def test_linear_wgrad_f32_without_bias_and_checks(B):
    gy = torch.randn(40, 32, device="cuda")
    x = torch.randn(40, 48, device="cuda")
    gw, gb = B.msda_linear_wgrad_f32(gy, x, bias=False)
    torch.cuda.synchronize()
    assert gb is None
    ref = gy.double().T @ x.double()
    assert (gw.double() - ref).abs().max().item() <= 2.0 ** -16 * (gy.abs().double().T @ x.abs().double()).max().item()
    with pytest.raises(B.MsdaError) as e:
        B.msda_linear_wgrad_f32(torch.zeros(8, 24, device="cuda"), torch.zeros(8, 32, device="cuda"))
    assert e.value.status == 3                                 # out_features not a multiple of 16


# ------------------------------------------------------------------ bias gradient
# msda_linear_bias_grad: fp32 column sums of grad_y against fp64.  Each sum is a
# thread's sequential sum over its rows, a sum over the CTA's row lanes and the
# CTAs' atomic additions, each rounding by <= 2^-24 of its running sum; a few
# hundred roundings at most: allowed 2^-14 of sum |grad_y|.

@pytest.mark.parametrize("rows,n,dtype", [
    (1, 16, torch.bfloat16), (88892, 256, torch.bfloat16), (44446, 256, torch.float32),
    (1000, 128, torch.float16), (517, 40, torch.float32), (300, 2048, torch.bfloat16),
])
def test_linear_bias_grad_matches_fp64(B, rows, n, dtype):
    g = torch.Generator().manual_seed(rows + n)
    gy = torch.randn(rows, n, generator=g).to(dtype)
    gb = B.msda_linear_bias_grad(gy.cuda())
    torch.cuda.synchronize()
    ref = gy.double().sum(0).numpy()
    err = np.abs(gb.cpu().double().numpy() - ref)
    assert (err <= 2.0 ** -14 * gy.double().abs().sum(0).numpy()).all(), err.max()


def test_linear_bias_grad_accumulates_and_checks(B):
    gy = torch.randn(70, 64, device="cuda")
    acc = torch.ones(64, device="cuda")
    B.msda_linear_bias_grad(gy, grad_b=acc, accumulate=True)
    torch.cuda.synchronize()
    assert torch.allclose(acc.double(), 1 + gy.double().sum(0), atol=1e-4)
    with pytest.raises(B.MsdaError) as e:
        B.msda_linear_bias_grad(torch.zeros(4, 12, dtype=torch.bfloat16, device="cuda"))
    assert e.value.status == 3                        # 12 bf16 columns: not whole 16-byte vectors


def test_linear_fp16_operands(B):
    """fp16 x and w (kind::f16 with f16 operands), fp32 and fp16 bias: the same
    bound with fp16's unit roundoff (one rounding of the result, 2^-11 relative)."""
    for rows, k, n, seed in ((300, 256, 256, 31), (1000, 64, 80, 32)):
        g = torch.Generator().manual_seed(seed)
        x = torch.randn(rows, k, generator=g).to(torch.float16)
        w = (torch.randn(n, k, generator=g) / np.sqrt(k)).to(torch.float16)
        for b in (torch.randn(n, generator=g), torch.randn(n, generator=g).to(torch.float16)):
            y = B.msda_linear(x.cuda(), w.cuda(), b.cuda())
            torch.cuda.synchronize()
            assert y.dtype == torch.float16
            ref = x.double().numpy() @ w.double().numpy().T + b.double().numpy()
            err = np.abs(y.double().cpu().numpy() - ref)
            assert (err <= 2.0 ** -10 * np.abs(ref) + 1e-4 * np.abs(ref).max()).all(), err.max()
