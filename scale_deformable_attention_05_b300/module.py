"""MSDeformAttn layer: the projections around the fused CUDA operator.

The layer of the Deformable DETR walk-through ("2.2.4 源码分析",
MSDeformAttn): four linear maps of width d_model and the sampling between
them,

    value   = value_proj(input_flatten)               [N, Len_in, M, D]
    offsets = sampling_offsets(query)                 [N, Len_q, M, L, P, 2]
    logits  = attention_weights(query)                [N, Len_q, M, L*P]
    out     = output_proj(msda(value masked by input_padding_mask,
                               softmax(logits), reference_points + offsets))

The four projections are dense GEMMs.  They run on the library's tensor-core
kernels (tcgen05.mma with the accumulator in tensor memory) for the forward and
for the input gradient (x-gradient = grad_y times the weight, i.e. the same
kernel with the transposed weight): ``msda_linear`` in bf16 and fp16,
``msda_linear_f32`` (three TF32 products per step, fp32 accuracy) in fp32.  The weight and bias
gradients (reductions over all tokens) use ``msda_linear_wgrad_f32`` in fp32;
in bf16 and fp16 the weight gradient uses torch (cuBLAS) and the bias gradient
``msda_linear_bias_grad``.  Everything between the projections -- masking,
softmax, locations from 2-d or 4-d reference points, bilinear sampling and
their backward -- is one launch of the fused entry points of ``libmsda.so``
each way.  The tensors the GEMMs produce are already in the operator's
layouts, so nothing is copied or transposed between them.
"""
from __future__ import annotations

import math
from typing import Optional

import torch
from torch import nn

from . import binding as B


_TC_DTYPES = (torch.bfloat16, torch.float16, torch.float32)


def _tensor_core_shape(in_features: int, out_features: int, dtype=torch.bfloat16) -> bool:
    k_step = 16 if dtype == torch.float32 else 64         # the kernels' K block
    return (in_features % k_step == 0 and out_features % 16 == 0 and
            in_features <= B.MSDA_LINEAR_MAX_FEATURES and
            out_features <= B.MSDA_LINEAR_MAX_FEATURES)


def _tc_linear(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor]) -> torch.Tensor:
    if x.dtype == torch.float32:
        return B.msda_linear_f32(x, weight, bias)
    return B.msda_linear(x, weight, bias)


class TensorCoreLinear(torch.autograd.Function):
    """y = x w^T + b with x and w of one dtype (bf16, fp16 or fp32) on the tensor
    cores (msda_linear / msda_linear_f32); the input gradient through the same
    kernel with w^T when its shape allows (else a cuBLAS matmul); the weight and
    bias gradients on the tensor cores in fp32 (msda_linear_wgrad_f32); in bf16
    and fp16 the weight gradient with torch (cuBLAS) and the bias gradient with
    msda_linear_bias_grad."""

    @staticmethod
    def forward(ctx, x, weight, bias):
        ctx.save_for_backward(x, weight)
        ctx.has_bias = bias is not None
        return _tc_linear(x.contiguous(), weight, bias)

    @staticmethod
    def backward(ctx, grad_y):
        x, weight = ctx.saved_tensors
        n_out, n_in = weight.shape
        gy = grad_y.contiguous()
        if _tensor_core_shape(n_out, n_in, weight.dtype):
            gx = _tc_linear(gy, weight.t().contiguous(), None)
        else:
            gx = gy @ weight
        g2 = gy.reshape(-1, n_out)
        if weight.dtype == torch.float32:
            gw, gb = B.msda_linear_wgrad_f32(g2, x.reshape(-1, n_in).contiguous(),
                                             bias=ctx.has_bias)
            return gx, gw, gb
        gw = g2.t() @ x.reshape(-1, n_in)
        gb = B.msda_linear_bias_grad(g2).to(weight.dtype) if ctx.has_bias else None
        return gx, gw, gb


def project(linear: nn.Linear, x: torch.Tensor, tensor_cores: bool = True) -> torch.Tensor:
    """linear(x), on the tensor-core kernels for bf16, fp16 or fp32 operands of supported widths."""
    if (tensor_cores and x.is_cuda and x.dtype in _TC_DTYPES and
            linear.weight.dtype == x.dtype and
            _tensor_core_shape(linear.in_features, linear.out_features, x.dtype)):
        if torch.is_grad_enabled() and (x.requires_grad or linear.weight.requires_grad):
            return TensorCoreLinear.apply(x, linear.weight, linear.bias)
        return _tc_linear(x.contiguous(), linear.weight, linear.bias)
    return linear(x)


class MSDeformAttn(nn.Module):
    """Multi-scale deformable attention with d_model channels split into
    n_heads heads, sampling n_points points on each of n_levels levels.
    tensor_core_projections: projections on the library's tensor-core kernels
    (True) or on torch.nn.Linear (False)."""

    tensor_core_projections = True

    def __init__(self, d_model: int = 256, n_levels: int = 4, n_heads: int = 8,
                 n_points: int = 4):
        super().__init__()
        if d_model % n_heads != 0:
            raise ValueError(f"d_model {d_model} is not a multiple of n_heads {n_heads}")
        head_dim = d_model // n_heads
        if head_dim % 8 != 0:
            raise ValueError(f"head_dim {head_dim} must be a multiple of 8 (16-byte rows)")
        if n_levels * n_points > B.MSDA_MAX_FUSED_LEVEL_POINTS:
            raise ValueError(f"n_levels * n_points must be <= {B.MSDA_MAX_FUSED_LEVEL_POINTS}")
        self.d_model, self.n_levels, self.n_heads, self.n_points = d_model, n_levels, n_heads, n_points
        self.sampling_offsets = nn.Linear(d_model, n_heads * n_levels * n_points * 2)
        self.attention_weights = nn.Linear(d_model, n_heads * n_levels * n_points)
        self.value_proj = nn.Linear(d_model, d_model)
        self.output_proj = nn.Linear(d_model, d_model)
        self.reset_parameters()

    @torch.no_grad()
    def reset_parameters(self) -> None:
        """The walk-through's initial state: offset and attention weights zero,
        so every query starts from fixed offsets and uniform attention.  Head h
        looks along the direction at angle 2*pi*h/n_heads, scaled so its larger
        component is 1; point p sits p+1 steps out along it, on every level.
        Value and output projections: Xavier-uniform weights, zero bias."""
        nn.init.zeros_(self.sampling_offsets.weight)
        theta = torch.arange(self.n_heads, dtype=torch.float64) * (2.0 * math.pi / self.n_heads)
        direction = torch.stack([theta.cos(), theta.sin()], -1)
        direction = direction / direction.abs().max(-1, keepdim=True).values
        steps = torch.arange(1, self.n_points + 1, dtype=torch.float64)
        bias = direction[:, None, None, :] * steps[None, None, :, None]          # [M, 1, P, 2]
        bias = bias.expand(self.n_heads, self.n_levels, self.n_points, 2)
        self.sampling_offsets.bias.copy_(bias.reshape(-1))
        nn.init.zeros_(self.attention_weights.weight)
        nn.init.zeros_(self.attention_weights.bias)
        nn.init.xavier_uniform_(self.value_proj.weight)
        nn.init.zeros_(self.value_proj.bias)
        nn.init.xavier_uniform_(self.output_proj.weight)
        nn.init.zeros_(self.output_proj.bias)

    def forward(self, query: torch.Tensor, reference_points: torch.Tensor,
                input_flatten: torch.Tensor, input_spatial_shapes: torch.Tensor,
                input_level_start_index: torch.Tensor,
                input_padding_mask: Optional[torch.Tensor] = None) -> torch.Tensor:
        """query [N, Len_q, d_model]; reference_points [N, Len_q, n_levels, 2]
        (normalised x, y) or [..., 4] (boxes x, y, w, h); input_flatten
        [N, Len_in, d_model] with Len_in = sum of H*W; input_padding_mask
        [N, Len_in] bool (True = padded) or None.  Returns [N, Len_q, d_model]."""
        N, Len_q, _ = query.shape
        Len_in = input_flatten.shape[1]
        M, L, P = self.n_heads, self.n_levels, self.n_points
        tc = self.tensor_core_projections
        value = project(self.value_proj, input_flatten, tc).view(N, Len_in, M, self.d_model // M)
        offsets = project(self.sampling_offsets, query, tc).view(N, Len_q, M, L, P, 2)
        logits = project(self.attention_weights, query, tc).view(N, Len_q, M, L * P)
        out = B.ms_deform_attn_fused(value, input_spatial_shapes, input_level_start_index,
                                     reference_points, offsets, logits, input_padding_mask)
        return project(self.output_proj, out, tc)
