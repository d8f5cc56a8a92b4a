"""O2b: the pages' own library formulation, restated in fp64 on the CPU (TEST INFRASTRUCTURE).

Deformable DETR walk-through, "2.2.4 源码分析", ``ms_deform_attn_core_pytorch``:
the value tensor is split per level, each level is viewed as an image batch of
(batch*heads) images with head_dim channels, sampled with
``torch.nn.functional.grid_sample(bilinear, zeros, align_corners=False)`` at
grid = 2*loc - 1, and the samples are weighted by the attention weights and
summed over levels and points.  Written here from that description (not
copied), in float64 on the CPU, so that torch.autograd gives an independent
fp64 backward.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def _forward_torch(value, spatial_shapes, level_start_index, loc, attn):
    bs, K, M, D = value.shape
    _, Q, _, L, P, _ = loc.shape
    grids = 2.0 * loc - 1.0
    acc = torch.zeros(bs * M, D, Q, dtype=value.dtype)
    for l in range(L):
        H, W = int(spatial_shapes[l][0]), int(spatial_shapes[l][1])
        s = int(level_start_index[l])
        # [bs, H*W, M, D] -> [bs*M, D, H, W]
        img = value[:, s:s + H * W].permute(0, 2, 3, 1).reshape(bs * M, D, H, W)
        # [bs, Q, M, P, 2] -> [bs*M, Q, P, 2]
        grid = grids[:, :, :, l].permute(0, 2, 1, 3, 4).reshape(bs * M, Q, P, 2)
        samp = F.grid_sample(img, grid, mode="bilinear", padding_mode="zeros",
                             align_corners=False)                       # [bs*M, D, Q, P]
        w = attn[:, :, :, l].permute(0, 2, 1, 3).reshape(bs * M, 1, Q, P)
        acc = acc + (samp * w).sum(-1)
    # [bs*M, D, Q] -> [bs, Q, M*D]
    return acc.reshape(bs, M, D, Q).permute(0, 3, 1, 2).reshape(bs, Q, M * D)


def forward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights):
    with torch.no_grad():
        out = _forward_torch(torch.as_tensor(np.asarray(value, np.float64)),
                             np.asarray(spatial_shapes), np.asarray(level_start_index),
                             torch.as_tensor(np.asarray(sampling_locations, np.float64)),
                             torch.as_tensor(np.asarray(attention_weights, np.float64)))
    return out.numpy()


def backward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
             grad_output):
    v = torch.tensor(np.asarray(value, np.float64), requires_grad=True)
    loc = torch.tensor(np.asarray(sampling_locations, np.float64), requires_grad=True)
    w = torch.tensor(np.asarray(attention_weights, np.float64), requires_grad=True)
    out = _forward_torch(v, np.asarray(spatial_shapes), np.asarray(level_start_index), loc, w)
    out.backward(torch.as_tensor(np.asarray(grad_output, np.float64)))
    return v.grad.numpy(), loc.grad.numpy(), w.grad.numpy()
