"""Oracle of the fused preparation + deformable attention (TEST INFRASTRUCTURE).

Only the tests and the benchmark's CPU legs use this module.  It composes the
steps of ``MSDeformAttn.forward`` in the Deformable DETR walk-through
("2.2.4 源码分析"), in the page's order, around the core oracle O1:

1. attention weights: softmax of the L*P logits of each (b, q, m), in fp64;
2. sampling locations from the reference points and the offsets:
   * 2-d references (one-stage): loc = ref[b,q,l,:] + off[b,q,m,l,p,:] / (W_l, H_l)
     (the walk-through's ``offset_normalizer = stack([W, H])``);
   * 4-d references (two-stage / box refinement, walk-through "2.4"):
     loc = ref[b,q,l,:2] + off[b,q,m,l,p,:] / P * ref[b,q,l,2:] * 0.5;
3. the core op (O1) on those locations and weights;
4. optional key padding mask: the walk-through's ``value.masked_fill(
   input_padding_mask[..., None], 0)`` -- every head's value row of a padded
   key (b, k) is zero before sampling, so those rows contribute nothing and,
   through the masked_fill, receive no gradient.

The locations decide which pixels are read, so the default mode takes the
module's expression in binary32 exactly as written, one correctly rounded
operation at a time, left to right, with IEEE division (the reading of "where
floating point decides an integer, both sides decide in the same precision"):
2-d: loc = fl(ref + fl(off / W)); 4-d: loc = fl(ref_xy + fl(fl(fl(off / P) *
ref_wh) * 0.5)).  ``exact=True`` forms them in fp64 instead (for finite
differences).  The backward is the chain rule through the same steps:

    grad_logits = a * (grad_a - sum_j a_j grad_a_j)          (softmax Jacobian)
    2-d: grad_off = grad_loc / (W, H);        grad_ref = sum_{m,p} grad_loc
    4-d: grad_off = grad_loc * ref_wh / (2P); grad_ref_xy = sum_{m,p} grad_loc,
         grad_ref_wh = sum_{m,p} grad_loc * off / (2P)
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

from . import backward as core_backward
from . import forward as core_forward


def softmax_weights(logits: np.ndarray, num_levels: int, num_points: int) -> np.ndarray:
    """[bs, Q, M, L*P] logits -> [bs, Q, M, L, P] fp64 softmax weights."""
    z = np.asarray(logits, np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    a = e / e.sum(axis=-1, keepdims=True)
    return a.reshape(*a.shape[:-1], num_levels, num_points)


def locations(reference_points: np.ndarray, sampling_offsets: np.ndarray,
              spatial_shapes: np.ndarray, exact: bool = False) -> np.ndarray:
    """Sampling locations [bs, Q, M, L, P, 2] (fp32 values, or fp64 when exact)."""
    ref = np.asarray(reference_points)
    off = np.asarray(sampling_offsets)
    L, P = off.shape[3], off.shape[4]
    ft = np.float64 if exact else np.float32
    ref = ref.astype(ft)[:, :, None, :, None, :]              # [bs, Q, 1, L, 1, 2|4]
    off = off.astype(ft)
    if ref.shape[-1] == 2:
        # offset_normalizer = stack([W, H]); each quotient rounded once
        norm = np.stack([np.asarray(spatial_shapes)[:, 1], np.asarray(spatial_shapes)[:, 0]], -1)
        return ref + off / norm.astype(ft)[None, None, None, :, None, :]
    if ref.shape[-1] == 4:
        # off / n_points * ref_wh * 0.5, evaluated left to right
        return ref[..., :2] + off / ft(P) * ref[..., 2:] * ft(0.5)
    raise ValueError("reference_points must end in 2 or 4")


def keep_rows(value: np.ndarray, padding_mask) -> np.ndarray:
    """[bs, K, 1, 1] factor: 0 for padded keys (mask true), 1 elsewhere."""
    bs, K = np.asarray(value).shape[:2]
    if padding_mask is None:
        return np.ones((bs, K, 1, 1))
    m = np.asarray(padding_mask).astype(bool)
    if m.shape != (bs, K):
        raise ValueError(f"padding_mask must be [bs, num_keys] = {(bs, K)}, got {m.shape}")
    return (~m).astype(np.float64)[:, :, None, None]


def masked_fill_grad(grad_value: np.ndarray, keep: np.ndarray) -> np.ndarray:
    """Gradient through masked_fill: padded rows receive none."""
    return grad_value * keep


def forward(value, spatial_shapes, level_start_index, reference_points, sampling_offsets,
            attention_logits, exact: bool = False, threads: int = 0,
            padding_mask=None) -> np.ndarray:
    """Output [bs, Q, M*D] in fp64."""
    off = np.asarray(sampling_offsets)
    L, P = off.shape[3], off.shape[4]
    a = softmax_weights(attention_logits, L, P)
    loc = locations(reference_points, sampling_offsets, spatial_shapes, exact)
    v = np.asarray(value, np.float64) * keep_rows(value, padding_mask)
    return core_forward(v, spatial_shapes, level_start_index, loc, a, exact_coords=exact,
                        threads=threads)


def backward(value, spatial_shapes, level_start_index, reference_points, sampling_offsets,
             attention_logits, grad_output, exact: bool = False, threads: int = 0,
             padding_mask=None) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """(grad_value, grad_sampling_offsets, grad_attention_logits, grad_reference_points), fp64.
    grad_value is the gradient with respect to the value before the padding mask."""
    ref = np.asarray(reference_points, np.float64)
    off = np.asarray(sampling_offsets, np.float64)
    bs, Q, M, L, P, _ = off.shape
    a = softmax_weights(attention_logits, L, P)
    loc = locations(reference_points, sampling_offsets, spatial_shapes, exact)
    keep = keep_rows(value, padding_mask)
    gv, gl, ga = core_backward(np.asarray(value, np.float64) * keep, spatial_shapes,
                               level_start_index, loc, a, grad_output, exact_coords=exact,
                               threads=threads)
    gv = masked_fill_grad(gv, keep)
    ga = ga.reshape(bs, Q, M, L * P)
    af = a.reshape(bs, Q, M, L * P)
    g_logits = af * (ga - (af * ga).sum(axis=-1, keepdims=True))
    if ref.shape[-1] == 2:
        shapes = np.asarray(spatial_shapes, np.float64)
        norm = np.stack([shapes[:, 1], shapes[:, 0]], -1)[None, None, None, :, None, :]
        g_off = gl / norm
        g_ref = gl.sum(axis=(2, 4))                                  # over heads and points
    else:
        wh = ref[:, :, None, :, None, 2:]
        g_off = gl * wh / (2.0 * P)
        g_ref = np.concatenate([gl.sum(axis=(2, 4)),
                                (gl * off / (2.0 * P)).sum(axis=(2, 4))], axis=-1)
    return gv, g_off, g_logits, g_ref
