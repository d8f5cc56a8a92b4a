"""O2a: brute-force tent-kernel formulation of the deformable sample (TEST INFRASTRUCTURE).

An independent statement of the bilinear, zero-padded sample used to pin the
C oracle: with the tent T(u) = max(0, 1 - |u|),

    sample(V, x, y) = sum over EVERY pixel (i, j) of V[i, j] * T(x - j) * T(y - i)

No floor, no corner enumeration and no range test appear here: pixels
outside the map simply do not exist in the sum, which is the zero padding of
grid_sample (Deformable DETR walk-through, "2.2.4 源码分析", the
``grid_sample(..., padding_mode='zeros', align_corners=False)`` call), and the
pixel coordinate is x = loc_x * W - 0.5 (``2*loc - 1`` mapped back with
align_corners=False).

The gradient with respect to x uses the right derivative of the tent,
T'(u) = +1 on [-1, 0), -1 on [0, 1), 0 elsewhere, matching the convention
that a sample on a pixel column belongs to the cell to its right.

Cost is O(points * H * W * D): tiny inputs only.
"""
from __future__ import annotations

import numpy as np


def _coords(loc: np.ndarray, size: int, fp32_contract: bool) -> np.ndarray:
    t = loc.astype(np.float64) * float(size) - 0.5      # exact in float64 for these inputs
    if fp32_contract:
        t = t.astype(np.float32).astype(np.float64)      # one rounding to binary32
    return t


def _tent(u: np.ndarray) -> np.ndarray:
    return np.maximum(0.0, 1.0 - np.abs(u))


def _tent_right_derivative(u: np.ndarray) -> np.ndarray:
    return np.where((u >= -1.0) & (u < 0.0), 1.0, np.where((u >= 0.0) & (u < 1.0), -1.0, 0.0))


def _level_views(value, spatial_shapes, level_start_index):
    bs, K, M, D = value.shape
    out = []
    for l, (H, W) in enumerate(np.asarray(spatial_shapes).tolist()):
        s = int(level_start_index[l])
        out.append((int(H), int(W), value[:, s:s + H * W].reshape(bs, H, W, M, D)))
    return out


def forward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
            fp32_contract: bool = False) -> np.ndarray:
    value = np.asarray(value, dtype=np.float64)
    loc = np.asarray(sampling_locations, dtype=np.float64)
    a = np.asarray(attention_weights, dtype=np.float64)
    bs, Q, M, L, P, _ = loc.shape
    D = value.shape[-1]
    out = np.zeros((bs, Q, M, D))
    for l, (H, W, V) in enumerate(_level_views(value, spatial_shapes, level_start_index)):
        x = _coords(loc[:, :, :, l, :, 0], W, fp32_contract)          # [bs,Q,M,P]
        y = _coords(loc[:, :, :, l, :, 1], H, fp32_contract)
        tx = _tent(x[..., None] - np.arange(W))                        # [bs,Q,M,P,W]
        ty = _tent(y[..., None] - np.arange(H))                        # [bs,Q,M,P,H]
        # sum_{i,j} V[b,i,j,m,:] * ty[...,i] * tx[...,j], weighted by a
        samp = np.einsum("bqmpi,bqmpj,bijmd->bqmpd", ty, tx, V)
        out += np.einsum("bqmp,bqmpd->bqmd", a[:, :, :, l], samp)
    return out.reshape(bs, Q, M * D)


def backward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
             grad_output, fp32_contract: bool = False):
    value = np.asarray(value, dtype=np.float64)
    loc = np.asarray(sampling_locations, dtype=np.float64)
    a = np.asarray(attention_weights, dtype=np.float64)
    bs, Q, M, L, P, _ = loc.shape
    D = value.shape[-1]
    g = np.asarray(grad_output, dtype=np.float64).reshape(bs, Q, M, D)
    gv = np.zeros_like(value)
    gl = np.zeros_like(loc)
    ga = np.zeros_like(a)
    for l, (H, W, V) in enumerate(_level_views(value, spatial_shapes, level_start_index)):
        s = int(level_start_index[l])
        x = _coords(loc[:, :, :, l, :, 0], W, fp32_contract)
        y = _coords(loc[:, :, :, l, :, 1], H, fp32_contract)
        ux = x[..., None] - np.arange(W)
        uy = y[..., None] - np.arange(H)
        tx, ty = _tent(ux), _tent(uy)
        dtx, dty = _tent_right_derivative(ux), _tent_right_derivative(uy)
        al = a[:, :, :, l]                                              # [bs,Q,M,P]
        samp = np.einsum("bqmpi,bqmpj,bijmd->bqmpd", ty, tx, V)
        ga[:, :, :, l] = np.einsum("bqmd,bqmpd->bqmp", g, samp)
        dsx = np.einsum("bqmpi,bqmpj,bijmd->bqmpd", ty, dtx, V)
        dsy = np.einsum("bqmpi,bqmpj,bijmd->bqmpd", dty, tx, V)
        gl[:, :, :, l, :, 0] = W * al * np.einsum("bqmd,bqmpd->bqmp", g, dsx)
        gl[:, :, :, l, :, 1] = H * al * np.einsum("bqmd,bqmpd->bqmp", g, dsy)
        contrib = np.einsum("bqmp,bqmpi,bqmpj,bqmd->bijmd", al, ty, tx, g)
        gv[:, s:s + H * W] += contrib.reshape(bs, H * W, M, D)
    return gv, gl, ga
