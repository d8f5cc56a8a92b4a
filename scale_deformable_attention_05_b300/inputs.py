"""Seeded synthetic inputs for multi-scale deformable attention (MSDeformAttn).

This module is shared by the tests, the benchmark and the oracle checks. It
holds none of the operator's arithmetic: only random draws, the flattened
multi-level layout that the operator's inputs are defined in, and the rounding
of fp32 draws to bf16.  Everything here is numpy on the host.

Layouts (C-contiguous, innermost last), as the Ascend DrivingSDK page
"multi_scale_deformable_attn" (parameter list) and the Deformable DETR
walk-through ("2.2.4 源码分析", ``ms_deform_attn_core_pytorch``) define them:

* value               [bs, num_keys, num_heads, head_dim]
* spatial_shapes      [num_levels, 2] int64, rows (H, W)
* level_start_index   [num_levels] int64, exclusive prefix sum of H*W
* sampling_locations  [bs, num_queries, num_heads, num_levels, num_points, 2],
                      last axis (x, y), x normalised by W and y by H
* attention_weights   [bs, num_queries, num_heads, num_levels, num_points]
* output / grad_output[bs, num_queries, num_heads * head_dim]

The five named workloads stand in for Deformable DETR on COCO-sized images
(about 800x1333 at strides 8/16/32/64); no dataset is read.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Dict, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "workload",
    "level_start_index",
    "num_keys",
    "encoder_reference_points",
    "grid_reference_points",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "f32_to_f16_bits",
    "f16_bits_to_f32",
    "make_inputs",
    "padding_mask",
    "make_fused_inputs",
    "random_workload",
]

# Deformable DETR feature pyramid for an ~800x1333 image at strides 8/16/32/64
# (walk-through "2.1.1 backbone生成多尺度特征").
DETR_PYRAMID: Tuple[Tuple[int, int], ...] = ((100, 167), (50, 84), (25, 42), (13, 21))
# Largest pyramid inside the Ascend operator envelope used for the head_dim=256 case.
ENVELOPE_PYRAMID: Tuple[Tuple[int, int], ...] = ((200, 200), (100, 100), (50, 50), (25, 25))


@dataclass(frozen=True)
class Workload:
    """One seeded synthetic problem.

    ``loc_kind`` selects how sampling locations are drawn:
      * ``"uniform"``  : every coordinate i.i.d. U[lo, hi] (``loc_range``)
      * ``"encoder"``  : pixel-centre reference point of the query's own level
                         + N(0, sigma) per (head, level, point, coord), clamped
      * ``"decoder"``  : U[0,1]^2 reference point per (b, q) + N(0, sigma)
      * ``"grid"``     : row-major sqrt(Q) x sqrt(Q) grid of cell centres + N(0, sigma)
    ``weight_kind``: ``"uniform"`` (U[0,1) + 1e-5) or ``"softmax"`` (softmax of
    N(0,1) logits over num_levels*num_points per (b, q, head)).
    ``value_kind``: ``"uniform_small"`` (U[0,1) * 0.01) or ``"normal"`` (N(0,1)).
    ``grad_kind``: ``"ones"`` or ``"normal"``.
    """

    name: str
    seed: int
    bs: int
    spatial_shapes: Tuple[Tuple[int, int], ...]
    num_heads: int
    head_dim: int
    num_points: int
    num_queries: int
    dtype: str = "f32"
    loc_kind: str = "uniform"
    loc_sigma: float = 0.0
    loc_clamp: Optional[Tuple[float, float]] = None
    loc_range: Tuple[float, float] = (-0.1, 1.1)
    weight_kind: str = "softmax"
    value_kind: str = "normal"
    grad_kind: str = "normal"
    description: str = ""

    @property
    def num_levels(self) -> int:
        return len(self.spatial_shapes)

    @property
    def num_keys(self) -> int:
        return num_keys(self.spatial_shapes)

    @property
    def points(self) -> int:
        """Sampled points per call: bs * Q * heads * levels * points."""
        return self.bs * self.num_queries * self.num_heads * self.num_levels * self.num_points

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype in ("bf16", "f16") else 4

    def compulsory_bytes(self, backward: bool) -> int:
        """Bytes every implementation must move to or from HBM at least once.

        forward : value + sampling_locations + attention_weights + output
        backward: value + locations + weights + grad_output
                  + grad_value + grad_sampling_loc + grad_attn_weight
        all at the I/O dtype.
        """
        e = self.elem_bytes
        value = self.bs * self.num_keys * self.num_heads * self.head_dim * e
        loc = self.points * 2 * e
        w = self.points * e
        out = self.bs * self.num_queries * self.num_heads * self.head_dim * e
        if not backward:
            return value + loc + w + out
        return value + loc + w + out + value + loc + w

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def num_keys(spatial_shapes: Sequence[Sequence[int]]) -> int:
    return int(sum(int(h) * int(w) for h, w in spatial_shapes))


def level_start_index(spatial_shapes: Sequence[Sequence[int]]) -> np.ndarray:
    """Start of each level in the flattened key axis: [0, cumsum(H*W)[:-1]].

    Deformable DETR walk-through, "2.3.1 DeformableTransformer" (the
    ``level_start_index`` line) and the Ascend page's call example.
    """
    sizes = np.array([int(h) * int(w) for h, w in spatial_shapes], dtype=np.int64)
    out = np.zeros(len(sizes), dtype=np.int64)
    if len(sizes) > 1:
        out[1:] = np.cumsum(sizes)[:-1]
    return out


def encoder_reference_points(spatial_shapes: Sequence[Sequence[int]]) -> np.ndarray:
    """Normalised pixel centres of every flattened position, levels concatenated.

    Row-major per level: position (i, j) of level l gets
    ((j + 0.5) / W_l, (i + 0.5) / H_l) (walk-through "2.2.4 源码分析", first
    step, ``get_reference_points`` with all valid ratios 1).  Returns
    float64 [num_keys, 2] as (x, y).
    """
    refs = []
    for h, w in spatial_shapes:
        ys = (np.arange(h, dtype=np.float64) + 0.5) / h
        xs = (np.arange(w, dtype=np.float64) + 0.5) / w
        yy, xx = np.meshgrid(ys, xs, indexing="ij")
        refs.append(np.stack([xx.reshape(-1), yy.reshape(-1)], axis=-1))
    return np.concatenate(refs, axis=0)


def grid_reference_points(n: int) -> np.ndarray:
    """Row-major n x n grid of cell centres in [0,1]^2 as (x, y), float64 [n*n, 2]."""
    c = (np.arange(n, dtype=np.float64) + 0.5) / n
    yy, xx = np.meshgrid(c, c, indexing="ij")
    return np.stack([xx.reshape(-1), yy.reshape(-1)], axis=-1)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); returns uint16 bits.

    Inputs here are finite draws; NaN payloads are not handled.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits to float32 exactly."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to IEEE half (numpy's cast: round to nearest, ties to even); uint16 bits."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen IEEE half bits to float32 exactly."""
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def _softmax_lastdim(x: np.ndarray) -> np.ndarray:
    z = x - x.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def make_inputs(wl: Workload, with_grad: bool = True) -> Dict[str, np.ndarray]:
    """Draw one seeded problem.

    Draw order is fixed: value, reference points, offsets (or locations),
    weights (or logits), grad_output.  Every draw is float64 in C order and
    is then cast to float32 (round to nearest even); for ``dtype == "bf16"`` the
    float32 arrays are further rounded to bf16.

    Returned keys: ``value``, ``sampling_locations``, ``attention_weights``,
    ``grad_output`` (float32 arrays holding exactly the values the operator
    sees, i.e. bf16-representable for bf16 workloads), ``spatial_shapes``,
    ``level_start_index`` (int64), and for bf16 / f16 workloads the uint16 bit
    patterns under ``*_bf16`` / ``*_f16`` keys.
    """
    rng = np.random.default_rng(wl.seed)
    bs, Q, M, D = wl.bs, wl.num_queries, wl.num_heads, wl.head_dim
    L, P = wl.num_levels, wl.num_points
    K = wl.num_keys
    shapes = np.array(wl.spatial_shapes, dtype=np.int64).reshape(L, 2)

    # 1. value
    if wl.value_kind == "uniform_small":
        value = rng.random((bs, K, M, D)) * 0.01
    elif wl.value_kind == "normal":
        value = rng.standard_normal((bs, K, M, D))
    else:
        raise ValueError(wl.value_kind)
    value = value.astype(np.float32)

    # 2./3. reference points and offsets, or locations directly
    loc_shape = (bs, Q, M, L, P, 2)
    if wl.loc_kind == "uniform":
        lo, hi = wl.loc_range
        loc = rng.uniform(lo, hi, size=loc_shape)
    else:
        if wl.loc_kind == "encoder":
            ref = encoder_reference_points(wl.spatial_shapes)
            if ref.shape[0] != Q:
                raise ValueError("encoder workload needs num_queries == num_keys")
            ref = np.broadcast_to(ref[None], (bs, Q, 2))
        elif wl.loc_kind == "decoder":
            ref = rng.random((bs, Q, 2))
        elif wl.loc_kind == "grid":
            n = int(round(np.sqrt(Q)))
            if n * n != Q:
                raise ValueError("grid workload needs a square num_queries")
            ref = np.broadcast_to(grid_reference_points(n)[None], (bs, Q, 2))
        else:
            raise ValueError(wl.loc_kind)
        off = rng.normal(0.0, wl.loc_sigma, size=loc_shape)
        loc = ref[:, :, None, None, None, :] + off
        if wl.loc_clamp is not None:
            loc = np.clip(loc, wl.loc_clamp[0], wl.loc_clamp[1])
    loc = loc.astype(np.float32)

    # 4. attention weights
    if wl.weight_kind == "uniform":
        w = rng.random((bs, Q, M, L, P)) + 1e-5
    elif wl.weight_kind == "softmax":
        logits = rng.standard_normal((bs, Q, M, L * P))
        w = _softmax_lastdim(logits).reshape(bs, Q, M, L, P)
    else:
        raise ValueError(wl.weight_kind)
    w = w.astype(np.float32)

    # 5. grad_output
    g = None
    if with_grad:
        if wl.grad_kind == "ones":
            g = np.ones((bs, Q, M * D), dtype=np.float32)
        elif wl.grad_kind == "normal":
            g = rng.standard_normal((bs, Q, M * D)).astype(np.float32)
        else:
            raise ValueError(wl.grad_kind)

    out: Dict[str, np.ndarray] = {
        "spatial_shapes": shapes,
        "level_start_index": level_start_index(wl.spatial_shapes),
    }
    arrays = {"value": value, "sampling_locations": loc, "attention_weights": w}
    if g is not None:
        arrays["grad_output"] = g
    for k, a in arrays.items():
        if wl.dtype == "bf16":
            bits = f32_to_bf16_bits(a)
            out[k + "_bf16"] = bits
            out[k] = bf16_bits_to_f32(bits).reshape(a.shape)
        elif wl.dtype == "f16":
            bits = f32_to_f16_bits(a)
            out[k + "_f16"] = bits
            out[k] = f16_bits_to_f32(bits).reshape(a.shape)
        elif wl.dtype == "f32":
            out[k] = np.ascontiguousarray(a)
        else:
            raise ValueError(wl.dtype)
    return out


def make_fused_inputs(wl: Workload, ref_dim: int = 2, offset_sigma: float = 2.0
                      ) -> Dict[str, np.ndarray]:
    """Seeded inputs of the fused entry points for workload ``wl``.

    Draw order: value, reference points (and box sizes for ``ref_dim == 4``),
    offsets, logits, grad_output.  Reference points follow ``wl.loc_kind``:
    ``encoder`` uses each query's pixel centre (all levels, valid ratios 1),
    ``grid`` the row-major grid of cell centres, anything else U[0.1, 0.9]^2
    per (b, q); the same point serves every level.  Box sizes are U[0.05, 0.4]
    per (b, q).  Offsets are N(0, offset_sigma) and logits N(0, 1).  Rounded to
    ``wl.dtype`` like ``make_inputs``; returned under ``reference_points``,
    ``sampling_offsets``, ``attention_logits`` (plus ``*_bf16`` / ``*_f16`` bits).
    """
    rng = np.random.default_rng(wl.seed + 50000 * ref_dim)
    bs, Q, M, D = wl.bs, wl.num_queries, wl.num_heads, wl.head_dim
    L, P, K = wl.num_levels, wl.num_points, wl.num_keys
    value = rng.standard_normal((bs, K, M, D))
    if wl.loc_kind == "encoder":
        ref = np.broadcast_to(encoder_reference_points(wl.spatial_shapes)[None], (bs, Q, 2))
    elif wl.loc_kind == "grid":
        n = int(round(np.sqrt(Q)))
        ref = np.broadcast_to(grid_reference_points(n)[None], (bs, Q, 2))
    else:
        ref = rng.uniform(0.1, 0.9, (bs, Q, 2))
    ref = np.broadcast_to(ref[:, :, None, :], (bs, Q, L, 2))
    if ref_dim == 4:
        wh = rng.uniform(0.05, 0.4, (bs, Q, 1, 2))
        ref = np.concatenate([ref, np.broadcast_to(wh, (bs, Q, L, 2))], -1)
    off = rng.normal(0.0, offset_sigma, (bs, Q, M, L, P, 2))
    logits = rng.standard_normal((bs, Q, M, L * P))
    g = rng.standard_normal((bs, Q, M * D))
    out: Dict[str, np.ndarray] = {
        "spatial_shapes": np.array(wl.spatial_shapes, dtype=np.int64).reshape(L, 2),
        "level_start_index": level_start_index(wl.spatial_shapes),
    }
    arrays = {"value": value, "reference_points": ref, "sampling_offsets": off,
              "attention_logits": logits, "grad_output": g}
    for k, a in arrays.items():
        a = np.ascontiguousarray(a, dtype=np.float32)
        if wl.dtype == "bf16":
            bits = f32_to_bf16_bits(a)
            out[k + "_bf16"] = bits
            out[k] = bf16_bits_to_f32(bits).reshape(a.shape)
        elif wl.dtype == "f16":
            bits = f32_to_f16_bits(a)
            out[k + "_f16"] = bits
            out[k] = f16_bits_to_f32(bits).reshape(a.shape)
        else:
            out[k] = a
    return out


def padding_mask(wl: Workload, min_ratio: float = 0.6) -> np.ndarray:
    """Seeded key padding mask [bs, num_keys] (bool, True = padded) shaped like
    the masks of a padded image batch: image b keeps the top-left
    ceil(rh_b * H_l) x ceil(rw_b * W_l) pixels of every level, with (rh_b, rw_b)
    ~ U[min_ratio, 1]^2 and image 0 unpadded (the batch is padded to it).  Drawn
    from its own stream (seed + 70000), so the other inputs do not change."""
    rng = np.random.default_rng(wl.seed + 70000)
    ratios = rng.uniform(min_ratio, 1.0, (wl.bs, 2))
    ratios[0] = 1.0
    mask = np.zeros((wl.bs, wl.num_keys), dtype=bool)
    start = 0
    for H, W in wl.spatial_shapes:
        for b in range(wl.bs):
            vh = int(np.ceil(ratios[b, 0] * H))
            vw = int(np.ceil(ratios[b, 1] * W))
            m = np.zeros((H, W), dtype=bool)
            m[vh:, :] = True
            m[:, vw:] = True
            mask[b, start:start + H * W] = m.reshape(-1)
        start += H * W
    return mask


def random_workload(seed: int, bs: int, spatial_shapes, num_heads: int, head_dim: int,
                    num_points: int, num_queries: int, dtype: str = "f32",
                    loc_range=(-0.2, 1.2)) -> Workload:
    """A small uniform-location problem for randomized shape sweeps."""
    return Workload(
        name=f"random-{seed}", seed=seed, bs=bs,
        spatial_shapes=tuple((int(h), int(w)) for h, w in spatial_shapes),
        num_heads=num_heads, head_dim=head_dim, num_points=num_points,
        num_queries=num_queries, dtype=dtype, loc_kind="uniform", loc_range=tuple(loc_range),
        weight_kind="softmax", value_kind="normal", grad_kind="normal",
    )


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload(
        name="tiny", seed=1001, bs=1, spatial_shapes=((100, 100),), num_heads=4, head_dim=32,
        num_points=8, num_queries=16, dtype="f32", loc_kind="uniform", loc_range=(-0.1, 1.1),
        weight_kind="uniform", value_kind="uniform_small", grad_kind="ones",
        description="Ascend call-example shape: bs=1, one 100x100 level, 4 heads, head_dim 32, "
                    "8 points, 16 queries; fp32 forward+backward",
    ),
    "encoder": Workload(
        name="encoder", seed=1002, bs=2, spatial_shapes=DETR_PYRAMID, num_heads=8, head_dim=32,
        num_points=4, num_queries=22223, dtype="f32", loc_kind="encoder", loc_sigma=0.02,
        loc_clamp=(-0.05, 1.05), weight_kind="softmax", value_kind="normal", grad_kind="normal",
        description="Deformable DETR encoder self-attention: bs=2, 4-level 100x167 pyramid "
                    "(22223 keys = queries), 8 heads, head_dim 32, 4 points; fp32",
    ),
    "decoder": Workload(
        name="decoder", seed=1003, bs=2, spatial_shapes=DETR_PYRAMID, num_heads=8, head_dim=32,
        num_points=4, num_queries=300, dtype="f32", loc_kind="decoder", loc_sigma=0.05,
        weight_kind="softmax", value_kind="normal", grad_kind="normal",
        description="Deformable DETR decoder cross-attention: bs=2, 300 object queries over the "
                    "encoder pyramid; fp32 forward+backward",
    ),
    "encoder_bf16": Workload(
        name="encoder_bf16", seed=1004, bs=4, spatial_shapes=DETR_PYRAMID, num_heads=8,
        head_dim=32, num_points=4, num_queries=22223, dtype="bf16", loc_kind="encoder",
        loc_sigma=0.02, loc_clamp=(-0.05, 1.05), weight_kind="softmax", value_kind="normal",
        grad_kind="normal",
        description="encoder shape with bs=4, bf16 I/O, fp32 accumulation; forward+backward",
    ),
    "encoder_f16": Workload(
        name="encoder_f16", seed=1006, bs=4, spatial_shapes=DETR_PYRAMID, num_heads=8,
        head_dim=32, num_points=4, num_queries=22223, dtype="f16", loc_kind="encoder",
        loc_sigma=0.02, loc_clamp=(-0.05, 1.05), weight_kind="softmax", value_kind="normal",
        grad_kind="normal",
        description="encoder shape with bs=4, fp16 I/O, fp32 accumulation; forward+backward",
    ),
    "envelope": Workload(
        name="envelope", seed=1005, bs=1, spatial_shapes=ENVELOPE_PYRAMID, num_heads=8,
        head_dim=256, num_points=16, num_queries=10000, dtype="f32", loc_kind="grid",
        loc_sigma=0.03, weight_kind="softmax", value_kind="normal", grad_kind="normal",
        description="operator-envelope limit: bs=1, 200x200 4-level pyramid, 8 heads, head_dim "
                    "256, 16 points (levels*points = 64), 10000 queries; fp32",
    ),
}

# Workloads by their position in the problem list (1-based), for the command line.
WORKLOAD_ORDER = ("tiny", "encoder", "decoder", "encoder_bf16", "envelope")


def workload(name_or_index) -> Workload:
    if isinstance(name_or_index, int) or (isinstance(name_or_index, str) and name_or_index.isdigit()):
        return WORKLOADS[WORKLOAD_ORDER[int(name_or_index) - 1]]
    return WORKLOADS[name_or_index]
