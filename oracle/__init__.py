"""fp64 CPU oracle for multi-scale deformable attention (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports it, and it imports nothing from the product.

Contents:
  * ``forward`` / ``backward``  -- O1, the plain C oracle (msda_oracle.c),
    loaded with ctypes; fp64 arithmetic, OpenMP over queries (forward) or
    over (batch, head) slices (backward, deterministic).
  * ``tent``                     -- O2a, brute-force tent-kernel sums over
    every pixel (independent formulation, tiny inputs only).
  * ``grid_sample_ref``          -- O2b, per-level torch ``grid_sample`` in
    fp64 on the CPU (the pages' own formulation restated) with autograd.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Tuple

import numpy as np

from . import build as _build

__all__ = ["forward", "backward", "touched_rows", "max_threads", "load"]

_LIB = None
_dbl_p = ctypes.POINTER(ctypes.c_double)
_i64_p = ctypes.POINTER(ctypes.c_int64)


def load(path: Optional[str] = None):
    """Compile (if stale) and load liboracle.so, or load the library at ``path``."""
    global _LIB
    if path is not None or _LIB is None:
        lib = ctypes.CDLL(path if path is not None else _build.build())
        dims = [ctypes.c_int] * 7
        lib.oracle_forward.argtypes = [_dbl_p, _i64_p, _i64_p, _dbl_p, _dbl_p, _dbl_p] + dims + [
            ctypes.c_int, ctypes.c_int]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_backward.argtypes = [_dbl_p, _i64_p, _i64_p, _dbl_p, _dbl_p, _dbl_p, _dbl_p,
                                        _dbl_p, _dbl_p] + dims + [ctypes.c_int, ctypes.c_int]
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_touched_rows.argtypes = [_i64_p, _i64_p, _dbl_p, _dbl_p, ctypes.c_void_p] + [
            ctypes.c_int] * 7
        lib.oracle_touched_rows.restype = ctypes.c_int64
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        if path is not None:
            return lib
        _LIB = lib
    return _LIB


def max_threads() -> int:
    return int(load().oracle_max_threads())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int64)


def _dims(value: np.ndarray, loc: np.ndarray) -> Tuple[int, ...]:
    bs, K, M, D = value.shape
    bs2, Q, M2, L, P, two = loc.shape
    if bs2 != bs or M2 != M or two != 2:
        raise ValueError("value / sampling_locations shapes disagree")
    return bs, K, M, D, L, P, Q


def forward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
            exact_coords: bool = False, threads: int = 0, lib=None) -> np.ndarray:
    """Output [bs, Q, M*D] in float64.

    ``exact_coords=False`` applies the fp32 coordinate contract (one rounding
    of loc*W - 0.5); the location inputs must then be float32-representable.
    """
    lib = lib or load()
    value, loc, w = _f64(value), _f64(sampling_locations), _f64(attention_weights)
    shapes, lsi = _i64(spatial_shapes), _i64(level_start_index)
    bs, K, M, D, L, P, Q = _dims(value, loc)
    out = np.empty((bs, Q, M * D), dtype=np.float64)
    rc = lib.oracle_forward(value.ctypes.data_as(_dbl_p), shapes.ctypes.data_as(_i64_p),
                            lsi.ctypes.data_as(_i64_p), loc.ctypes.data_as(_dbl_p),
                            w.ctypes.data_as(_dbl_p), out.ctypes.data_as(_dbl_p),
                            bs, K, M, D, L, P, Q, 1 if exact_coords else 0, int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_forward failed ({rc})")
    return out


def backward(value, spatial_shapes, level_start_index, sampling_locations, attention_weights,
             grad_output, exact_coords: bool = False, threads: int = 0, lib=None
             ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(grad_value, grad_sampling_loc, grad_attention_weights), float64."""
    lib = lib or load()
    value, loc, w = _f64(value), _f64(sampling_locations), _f64(attention_weights)
    g = _f64(grad_output)
    shapes, lsi = _i64(spatial_shapes), _i64(level_start_index)
    bs, K, M, D, L, P, Q = _dims(value, loc)
    if g.shape != (bs, Q, M * D):
        raise ValueError("grad_output shape")
    gv = np.empty_like(value)
    gl = np.empty_like(loc)
    gw = np.empty_like(w)
    rc = lib.oracle_backward(value.ctypes.data_as(_dbl_p), shapes.ctypes.data_as(_i64_p),
                             lsi.ctypes.data_as(_i64_p), loc.ctypes.data_as(_dbl_p),
                             w.ctypes.data_as(_dbl_p), g.ctypes.data_as(_dbl_p),
                             gv.ctypes.data_as(_dbl_p), gl.ctypes.data_as(_dbl_p),
                             gw.ctypes.data_as(_dbl_p), bs, K, M, D, L, P, Q,
                             1 if exact_coords else 0, int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_backward failed ({rc})")
    return gv, gl, gw


def touched_rows(spatial_shapes, level_start_index, sampling_locations, attention_weights,
                 bs: int, num_keys: int, num_heads: int, lib=None) -> int:
    """Distinct (b, key, m) value rows read with a non-zero weight by one forward
    (fp32 coordinate contract)."""
    lib = lib if lib is not None else load()
    loc, w = _f64(sampling_locations), _f64(attention_weights)
    shapes, lsi = _i64(spatial_shapes), _i64(level_start_index)
    _, Q, M, L, P, _ = loc.shape
    mark = np.empty(bs * num_keys * num_heads, dtype=np.uint8)
    return int(lib.oracle_touched_rows(shapes.ctypes.data_as(_i64_p), lsi.ctypes.data_as(_i64_p),
                                       loc.ctypes.data_as(_dbl_p), w.ctypes.data_as(_dbl_p),
                                       mark.ctypes.data, bs, num_keys, num_heads, L, P, Q, 0))


def run_inputs(inputs: Dict[str, np.ndarray], backward_pass: bool = True, threads: int = 0):
    """Oracle on a dict produced by the seeded input generator."""
    args = (inputs["value"], inputs["spatial_shapes"], inputs["level_start_index"],
            inputs["sampling_locations"], inputs["attention_weights"])
    out = forward(*args, threads=threads)
    if not backward_pass:
        return out, None
    return out, backward(*args, inputs["grad_output"], threads=threads)
