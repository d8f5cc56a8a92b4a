"""Thin Python binding of the C ABI in ``include/msda.h`` (``libmsda.so``).

Argument marshalling only: every step of the operator runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (torch is used for device
memory and streams); their data pointers, the dims and the current CUDA
stream are handed to the C functions of the same names.  There is no CPU
path: if the library is missing this module raises on import, and tensors
that are not on a CUDA device are rejected.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

import torch

__all__ = [
    "MSDA_F32", "MSDA_BF16", "MSDA_F16", "MSDA_INDEX_INT32", "MSDA_GRAD_VALUE_ACCUMULATE",
    "MsdaError", "LIB_PATH",
    "msda_forward", "msda_backward", "msda_backward_workspace_bytes", "msda_zero_fill",
    "msda_check_shapes", "msda_last_device_error", "msda_status_string", "msda_version",
    "msda_backward_noalloc", "msda_forward_fused", "msda_backward_fused", "msda_linear",
    "msda_linear_f32", "msda_linear_workspace_bytes", "msda_linear_wgrad_f32",
    "msda_linear_bias_grad", "MSDeformAttnFunction", "MSDeformAttnFusedFunction", "ms_deform_attn", "ms_deform_attn_fused",
    "EXPORTED_SYMBOLS", "load_library",
]

MSDA_F32 = 0
MSDA_BF16 = 1
MSDA_F16 = 2
MSDA_INDEX_INT32 = 0x100
MSDA_GRAD_VALUE_ACCUMULATE = 1
MSDA_MAX_FUSED_LEVEL_POINTS = 64
MSDA_LINEAR_MAX_FEATURES = 256
MSDA_LINEAR_BIAS_HALF = 0x200
MSDA_LINEAR_BIAS_BF16 = MSDA_LINEAR_BIAS_HALF

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmsda.so")
EXPORTED_SYMBOLS = (
    "msda_forward", "msda_backward", "msda_backward_workspace_bytes", "msda_zero_fill",
    "msda_check_shapes", "msda_last_device_error", "msda_status_string", "msda_version",
    "msda_backward_noalloc", "msda_forward_fused", "msda_backward_fused", "msda_linear",
    "msda_linear_f32", "msda_linear_workspace_bytes", "msda_linear_wgrad_f32",
    "msda_linear_bias_grad",
)

_vp = ctypes.c_void_p
_int = ctypes.c_int
_DIMS = [_int] * 7


class MsdaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {msda_status_string(status)} (status {status})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m scale_deformable_attention_05_b300.build`"
            " (nvcc, sm_103a); there is no fallback implementation")
    lib = ctypes.CDLL(path)
    lib.msda_forward.argtypes = [_vp] * 6 + _DIMS + [_int, _vp]
    lib.msda_forward.restype = _int
    lib.msda_backward_workspace_bytes.argtypes = [_int] * 5
    lib.msda_backward_workspace_bytes.restype = ctypes.c_size_t
    lib.msda_backward.argtypes = [_vp] * 10 + [ctypes.c_size_t] + _DIMS + [_int, ctypes.c_uint, _vp]
    lib.msda_backward.restype = _int
    lib.msda_zero_fill.argtypes = [_vp, ctypes.c_size_t, _vp]
    lib.msda_zero_fill.restype = _int
    lib.msda_check_shapes.argtypes = [_vp, _vp, _int, _int, _vp]
    lib.msda_check_shapes.restype = _int
    lib.msda_last_device_error.argtypes = [_vp]
    lib.msda_last_device_error.restype = _int
    lib.msda_status_string.argtypes = [_int]
    lib.msda_status_string.restype = ctypes.c_char_p
    lib.msda_version.argtypes = []
    lib.msda_version.restype = _int
    lib.msda_backward_noalloc.argtypes = [_vp] * 9 + _DIMS + [_int, ctypes.c_uint, _vp]
    lib.msda_backward_noalloc.restype = _int
    lib.msda_linear.argtypes = [_vp] * 4 + [_int] * 4 + [_vp]
    lib.msda_linear.restype = _int
    lib.msda_linear_workspace_bytes.argtypes = [_int] * 4
    lib.msda_linear_workspace_bytes.restype = ctypes.c_size_t
    lib.msda_linear_f32.argtypes = [_vp] * 5 + [ctypes.c_size_t] + [_int] * 3 + [_vp]
    lib.msda_linear_f32.restype = _int
    lib.msda_linear_wgrad_f32.argtypes = [_vp] * 4 + [_int] * 3 + [ctypes.c_uint, _vp]
    lib.msda_linear_wgrad_f32.restype = _int
    lib.msda_linear_bias_grad.argtypes = [_vp, _vp, _int, _int, _int, ctypes.c_uint, _vp]
    lib.msda_linear_bias_grad.restype = _int
    lib.msda_forward_fused.argtypes = [_vp] * 8 + _DIMS + [_int, _int, _vp]
    lib.msda_forward_fused.restype = _int
    lib.msda_backward_fused.argtypes = ([_vp] * 13 + [ctypes.c_size_t] + _DIMS +
                                        [_int, _int, ctypes.c_uint, _vp])
    lib.msda_backward_fused.restype = _int
    return lib


_LIB = load_library()


def msda_status_string(status: int) -> str:
    return _LIB.msda_status_string(int(status)).decode()


def msda_version() -> int:
    return int(_LIB.msda_version())


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MsdaError(fn, status)


def _dtype_code(t: torch.Tensor, index: Optional[torch.Tensor] = None) -> int:
    """ABI dtype code of value tensor t, with MSDA_INDEX_INT32 when the index
    tensors are int32."""
    if t.dtype == torch.float32:
        code = MSDA_F32
    elif t.dtype == torch.bfloat16:
        code = MSDA_BF16
    elif t.dtype == torch.float16:
        code = MSDA_F16
    else:
        raise TypeError(f"unsupported dtype {t.dtype} (float32, bfloat16 or float16)")
    if index is not None and index.dtype == torch.int32:
        code |= MSDA_INDEX_INT32
    return code


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if t.device.type != "cuda":
        raise ValueError("tensors must be on a CUDA device (no CPU path)")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr() if t.numel() > 0 else None


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _dims(value: torch.Tensor, spatial_shapes: torch.Tensor, sampling_loc: torch.Tensor
          ) -> Tuple[int, ...]:
    if value.dim() != 4 or sampling_loc.dim() != 6:
        raise ValueError("value must be [bs,K,M,D] and sampling_loc [bs,Q,M,L,P,2]")
    bs, K, M, D = value.shape
    bs2, Q, M2, L, P, two = sampling_loc.shape
    if bs2 != bs or M2 != M or two != 2 or spatial_shapes.shape != (L, 2):
        raise ValueError("inconsistent shapes between value, sampling_loc and spatial_shapes")
    return int(bs), int(K), int(M), int(D), int(L), int(P), int(Q)


def _expect(t: Optional[torch.Tensor], shape, like: torch.Tensor, name: str) -> None:
    """t (if given) has this shape and like's dtype and device: the kernels read
    every float tensor as the value's element type, so a mismatch is refused
    here instead of being read with the wrong width."""
    if t is None:
        return
    if tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != like.dtype:
        raise TypeError(f"{name} must have the value's dtype {like.dtype}, got {t.dtype}")
    if t.device != like.device:
        raise ValueError(f"{name} is on {t.device}, value on {like.device}")


def _index(t: torch.Tensor, like: Optional[torch.Tensor] = None) -> torch.Tensor:
    if t.dtype not in (torch.int64, torch.int32):
        raise TypeError("spatial_shapes and level_start_index must be int64 or int32")
    if like is not None and t.dtype != like.dtype:
        raise TypeError("spatial_shapes and level_start_index must have the same dtype")
    return t


def msda_forward(value: torch.Tensor, spatial_shapes: torch.Tensor,
                 level_start_index: torch.Tensor, sampling_loc: torch.Tensor,
                 attn_weight: torch.Tensor, output: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """output [bs, Q, M*D] = MSDeformAttn forward (see include/msda.h)."""
    bs, K, M, D, L, P, Q = _dims(value, spatial_shapes, sampling_loc)
    code = _dtype_code(value, spatial_shapes)
    _expect(sampling_loc, (bs, Q, M, L, P, 2), value, "sampling_loc")
    _expect(attn_weight, (bs, Q, M, L, P), value, "attn_weight")
    _expect(output, (bs, Q, M * D), value, "output")
    if output is None:
        output = torch.empty((bs, Q, M * D), dtype=value.dtype, device=value.device)
    _check("msda_forward", _LIB.msda_forward(
        _ptr(value), _ptr(_index(spatial_shapes)), _ptr(_index(level_start_index, spatial_shapes)),
        _ptr(sampling_loc), _ptr(attn_weight), _ptr(output), bs, K, M, D, L, P, Q, code,
        _stream(stream)))
    return output


def msda_backward_workspace_bytes(bs: int, num_keys: int, num_heads: int, head_dim: int,
                                  dtype: int) -> int:
    return int(_LIB.msda_backward_workspace_bytes(bs, num_keys, num_heads, head_dim, dtype))


def _check_grads(value, loc, attn, grad_output, grad_value, grad_loc, grad_attn, attn_shape,
                 out_shape):
    _expect(loc, tuple(attn_shape) + (2,), value, "sampling locations / offsets")
    _expect(attn, attn_shape, value, "attention weights / logits")
    _expect(grad_output, out_shape, value, "grad_output")
    _expect(grad_value, value.shape, value, "grad_value")
    _expect(grad_loc, tuple(attn_shape) + (2,), value, "grad of locations / offsets")
    _expect(grad_attn, attn_shape, value, "grad of weights / logits")


def msda_backward(value, spatial_shapes, level_start_index, sampling_loc, attn_weight,
                  grad_output, grad_value=None, grad_sampling_loc=None, grad_attn_weight=None,
                  workspace: Optional[torch.Tensor] = None, accumulate: bool = False,
                  stream=None):
    """(grad_value, grad_sampling_loc, grad_attn_weight) of MSDeformAttn (see include/msda.h)."""
    bs, K, M, D, L, P, Q = _dims(value, spatial_shapes, sampling_loc)
    code = _dtype_code(value, spatial_shapes)
    dev = value.device
    _check_grads(value, sampling_loc, attn_weight, grad_output, grad_value, grad_sampling_loc,
                 grad_attn_weight, (bs, Q, M, L, P), (bs, Q, M * D))
    if grad_value is None:
        grad_value = torch.empty_like(value)
    if grad_sampling_loc is None:
        grad_sampling_loc = torch.empty_like(sampling_loc)
    if grad_attn_weight is None:
        grad_attn_weight = torch.empty_like(attn_weight)
    need = msda_backward_workspace_bytes(bs, K, M, D, code)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("msda_backward", _LIB.msda_backward(
        _ptr(value), _ptr(_index(spatial_shapes)), _ptr(_index(level_start_index, spatial_shapes)),
        _ptr(sampling_loc), _ptr(attn_weight), _ptr(grad_output), _ptr(grad_value),
        _ptr(grad_sampling_loc), _ptr(grad_attn_weight),
        _ptr(workspace) if workspace is not None else None, ws_bytes,
        bs, K, M, D, L, P, Q, code, MSDA_GRAD_VALUE_ACCUMULATE if accumulate else 0,
        _stream(stream)))
    return grad_value, grad_sampling_loc, grad_attn_weight


def msda_backward_noalloc(value, spatial_shapes, level_start_index, sampling_loc, attn_weight,
                          grad_output, grad_value, grad_sampling_loc, grad_attn_weight,
                          accumulate: bool = False, stream=None):
    """bf16 backward into caller-provided gradient tensors, with the library's own
    fixed scratch array instead of a workspace (see msda_backward_noalloc in
    include/msda.h); the library allocates nothing."""
    bs, K, M, D, L, P, Q = _dims(value, spatial_shapes, sampling_loc)
    _check_grads(value, sampling_loc, attn_weight, grad_output, grad_value, grad_sampling_loc,
                 grad_attn_weight, (bs, Q, M, L, P), (bs, Q, M * D))
    _check("msda_backward_noalloc", _LIB.msda_backward_noalloc(
        _ptr(value), _ptr(_index(spatial_shapes)), _ptr(_index(level_start_index, spatial_shapes)),
        _ptr(sampling_loc), _ptr(attn_weight), _ptr(grad_output), _ptr(grad_value),
        _ptr(grad_sampling_loc), _ptr(grad_attn_weight), bs, K, M, D, L, P, Q,
        _dtype_code(value, spatial_shapes), MSDA_GRAD_VALUE_ACCUMULATE if accumulate else 0,
        _stream(stream)))
    return grad_value, grad_sampling_loc, grad_attn_weight


def msda_linear(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y = x @ weight.T + bias on the tensor cores (see msda_linear in include/msda.h):
    x [..., in] and weight [out, in] bf16 (or both fp16) CUDA tensors, bias fp32 or
    the operands' dtype [out] or None; returns [..., out] in the operands' dtype."""
    if x.dtype not in (torch.bfloat16, torch.float16) or weight.dtype != x.dtype:
        raise TypeError("msda_linear takes bf16 (or fp16) x and weight of one dtype")
    if not (x.is_cuda and weight.is_cuda) or x.device != weight.device:
        raise ValueError("x and weight must be CUDA tensors on one device")
    if weight.dim() != 2 or x.shape[-1] != weight.shape[1]:
        raise ValueError("weight must be [out_features, in_features] with in_features = x.shape[-1]")
    x2 = x.reshape(-1, x.shape[-1])
    if not x2.is_contiguous():
        raise ValueError("x must be contiguous")
    weight = weight.contiguous()
    n_out = int(weight.shape[0])
    code = MSDA_BF16 if x.dtype == torch.bfloat16 else MSDA_F16
    if bias is not None:
        if (bias.dtype not in (torch.float32, x.dtype) or bias.shape != (n_out,)
                or bias.device != x.device):
            raise ValueError("bias must be an fp32 or x-dtype [out_features] tensor on x's device")
        bias = bias.contiguous()
        if bias.dtype == x.dtype:
            code |= MSDA_LINEAR_BIAS_HALF
    if out is None:
        out = torch.empty(*x.shape[:-1], n_out, dtype=x.dtype, device=x.device)
    elif out.dtype != x.dtype or out.shape != (*x.shape[:-1], n_out) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [..., out_features] tensor of x's dtype")
    _check("msda_linear", _LIB.msda_linear(
        _ptr(x2), _ptr(weight), _ptr(bias) if bias is not None else None, _ptr(out),
        int(x2.shape[0]), int(x2.shape[1]), n_out, code, _stream(stream)))
    return out


def msda_linear_workspace_bytes(rows: int, in_features: int, out_features: int,
                                dtype: int = MSDA_F32) -> int:
    return int(_LIB.msda_linear_workspace_bytes(rows, in_features, out_features, dtype))


def msda_linear_f32(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor] = None,
                    out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    """y = x @ weight.T + bias in fp32 on the tensor cores, three TF32 products
    (see msda_linear_f32 in include/msda.h): x [..., in], weight [out, in] and
    bias [out] (or None) fp32 CUDA tensors; returns fp32 [..., out].  The split
    operands go to `workspace` (allocated here when None)."""
    if x.dtype != torch.float32 or weight.dtype != torch.float32:
        raise TypeError("msda_linear_f32 takes fp32 x and weight")
    if not (x.is_cuda and weight.is_cuda) or x.device != weight.device:
        raise ValueError("x and weight must be CUDA tensors on one device")
    if weight.dim() != 2 or x.shape[-1] != weight.shape[1]:
        raise ValueError("weight must be [out_features, in_features] with in_features = x.shape[-1]")
    x2 = x.reshape(-1, x.shape[-1])
    if not x2.is_contiguous():
        raise ValueError("x must be contiguous")
    weight = weight.contiguous()
    rows, n_in, n_out = int(x2.shape[0]), int(x2.shape[1]), int(weight.shape[0])
    if bias is not None:
        if bias.dtype != torch.float32 or bias.shape != (n_out,) or bias.device != x.device:
            raise ValueError("bias must be an fp32 [out_features] tensor on x's device")
        bias = bias.contiguous()
    if out is None:
        out = torch.empty(*x.shape[:-1], n_out, dtype=torch.float32, device=x.device)
    elif out.dtype != torch.float32 or out.shape != (*x.shape[:-1], n_out) or not out.is_contiguous():
        raise ValueError("out must be a contiguous fp32 [..., out_features] tensor")
    need = msda_linear_workspace_bytes(rows, n_in, n_out, MSDA_F32)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("msda_linear_f32", _LIB.msda_linear_f32(
        _ptr(x2), _ptr(weight), _ptr(bias) if bias is not None else None, _ptr(out),
        _ptr(workspace), ws_bytes, rows, n_in, n_out, _stream(stream)))
    return out


def msda_linear_wgrad_f32(grad_y: torch.Tensor, x: torch.Tensor, bias: bool = True,
                          grad_w: Optional[torch.Tensor] = None,
                          grad_b: Optional[torch.Tensor] = None, accumulate: bool = False,
                          stream=None):
    """(grad_w, grad_b) of y = x @ w.T + b in fp32 on the tensor cores (see
    msda_linear_wgrad_f32 in include/msda.h): grad_y [..., out] and x [..., in]
    fp32 CUDA tensors; grad_w = grad_y^T x [out, in], grad_b = sum of grad_y
    [out] (None unless `bias`).  With `accumulate` the sums are added to the
    given grad_w / grad_b."""
    if grad_y.dtype != torch.float32 or x.dtype != torch.float32:
        raise TypeError("msda_linear_wgrad_f32 takes fp32 grad_y and x")
    if not (grad_y.is_cuda and x.is_cuda) or grad_y.device != x.device:
        raise ValueError("grad_y and x must be CUDA tensors on one device")
    g2 = grad_y.reshape(-1, grad_y.shape[-1])
    x2 = x.reshape(-1, x.shape[-1])
    if g2.shape[0] != x2.shape[0] or not (g2.is_contiguous() and x2.is_contiguous()):
        raise ValueError("grad_y and x must be contiguous with the same leading dimensions")
    rows, n_out, n_in = int(g2.shape[0]), int(g2.shape[1]), int(x2.shape[1])
    dev = x.device
    if grad_w is None:
        if accumulate:
            raise ValueError("accumulate needs grad_w")
        grad_w = torch.empty(n_out, n_in, dtype=torch.float32, device=dev)
    elif grad_w.shape != (n_out, n_in) or grad_w.dtype != torch.float32 or not grad_w.is_contiguous():
        raise ValueError("grad_w must be a contiguous fp32 [out_features, in_features] tensor")
    if bias:
        if grad_b is None:
            if accumulate:
                raise ValueError("accumulate needs grad_b")
            grad_b = torch.empty(n_out, dtype=torch.float32, device=dev)
        elif grad_b.shape != (n_out,) or grad_b.dtype != torch.float32:
            raise ValueError("grad_b must be an fp32 [out_features] tensor")
    else:
        grad_b = None
    _check("msda_linear_wgrad_f32", _LIB.msda_linear_wgrad_f32(
        _ptr(g2), _ptr(x2), _ptr(grad_w), _ptr(grad_b) if grad_b is not None else None,
        rows, n_in, n_out, MSDA_GRAD_VALUE_ACCUMULATE if accumulate else 0, _stream(stream)))
    return grad_w, grad_b


def msda_linear_bias_grad(grad_y: torch.Tensor, grad_b: Optional[torch.Tensor] = None,
                          accumulate: bool = False, stream=None) -> torch.Tensor:
    """fp32 column sums of grad_y [..., features] (fp32, bf16 or fp16 CUDA tensor):
    the bias gradient of a projection (see msda_linear_bias_grad in include/msda.h)."""
    g2 = grad_y.reshape(-1, grad_y.shape[-1])
    if not (g2.is_cuda and g2.is_contiguous()):
        raise ValueError("grad_y must be a contiguous CUDA tensor")
    n = int(g2.shape[1])
    if grad_b is None:
        if accumulate:
            raise ValueError("accumulate needs grad_b")
        grad_b = torch.empty(n, dtype=torch.float32, device=g2.device)
    elif grad_b.shape != (n,) or grad_b.dtype != torch.float32 or grad_b.device != g2.device:
        raise ValueError("grad_b must be an fp32 [features] tensor on grad_y's device")
    _check("msda_linear_bias_grad", _LIB.msda_linear_bias_grad(
        _ptr(g2), _ptr(grad_b), int(g2.shape[0]), n, _dtype_code(g2),
        MSDA_GRAD_VALUE_ACCUMULATE if accumulate else 0, _stream(stream)))
    return grad_b


def _fused_dims(value, spatial_shapes, reference_points, sampling_offsets, attn_logits):
    bs, K, M, D, L, P, Q = _dims(value, spatial_shapes, sampling_offsets)
    if reference_points.dim() != 4 or tuple(reference_points.shape[:3]) != (bs, Q, L):
        raise ValueError("reference_points must be [bs, Q, L, 2 or 4]")
    ref_dim = int(reference_points.shape[3])
    _expect(reference_points, (bs, Q, L, ref_dim), value, "reference_points")
    _expect(sampling_offsets, (bs, Q, M, L, P, 2), value, "sampling_offsets")
    _expect(attn_logits, (bs, Q, M, L * P), value, "attn_logits")
    return bs, K, M, D, L, P, Q, ref_dim


def _mask(key_padding_mask: Optional[torch.Tensor], bs: int, K: int) -> Optional[torch.Tensor]:
    """The [bs, K] key padding mask as one byte per key (True / nonzero = padded)."""
    if key_padding_mask is None:
        return None
    if tuple(key_padding_mask.shape) != (bs, K):
        raise ValueError(f"key_padding_mask must be [bs, num_keys] = {(bs, K)}")
    if key_padding_mask.dtype not in (torch.bool, torch.uint8):
        raise TypeError("key_padding_mask must be torch.bool or torch.uint8")
    if key_padding_mask.device.type != "cuda":
        raise ValueError("key_padding_mask must be on the CUDA device")
    return key_padding_mask.contiguous()


def msda_forward_fused(value, spatial_shapes, level_start_index, reference_points,
                       sampling_offsets, attn_logits, key_padding_mask=None, output=None,
                       stream=None) -> torch.Tensor:
    """output [bs, Q, M*D]: softmax of the logits, locations from the reference
    points and offsets, and the optional key padding mask applied to value, then
    the operator, in one kernel (see include/msda.h)."""
    bs, K, M, D, L, P, Q, ref_dim = _fused_dims(value, spatial_shapes, reference_points,
                                                sampling_offsets, attn_logits)
    code = _dtype_code(value, spatial_shapes)
    _expect(output, (bs, Q, M * D), value, "output")
    mask = _mask(key_padding_mask, bs, K)
    if output is None:
        output = torch.empty((bs, Q, M * D), dtype=value.dtype, device=value.device)
    _check("msda_forward_fused", _LIB.msda_forward_fused(
        _ptr(value), _ptr(_index(spatial_shapes)), _ptr(_index(level_start_index, spatial_shapes)),
        _ptr(reference_points), _ptr(sampling_offsets), _ptr(attn_logits), _ptr(mask),
        _ptr(output),
        bs, K, M, D, L, P, Q, ref_dim, code, _stream(stream)))
    return output


def msda_backward_fused(value, spatial_shapes, level_start_index, reference_points,
                        sampling_offsets, attn_logits, grad_output, key_padding_mask=None,
                        grad_value=None, grad_sampling_offsets=None, grad_attn_logits=None,
                        reference_grad: bool = True, workspace: Optional[torch.Tensor] = None,
                        accumulate: bool = False, stream=None):
    """(grad_value, grad_sampling_offsets, grad_attn_logits, grad_reference_points or None);
    the reference-point gradient is an fp32 tensor [bs, Q, L, ref_dim].  With a key
    padding mask, grad_value is taken with respect to the value before masking."""
    bs, K, M, D, L, P, Q, ref_dim = _fused_dims(value, spatial_shapes, reference_points,
                                                sampling_offsets, attn_logits)
    code = _dtype_code(value, spatial_shapes)
    dev = value.device
    _expect(grad_output, (bs, Q, M * D), value, "grad_output")
    _expect(grad_value, value.shape, value, "grad_value")
    _expect(grad_sampling_offsets, sampling_offsets.shape, value, "grad_sampling_offsets")
    _expect(grad_attn_logits, attn_logits.shape, value, "grad_attn_logits")
    mask = _mask(key_padding_mask, bs, K)
    if grad_value is None:
        grad_value = torch.empty_like(value)
    if grad_sampling_offsets is None:
        grad_sampling_offsets = torch.empty_like(sampling_offsets)
    if grad_attn_logits is None:
        grad_attn_logits = torch.empty_like(attn_logits)
    grad_ref = (torch.empty((bs, Q, L, ref_dim), dtype=torch.float32, device=dev)
                if reference_grad else None)
    need = msda_backward_workspace_bytes(bs, K, M, D, code)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("msda_backward_fused", _LIB.msda_backward_fused(
        _ptr(value), _ptr(_index(spatial_shapes)), _ptr(_index(level_start_index, spatial_shapes)),
        _ptr(reference_points), _ptr(sampling_offsets), _ptr(attn_logits), _ptr(mask),
        _ptr(grad_output),
        _ptr(grad_value), _ptr(grad_sampling_offsets), _ptr(grad_attn_logits), _ptr(grad_ref),
        _ptr(workspace) if workspace is not None else None, ws_bytes,
        bs, K, M, D, L, P, Q, ref_dim, code, MSDA_GRAD_VALUE_ACCUMULATE if accumulate else 0,
        _stream(stream)))
    return grad_value, grad_sampling_offsets, grad_attn_logits, grad_ref


def msda_zero_fill(t: torch.Tensor, stream=None) -> torch.Tensor:
    _check("msda_zero_fill", _LIB.msda_zero_fill(_ptr(t), t.numel() * t.element_size(),
                                                 _stream(stream)))
    return t


def msda_check_shapes(spatial_shapes: torch.Tensor, level_start_index: torch.Tensor,
                      num_keys: int, stream=None) -> int:
    """BLOCKING. 0 (MSDA_OK) or 7 (MSDA_ERR_SHAPES); raises on other errors (int64 indices)."""
    if spatial_shapes.dtype != torch.int64 or level_start_index.dtype != torch.int64:
        raise TypeError("msda_check_shapes takes int64 index tensors")
    st = _LIB.msda_check_shapes(_ptr(_index(spatial_shapes)), _ptr(_index(level_start_index)),
                                int(spatial_shapes.shape[0]), int(num_keys), _stream(stream))
    if st not in (0, 7):
        _check("msda_check_shapes", st)
    return st


def msda_last_device_error(stream=None) -> int:
    """BLOCKING. 0, or 8 (MSDA_ERR_DEVICE_BOUNDS) when a kernel skipped an inconsistent level."""
    st = _LIB.msda_last_device_error(_stream(stream))
    if st not in (0, 8):
        _check("msda_last_device_error", st)
    return st


class MSDeformAttnFunction(torch.autograd.Function):
    """Autograd wrapper with the argument order of the DQ-DETR ops page's
    ``MSDeformAttnFunction``: (value, spatial_shapes, level_start_index,
    sampling_loc, attn_weight, im2col_step).  ``im2col_step`` is accepted and
    ignored (the kernels keep no column buffer).  backward returns
    (grad_value, None, None, grad_sampling_loc, grad_attn_weight, None)."""

    @staticmethod
    def forward(ctx, value, spatial_shapes, level_start_index, sampling_loc, attn_weight,
                im2col_step=64):
        value, sampling_loc, attn_weight = (value.contiguous(), sampling_loc.contiguous(),
                                            attn_weight.contiguous())
        out = msda_forward(value, spatial_shapes, level_start_index, sampling_loc, attn_weight)
        ctx.save_for_backward(value, spatial_shapes, level_start_index, sampling_loc, attn_weight)
        return out

    @staticmethod
    def backward(ctx, grad_output):
        value, spatial_shapes, level_start_index, sampling_loc, attn_weight = ctx.saved_tensors
        gv, gl, ga = msda_backward(value, spatial_shapes, level_start_index, sampling_loc,
                                   attn_weight, grad_output.contiguous())
        return gv, None, None, gl, ga, None


class MSDeformAttnFusedFunction(torch.autograd.Function):
    """Autograd wrapper of the fused entry points: (value, spatial_shapes,
    level_start_index, reference_points, sampling_offsets, attn_logits,
    key_padding_mask or None) -> output; backward returns gradients for value
    (before masking), reference_points (when it requires grad),
    sampling_offsets and attn_logits."""

    @staticmethod
    def forward(ctx, value, spatial_shapes, level_start_index, reference_points,
                sampling_offsets, attn_logits, key_padding_mask=None):
        value, reference_points = value.contiguous(), reference_points.contiguous()
        sampling_offsets, attn_logits = sampling_offsets.contiguous(), attn_logits.contiguous()
        out = msda_forward_fused(value, spatial_shapes, level_start_index, reference_points,
                                 sampling_offsets, attn_logits, key_padding_mask)
        ctx.save_for_backward(value, spatial_shapes, level_start_index, reference_points,
                              sampling_offsets, attn_logits, key_padding_mask)
        return out

    @staticmethod
    def backward(ctx, grad_output):
        value, shapes, lsi, ref, off, logits, mask = ctx.saved_tensors
        need_ref = ctx.needs_input_grad[3]
        gv, goff, glog, gref = msda_backward_fused(value, shapes, lsi, ref, off, logits,
                                                   grad_output.contiguous(), mask,
                                                   reference_grad=need_ref)
        return gv, None, None, (gref.to(ref.dtype) if need_ref else None), goff, glog, None


def ms_deform_attn_fused(value, spatial_shapes, level_start_index, reference_points,
                         sampling_offsets, attn_logits, key_padding_mask=None):
    return MSDeformAttnFusedFunction.apply(value, spatial_shapes, level_start_index,
                                           reference_points, sampling_offsets, attn_logits,
                                           key_padding_mask)


def ms_deform_attn(value, spatial_shapes, level_start_index, sampling_loc, attn_weight):
    return MSDeformAttnFunction.apply(value, spatial_shapes, level_start_index, sampling_loc,
                                      attn_weight, 64)
