"""Helpers shared by the GPU tests: device copies of seeded inputs and the
comparison rules (tolerances) the parity tests apply."""
from __future__ import annotations

import numpy as np
import torch

from scale_deformable_attention_05_b300 import inputs as gen

# fp32 forward: |err| <= 1e-5 + 1e-5 |ref| element-wise.
# fp32 grads:   max|err| <= 1e-4 * max|ref| per tensor.
# bf16 output:  |err| <= 1e-2 + 1e-2 |ref| element-wise.
# bf16 grads:   max|err| <= 1e-2 * max|ref| per tensor.
# fp16 output:  |err| <= 1e-3 + 1e-3 |ref| element-wise (one RNE rounding to an
#               11-bit significand is <= 2^-12 |ref|; fp32 accumulation adds ~1e-7).
# fp16 grads:   max|err| <= 1e-3 * max|ref| per tensor.
TOL = {
    "f32": {"out": (1e-5, 1e-5), "grad": 1e-4},
    "bf16": {"out": (1e-2, 1e-2), "grad": 1e-2},
    "f16": {"out": (1e-3, 1e-3), "grad": 1e-3},
}


def to_device(inp, wl, device="cuda"):
    """Torch CUDA tensors holding exactly the generator's values (bf16 from its bits)."""
    def t(name):
        if wl.dtype in ("bf16", "f16"):
            bits = inp[name + "_" + wl.dtype]
            tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
            x = torch.from_numpy(bits.view(np.int16).copy()).view(tdt)
            return x.to(device)
        return torch.from_numpy(np.ascontiguousarray(inp[name])).to(device)

    d = {k: t(k) for k in ("value", "sampling_locations", "attention_weights")}
    if "grad_output" in inp:
        d["grad_output"] = t("grad_output")
    d["spatial_shapes"] = torch.from_numpy(inp["spatial_shapes"]).to(device)
    d["level_start_index"] = torch.from_numpy(inp["level_start_index"]).to(device)
    return d


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_out_close(got: np.ndarray, ref: np.ndarray, dtype: str, what="output"):
    rtol, atol = TOL[dtype]["out"]
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r}")


def assert_grad_close(got: np.ndarray, ref: np.ndarray, dtype: str, what="grad"):
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    tol = TOL[dtype]["grad"] * scale
    if err > tol and err > 1e-30:
        raise AssertionError(f"{what}: max|err| {err:.3e} > {TOL[dtype]['grad']} * max|ref| "
                             f"({scale:.3e})")


def empty_cache():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
