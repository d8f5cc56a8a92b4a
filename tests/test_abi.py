"""The C ABI library loads, exports every symbol include/msda.h declares, and
rejects bad arguments on the host before touching the device.

No test here launches device work: every call made below fails a host-side
check and returns before the first CUDA runtime call, so these run on a
machine without a GPU.
"""
import ctypes
import os
import re
import subprocess

import pytest

from scale_deformable_attention_05_b300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msda.h")


def _declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MSDA_API\s+[\w\s\*]+?\b(msda_\w+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    assert set(B.EXPORTED_SYMBOLS) <= set(names)
    assert len(names) >= 8


def test_library_exports_every_declared_symbol():
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in _declared_functions() if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in _declared_functions():
        assert getattr(lib, n) is not None


def test_library_exports_nothing_else():
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(_declared_functions())


def test_version_and_status_strings():
    assert B.msda_version() == 1
    for code in range(9):
        s = B.msda_status_string(code)
        assert s and s != "unknown status"
    assert B.msda_status_string(99) == "unknown status"


def test_workspace_bytes():
    assert B.msda_backward_workspace_bytes(2, 22223, 8, 32, B.MSDA_F32) == 0
    assert B.msda_backward_workspace_bytes(4, 22223, 8, 32, B.MSDA_BF16) == 4 * 22223 * 8 * 32 * 4
    assert B.msda_backward_workspace_bytes(1, 100, 2, 8, B.MSDA_F16) == 100 * 2 * 8 * 4
    assert B.msda_backward_workspace_bytes(
        1, 100, 2, 8, B.MSDA_F16 | B.MSDA_INDEX_INT32) == 100 * 2 * 8 * 4
    assert B.msda_backward_workspace_bytes(1, 100, 2, 8, B.MSDA_F32 | B.MSDA_INDEX_INT32) == 0
    assert B.msda_backward_workspace_bytes(1, 100, 2, 8, 3) == 0          # unknown dtype
    assert B.msda_backward_workspace_bytes(1, 100, 2, 8, 0x201) == 0      # unknown flag bit
    assert B.msda_backward_workspace_bytes(-1, 10, 8, 32, B.MSDA_BF16) == 0


# ----------------------------------------------------- host-side rejections
L = B._LIB
A = 0x10000  # an aligned, never-dereferenced stand-in address
DIMS = dict(bs=1, K=10000, M=4, D=32, L=1, P=8, Q=16)


def _fwd(value=A, shapes=A, lsi=A, loc=A, w=A, out=A, dtype=0, **kw):
    d = dict(DIMS, **kw)
    return L.msda_forward(value, shapes, lsi, loc, w, out, d["bs"], d["K"], d["M"], d["D"],
                          d["L"], d["P"], d["Q"], dtype, None)


def _bwd(value=A, shapes=A, lsi=A, loc=A, w=A, g=A, gv=A, gl=A, gw=A, ws=None, ws_bytes=0,
         dtype=0, flags=0, **kw):
    d = dict(DIMS, **kw)
    return L.msda_backward(value, shapes, lsi, loc, w, g, gv, gl, gw, ws, ws_bytes, d["bs"],
                           d["K"], d["M"], d["D"], d["L"], d["P"], d["Q"], dtype, flags, None)


@pytest.mark.parametrize("kw,status", [
    (dict(out=None), 1),
    (dict(value=None), 1),
    (dict(loc=None), 1),
    (dict(w=None), 1),
    (dict(shapes=None), 1),
    (dict(lsi=None), 1),
    (dict(bs=-1), 2),
    (dict(Q=-3), 2),
    (dict(D=12), 3),
    (dict(D=520), 3),
    (dict(L=17, P=1), 3),
    (dict(L=4, P=65), 3),
    (dict(dtype=3), 3),          # unknown element type
    (dict(dtype=0x200), 3),      # unknown flag bit
    (dict(dtype=0x103), 3),      # int32 indices with an unknown element type
    (dict(value=A + 8), 4),
    (dict(loc=A + 4), 4),
    (dict(out=A + 2), 4),
    (dict(bs=70000, Q=70000), 2),
])
def test_forward_rejects_on_host(kw, status):
    assert _fwd(**kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(gv=None), 1),
    (dict(gl=None), 1),
    (dict(gw=None), 1),
    (dict(g=None), 1),
    (dict(flags=2), 3),
    (dict(D=4), 3),
    (dict(gl=A + 8), 4),
    (dict(dtype=1), 5),                       # bf16 needs a workspace
    (dict(dtype=2), 5),                       # so does fp16
    (dict(dtype=2 | 0x100), 5),               # with int32 indices too
    (dict(dtype=3), 3),                       # unknown element type
    (dict(dtype=1, ws=A, ws_bytes=16), 5),    # too small
    (dict(dtype=1, ws=A + 4, ws_bytes=1 << 30), 4),
])
def test_backward_rejects_on_host(kw, status):
    assert _bwd(**kw) == status


def test_fused_entry_points_reject_on_host():
    d = DIMS
    fwd = lambda ref_dim=2, L=1, P=8, ref=A: L_.msda_forward_fused(
        A, A, A, ref, A, A, None, A, d["bs"], d["K"], d["M"], d["D"], L, P, d["Q"], ref_dim, 0,
        None)
    L_ = L
    assert fwd(ref_dim=3) == 3                 # references are (x, y) or (x, y, w, h)
    assert fwd(L=5, P=16) == 3                 # L*P above MSDA_MAX_FUSED_LEVEL_POINTS
    assert fwd(ref=None) == 1
    assert fwd(ref=A + 4) == 4
    bwd = lambda ref_dim=2, gref=None, dtype=0: L.msda_backward_fused(
        A, A, A, A, A, A, None, A, A, A, A, gref, None, 0, d["bs"], d["K"], d["M"], d["D"], 1, 8,
        d["Q"], ref_dim, dtype, 0, None)
    assert bwd(ref_dim=1) == 3
    assert bwd(gref=A + 8) == 4                # fp32 reference gradient must be 16-byte aligned
    assert bwd(dtype=1) == 5                   # bf16 still needs the grad_value workspace


def test_zero_fill_and_check_shapes_reject_on_host():
    assert L.msda_zero_fill(None, 16, None) == 1
    assert L.msda_zero_fill(A + 4, 16, None) == 4
    assert L.msda_zero_fill(A, 15, None) == 4
    assert L.msda_zero_fill(None, 0, None) == 0
    assert L.msda_check_shapes(None, None, 1, 10, None) == 1
    assert L.msda_check_shapes(A, A, 17, 10, None) == 3
    assert L.msda_check_shapes(A, A, -1, 10, None) == 2
    assert L.msda_check_shapes(None, None, 0, 0, None) == 0
    assert L.msda_check_shapes(None, None, 0, 5, None) == 7


def test_binding_rejects_cpu_tensors():
    import torch
    v = torch.zeros(1, 4, 1, 8)
    loc = torch.zeros(1, 2, 1, 1, 1, 2)
    w = torch.zeros(1, 2, 1, 1, 1)
    shapes = torch.tensor([[2, 2]])
    lsi = torch.tensor([0])
    with pytest.raises(ValueError, match="CUDA"):
        B.msda_forward(v, shapes, lsi, loc, w)


def test_binding_rejects_mismatched_dtypes_and_shapes():
    """Every float tensor is read with the value's element type: the binding
    refuses mismatches before the library sees a pointer."""
    import torch
    v = torch.zeros(1, 4, 1, 8)
    loc = torch.zeros(1, 2, 1, 1, 1, 2)
    w = torch.zeros(1, 2, 1, 1, 1)
    shapes = torch.tensor([[2, 2]])
    lsi = torch.tensor([0])
    with pytest.raises(TypeError, match="dtype"):
        B.msda_forward(v, shapes, lsi, loc.bfloat16(), w)
    with pytest.raises(TypeError, match="dtype"):
        B.msda_forward(v, shapes, lsi, loc, w.half())
    with pytest.raises(ValueError, match="shape"):
        B.msda_forward(v, shapes, lsi, loc, torch.zeros(1, 2, 1, 1, 2))
    with pytest.raises(ValueError, match="shape"):
        B.msda_backward(v, shapes, lsi, loc, w, torch.zeros(1, 2, 4))
    ref = torch.zeros(1, 2, 1, 2)
    lg = torch.zeros(1, 2, 1, 1)
    with pytest.raises(TypeError, match="dtype"):
        B.msda_forward_fused(v, shapes, lsi, ref.double(), loc, lg)
    with pytest.raises(ValueError, match="key_padding_mask"):
        B.msda_forward_fused(v, shapes, lsi, ref, loc, lg, torch.zeros(1, 3, dtype=torch.bool))
    with pytest.raises(TypeError, match="key_padding_mask"):
        B.msda_forward_fused(v, shapes, lsi, ref, loc, lg, torch.zeros(1, 4))


def test_python_constants_match_header():
    text = open(HEADER).read()
    for name in ("MSDA_F32", "MSDA_BF16", "MSDA_F16", "MSDA_INDEX_INT32",
                 "MSDA_MAX_FUSED_LEVEL_POINTS", "MSDA_GRAD_VALUE_ACCUMULATE"):
        m = re.search(name + r"\s*=?\s*(0x[0-9a-fA-F]+|\d+)", text)
        assert m, name
        assert int(m.group(1), 0) == getattr(B, name), name


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "scale_deformable_attention_05_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".cpp", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "msda_oracle" not in text and "liboracle" not in text, f


def test_module_initial_state():
    """MSDeformAttn starts with zero offset / attention weights and the offset
    bias on the ring of head directions, point p at p + 1 steps (checked against
    the directions written out by hand for 8 heads)."""
    import torch
    from scale_deformable_attention_05_b300.module import MSDeformAttn
    layer = MSDeformAttn(64, n_levels=2, n_heads=8, n_points=3)
    assert not layer.sampling_offsets.weight.any()
    assert not layer.attention_weights.weight.any() and not layer.attention_weights.bias.any()
    assert not layer.value_proj.bias.any() and not layer.output_proj.bias.any()
    b = layer.sampling_offsets.bias.detach().double().reshape(8, 2, 3, 2)
    ring = torch.tensor([[1, 0], [1, 1], [0, 1], [-1, 1], [-1, 0], [-1, -1], [0, -1], [1, -1]],
                        dtype=torch.float64)
    for p in range(3):
        for lvl in range(2):
            torch.testing.assert_close(b[:, lvl, p], ring * (p + 1), rtol=0, atol=1e-6)
    with pytest.raises(ValueError):
        MSDeformAttn(60, n_heads=8)                 # d_model not a multiple of n_heads
    with pytest.raises(ValueError):
        MSDeformAttn(64, n_levels=5, n_heads=8, n_points=16)   # L*P above the fused limit


def test_projection_entry_points_reject_on_host():
    """msda_linear, msda_linear_f32, msda_linear_wgrad_f32 and msda_linear_bias_grad
    refuse unsupported widths, types, flags, missing or misaligned pointers and
    short workspaces before their first CUDA call."""
    lin = lambda x=A, w=A, b=None, y=A, rows=8, k=64, n=16, dtype=1: L.msda_linear(
        x, w, b, y, rows, k, n, dtype, None)
    assert lin(dtype=0) == 3                     # fp32 operands go to msda_linear_f32
    assert lin(dtype=1 | 0x100) == 3             # no index flag here
    assert lin(k=32) == 3 and lin(k=320) == 3    # K a multiple of 64, at most 256
    assert lin(n=24) == 3 and lin(n=272) == 3    # N a multiple of 16, at most 256
    assert lin(rows=-1) == 2
    assert lin(rows=0, x=None) == 0              # nothing to do
    assert lin(x=None) == 1 and lin(y=None) == 1
    assert lin(x=A + 2) == 4 and lin(b=A + 8) == 4
    f32 = lambda x=A, w=A, y=A, ws=A, wsb=1 << 20, rows=8, k=32, n=16: L.msda_linear_f32(
        x, w, None, y, ws, wsb, rows, k, n, None)
    assert f32(k=24) == 3 and f32(n=8) == 3
    assert f32(ws=None) == 5
    assert f32(wsb=B.msda_linear_workspace_bytes(8, 32, 16) - 16) == 5
    assert f32(ws=A + 4) == 4 and f32(w=A + 4) == 4
    assert B.msda_linear_workspace_bytes(8, 32, 16) == 8 * 32 * 16
    assert B.msda_linear_workspace_bytes(8, 32, 16, B.MSDA_BF16) == 0
    wg = lambda gy=A, x=A, gw=A, gb=A, rows=8, k=32, n=16, flags=1: L.msda_linear_wgrad_f32(
        gy, x, gw, gb, rows, k, n, flags, None)
    assert wg(flags=2) == 3 and wg(k=8) == 3 and wg(n=24) == 3
    assert wg(gw=None) == 1 and wg(gy=None) == 1
    assert wg(gw=A + 4) == 4 and wg(gb=A + 4) == 4
    assert wg(rows=0) == 0                       # accumulating nothing: no launch
    bg = lambda gy=A, gb=A, rows=8, n=16, dtype=1, flags=1: L.msda_linear_bias_grad(
        gy, gb, rows, n, dtype, flags, None)
    assert bg(dtype=3) == 3 and bg(n=12) == 3 and bg(n=8 * 257) == 3
    assert bg(dtype=0, n=6) == 3                 # 4 fp32 columns per 16-byte vector
    assert bg(gb=None) == 1 and bg(gy=None) == 1 and bg(gb=A + 4) == 4
    assert bg(rows=0) == 0


def test_projection_constants_match_header():
    text = open(HEADER).read()
    for name in ("MSDA_LINEAR_MAX_FEATURES", "MSDA_LINEAR_BIAS_HALF"):
        m = re.search(r"#define\s+" + name + r"\s+(0x[0-9a-fA-F]+|\d+)", text)
        assert m, name
        assert int(m.group(1), 0) == getattr(B, name), name
    assert B.MSDA_LINEAR_BIAS_BF16 == B.MSDA_LINEAR_BIAS_HALF
