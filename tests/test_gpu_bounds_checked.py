"""The bounds-checked build (libmsda_checked.so, -DMSDA_BOUNDS_CHECK) on
randomized shapes of every dtype, both backward kernels and the fused entry
points: every value / grad_value row the kernels touch must lie inside its
tensor (the checked build records any that does not in the device error word,
which msda_last_device_error reports, and skips it), and the results must
still match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fused as ofused
from scale_deformable_attention_05_b300 import inputs as gen
from tests.gpu_helpers import assert_grad_close, assert_out_close, host

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_05_b300 import binding as B
    from scale_deformable_attention_05_b300 import build
    return B.load_library(build.build_checked())


CASES = [
    # (seed, bs, shapes, M, D, P, Q, dtype)
    (201, 2, ((7, 9), (4, 5), (1, 1)), 2, 32, 4, 13, "f32"),
    (202, 1, ((9, 7),), 3, 8, 9, 6, "f32"),
    (203, 2, ((5, 6), (3, 3)), 2, 64, 2, 9, "bf16"),
    (204, 1, ((8, 8), (4, 4)), 1, 256, 16, 5, "f32"),      # merge kernel (one group per warp)
    (205, 2, ((6, 5), (3, 2)), 2, 16, 3, 11, "f16"),
    # fp32 backward's dense shape: 4,400 tiles in a grid of 1,100 CTAs, 7 per SM on 148 SMs
    (206, 2, ((60, 80), (30, 40)), 8, 32, 4, 1100, "f32"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"seed{c[0]}")
def test_checked_build_plain(lib, case):
    seed, bs, shapes, M, D, P, Q, dtype = case
    wl = gen.random_workload(seed, bs, shapes, M, D, P, Q, dtype=dtype)
    inp = gen.make_inputs(wl)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]

    def dev(k):
        if dtype == "f32":
            return torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()
        return torch.from_numpy(inp[k + "_" + dtype].view(np.int16).copy()).view(tdt).cuda()

    v, loc, w, g = dev("value"), dev("sampling_locations"), dev("attention_weights"), \
        dev("grad_output")
    sh = torch.from_numpy(inp["spatial_shapes"]).cuda()
    lsi = torch.from_numpy(inp["level_start_index"]).cuda()
    code = {"f32": 0, "bf16": 1, "f16": 2}[dtype]
    dims = (wl.bs, wl.num_keys, wl.num_heads, wl.head_dim, wl.num_levels, wl.num_points,
            wl.num_queries)
    out = torch.empty(bs, Q, M * D, dtype=tdt, device="cuda")
    gv, gl, gw = torch.empty_like(v), torch.empty_like(loc), torch.empty_like(w)
    ws = torch.empty(max(16, int(lib.msda_backward_workspace_bytes(bs, wl.num_keys, M, D, code))),
                     dtype=torch.uint8, device="cuda")
    P_ = lambda t: t.data_ptr()
    st = torch.cuda.current_stream().cuda_stream
    assert lib.msda_forward(P_(v), P_(sh), P_(lsi), P_(loc), P_(w), P_(out), *dims, code, st) == 0
    assert lib.msda_backward(P_(v), P_(sh), P_(lsi), P_(loc), P_(w), P_(g), P_(gv), P_(gl),
                             P_(gw), P_(ws), ws.numel(), *dims, code, 0, st) == 0
    torch.cuda.synchronize()
    assert lib.msda_last_device_error(None) == 0          # no row outside its tensor
    ref_out, (rv, rl, rw) = oracle.run_inputs(inp)
    assert_out_close(host(out), ref_out, dtype)
    assert_grad_close(host(gv), rv, dtype, "grad_value")
    assert_grad_close(host(gl), rl, dtype, "grad_sampling_loc")
    assert_grad_close(host(gw), rw, dtype, "grad_attn_weight")


@pytest.mark.parametrize("ref_dim", [2, 4])
def test_checked_build_fused_with_mask(lib, ref_dim):
    wl = gen.random_workload(210 + ref_dim, 2, ((9, 7), (5, 4), (3, 2)), 2, 32, 4, 13)
    inp = gen.make_fused_inputs(wl, ref_dim)
    mask = gen.padding_mask(wl, min_ratio=0.5)
    t = lambda k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()
    v, ref, off, lg, g = (t(k) for k in ("value", "reference_points", "sampling_offsets",
                                         "attention_logits", "grad_output"))
    sh = torch.from_numpy(inp["spatial_shapes"]).cuda()
    lsi = torch.from_numpy(inp["level_start_index"]).cuda()
    dm = torch.from_numpy(mask).cuda()
    dims = (wl.bs, wl.num_keys, wl.num_heads, wl.head_dim, wl.num_levels, wl.num_points,
            wl.num_queries)
    out = torch.empty(wl.bs, wl.num_queries, wl.num_heads * wl.head_dim, device="cuda")
    gv, goff, glog = torch.empty_like(v), torch.empty_like(off), torch.empty_like(lg)
    gref = torch.empty(ref.shape, device="cuda")
    P_ = lambda x: x.data_ptr()
    st = torch.cuda.current_stream().cuda_stream
    assert lib.msda_forward_fused(P_(v), P_(sh), P_(lsi), P_(ref), P_(off), P_(lg), P_(dm),
                                  P_(out), *dims, ref_dim, 0, st) == 0
    assert lib.msda_backward_fused(P_(v), P_(sh), P_(lsi), P_(ref), P_(off), P_(lg), P_(dm),
                                   P_(g), P_(gv), P_(goff), P_(glog), P_(gref), None, 0, *dims,
                                   ref_dim, 0, 0, st) == 0
    torch.cuda.synchronize()
    assert lib.msda_last_device_error(None) == 0
    oargs = tuple(inp[k] for k in ("value", "spatial_shapes", "level_start_index",
                                   "reference_points", "sampling_offsets", "attention_logits"))
    assert_out_close(host(out), ofused.forward(*oargs, padding_mask=mask), "f32")
    rv, roff, rlog, rref = ofused.backward(*oargs, inp["grad_output"], padding_mask=mask)
    assert_grad_close(host(gv), rv, "f32", "grad_value")
    assert_grad_close(host(goff), roff, "f32", "grad_sampling_offsets")
    assert_grad_close(host(glog), rlog, "f32", "grad_attn_logits")
    assert_grad_close(host(gref), rref, "f32", "grad_reference_points")
