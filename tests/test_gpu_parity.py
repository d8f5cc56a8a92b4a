"""GPU (sm_103a) results against the fp64 CPU oracle, through the C ABI.

Every case draws seeded inputs, runs the CUDA library through its Python
binding (argument marshalling over the C functions of include/msda.h) and the
oracle on the same values, and compares element by element:
  fp32 forward |err| <= 1e-5 + 1e-5|ref|, fp32 grads max|err| <= 1e-4 max|ref|,
  bf16 forward |err| <= 1e-2 + 1e-2|ref|, bf16 grads max|err| <= 1e-2 max|ref|;
and index work (which value rows a sample touches) bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from scale_deformable_attention_05_b300 import inputs as gen
from tests.gpu_helpers import (assert_grad_close, assert_out_close, empty_cache, host,
                               to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_05_b300 import binding
    return binding


def _run(B, wl, inp, backward=True):
    d = to_device(inp, wl)
    args = (d["value"], d["spatial_shapes"], d["level_start_index"], d["sampling_locations"],
            d["attention_weights"])
    out = B.msda_forward(*args)
    grads = B.msda_backward(*args, d["grad_output"]) if backward else None
    torch.cuda.synchronize()
    assert B.msda_last_device_error() == 0
    res = (host(out), tuple(host(g) for g in grads) if grads else None)
    del d, out, grads
    return res


def _check(wl, inp, got_out, got_grads):
    ref_out, ref_grads = oracle.run_inputs(inp, backward_pass=got_grads is not None)
    assert_out_close(got_out, ref_out, wl.dtype)
    if got_grads is not None:
        gv, gl, gw = got_grads
        rv, rl, rw = ref_grads
        assert_grad_close(gv, rv, wl.dtype, "grad_value")
        assert_grad_close(gl, rl, wl.dtype, "grad_sampling_loc")
        assert_grad_close(gw, rw, wl.dtype, "grad_attn_weight")
        # which value rows received gradient is index work: identical sets
        touched_ref = np.any(rv != 0, axis=-1)
        touched_gpu = np.any(gv != 0, axis=-1)
        assert np.array_equal(touched_ref, touched_gpu), "grad_value sparsity pattern differs"


@pytest.mark.parametrize("name", ["tiny", "encoder", "decoder", "encoder_bf16", "encoder_f16",
                                  "envelope"])
def test_named_workload_parity(B, name):
    wl = gen.WORKLOADS[name]
    inp = gen.make_inputs(wl)
    out, grads = _run(B, wl, inp)
    _check(wl, inp, out, grads)
    empty_cache()


RANDOM_CASES = [
    # (seed, bs, shapes, M, D, P, Q, dtype)
    (1, 1, ((7, 9),), 1, 8, 1, 1, "f32"),
    (2, 2, ((5, 3), (1, 1)), 3, 16, 2, 7, "f32"),
    (3, 1, ((13, 1), (1, 11), (4, 4)), 2, 24, 3, 33, "f32"),
    (4, 3, ((9, 7), (5, 4), (3, 2), (2, 1), (1, 1)), 5, 64, 5, 17, "f32"),
    (5, 1, ((31, 17), (16, 9)), 8, 256, 16, 9, "f32"),
    (6, 2, ((11, 6), (6, 3), (3, 2)), 4, 40, 7, 129, "f32"),
    (7, 1, ((7, 9),), 1, 8, 1, 1, "bf16"),
    (8, 2, ((5, 3), (1, 1)), 3, 16, 2, 7, "bf16"),
    (9, 3, ((9, 7), (5, 4), (3, 2), (2, 1), (1, 1)), 5, 64, 5, 17, "bf16"),
    (10, 1, ((31, 17), (16, 9)), 8, 256, 16, 9, "bf16"),
    (11, 2, ((12, 10), (6, 5)), 2, 128, 4, 65, "f32"),
    (12, 1, ((6, 6),), 2, 512, 3, 5, "f32"),
    (13, 1, ((6, 6),), 2, 512, 3, 5, "bf16"),
    (14, 1, tuple((3, 2) for _ in range(16)), 2, 8, 16, 6, "f32"),
    (15, 2, ((4, 5), (2, 3)), 3, 8, 128, 3, "f32"),
    (16, 2, ((4, 5), (2, 3)), 1, 8, 128, 40, "bf16"),
    # fp16 I/O (the Ascend page's half type)
    (17, 2, ((9, 7), (5, 4)), 2, 32, 4, 33, "f16"),
    (18, 1, ((31, 17), (16, 9)), 8, 256, 16, 9, "f16"),
    (19, 2, ((5, 3), (1, 1)), 3, 16, 2, 7, "f16"),
    (20, 1, ((6, 6),), 2, 512, 3, 5, "f16"),
    (21, 3, ((9, 7), (5, 4), (3, 2), (2, 1), (1, 1)), 5, 64, 5, 17, "f16"),
]


@pytest.mark.parametrize("case", RANDOM_CASES, ids=lambda c: f"seed{c[0]}-D{c[4]}-{c[7]}")
def test_random_shape_parity(B, case):
    seed, bs, shapes, M, D, P, Q, dtype = case
    wl = gen.random_workload(seed, bs, shapes, M, D, P, Q, dtype=dtype)
    inp = gen.make_inputs(wl)
    out, grads = _run(B, wl, inp)
    _check(wl, inp, out, grads)


def test_encoder_shape_fp16(B):
    """The encoder pyramid and sampling pattern in fp16 I/O (one image)."""
    wl = gen.WORKLOADS["encoder_f16"].with_(bs=1, seed=1016)
    inp = gen.make_inputs(wl)
    out, grads = _run(B, wl, inp)
    _check(wl, inp, out, grads)
    empty_cache()


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_int32_index_tensors_give_the_same_results(B, dtype):
    """spatial_shapes / level_start_index as int32 (MSDA_INDEX_INT32) select the
    same pixels: output and the per-sample gradients are bit-identical to the
    int64 call; grad_value (fp32 atomics) agrees within the gradient tolerance."""
    wl = gen.random_workload(33, 2, ((9, 7), (5, 4), (3, 3)), 2, 32, 4, 21, dtype=dtype)
    inp = gen.make_inputs(wl)
    d = to_device(inp, wl)
    a64 = (d["value"], d["spatial_shapes"], d["level_start_index"], d["sampling_locations"],
           d["attention_weights"])
    a32 = (d["value"], d["spatial_shapes"].int(), d["level_start_index"].int(),
           d["sampling_locations"], d["attention_weights"])
    o64, o32 = B.msda_forward(*a64), B.msda_forward(*a32)
    g64 = B.msda_backward(*a64, d["grad_output"])
    g32 = B.msda_backward(*a32, d["grad_output"])
    torch.cuda.synchronize()
    assert torch.equal(o64, o32)
    assert torch.equal(g64[1], g32[1]) and torch.equal(g64[2], g32[2])
    assert_grad_close(host(g32[0]), host(g64[0]), wl.dtype, "grad_value (int32 indices)")


def test_key_index_field_is_exact(B):
    """value[b,k,m,d] = k + 4096*m + 0.25*d at pixel centres of power-of-two maps,
    one-hot weights: the output is the flattened key, bit for bit."""
    shapes = ((64, 32), (32, 16), (16, 8), (8, 4))
    bs, M, D, P, Q = 2, 3, 16, 2, 57
    rng = np.random.default_rng(5)
    L = len(shapes)
    K = gen.num_keys(shapes)
    lsi = gen.level_start_index(shapes)
    value = (np.arange(K)[None, :, None, None] + 4096.0 * np.arange(M)[None, None, :, None]
             + 0.25 * np.arange(D)[None, None, None, :] + np.zeros((bs, 1, 1, 1)))
    value = value.astype(np.float32)
    loc = np.empty((bs, Q, M, L, P, 2), np.float32)
    keys = np.empty((bs, Q, M, L, P), np.int64)
    for l, (H, W) in enumerate(shapes):
        ix = rng.integers(0, W, size=(bs, Q, M, P))
        iy = rng.integers(0, H, size=(bs, Q, M, P))
        loc[:, :, :, l, :, 0] = (ix + 0.5) / W
        loc[:, :, :, l, :, 1] = (iy + 0.5) / H
        keys[:, :, :, l, :] = lsi[l] + iy * W + ix
    w = np.zeros((bs, Q, M, L, P), np.float32)
    pick_l = rng.integers(0, L, size=(bs, Q, M))
    pick_p = rng.integers(0, P, size=(bs, Q, M))
    bb, qq, mm = np.meshgrid(np.arange(bs), np.arange(Q), np.arange(M), indexing="ij")
    w[bb, qq, mm, pick_l, pick_p] = 1.0
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = B.msda_forward(dev(value), dev(np.array(shapes, np.int64)), dev(lsi), dev(loc), dev(w))
    got = out.cpu().numpy().reshape(bs, Q, M, D)
    k = keys[bb, qq, mm, pick_l, pick_p]
    want = (k[..., None] + 4096.0 * mm[..., None] + 0.25 * np.arange(D)).astype(np.float32)
    assert np.array_equal(got, want)


def test_out_of_range_and_empty_inputs(B):
    wl = gen.random_workload(21, 2, ((6, 10), (3, 5)), 2, 32, 4, 9)
    inp = gen.make_inputs(wl)
    inp["sampling_locations"][:] = np.float32(2.0)      # every sample off the map
    out, grads = _run(B, wl, inp)
    assert np.all(out == 0)
    assert all(np.all(g == 0) for g in grads)
    # empty problems: Q = 0, P = 0 and bs = 0 leave zero-sized or zero-filled outputs
    for kw in (dict(Q=0), dict(P=0), dict(bs=0)):
        bs = kw.get("bs", 2)
        Q = kw.get("Q", 5)
        P = kw.get("P", 3)
        shapes = ((4, 4), (2, 2))
        K = gen.num_keys(shapes)
        v = torch.randn(bs, K, 2, 16, device="cuda")
        loc = torch.rand(bs, Q, 2, 2, P, 2, device="cuda")
        w = torch.rand(bs, Q, 2, 2, P, device="cuda")
        g = torch.randn(bs, Q, 32, device="cuda")
        sh = torch.tensor(shapes, device="cuda")
        lsi = torch.from_numpy(gen.level_start_index(shapes)).cuda()
        out = torch.full((bs, Q, 32), 7.0, device="cuda")
        B.msda_forward(v, sh, lsi, loc, w, output=out)
        gv = torch.full_like(v, 3.0)
        gl = torch.full_like(loc, 3.0)
        gw = torch.full_like(w, 3.0)
        B.msda_backward(v, sh, lsi, loc, w, g, gv, gl, gw)
        torch.cuda.synchronize()
        assert torch.all(out == 0) and torch.all(gv == 0)
        assert torch.all(gl == 0) and torch.all(gw == 0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_no_value_rows_zero_fills_odd_sized_gradients(B, dtype):
    """head_dim 0 leaves nothing to read: every gradient, of any element count, is zeroed."""
    shapes = ((3, 3),)
    v = torch.ones(1, 9, 1, 0, device="cuda", dtype=dtype)
    loc = torch.rand(1, 3, 1, 1, 3, 2, device="cuda").to(dtype)   # 9 samples: odd sizes
    w = torch.rand(1, 3, 1, 1, 3, device="cuda").to(dtype)
    g = torch.ones(1, 3, 0, device="cuda", dtype=dtype)
    sh = torch.tensor(shapes, device="cuda")
    lsi = torch.tensor([0], device="cuda")
    gv = torch.empty_like(v)
    gl = torch.full_like(loc, 5.0)
    gw = torch.full_like(w, 5.0)
    B.msda_backward(v, sh, lsi, loc, w, g, gv, gl, gw)
    torch.cuda.synchronize()
    assert torch.all(gl == 0) and torch.all(gw == 0)


def test_inconsistent_level_is_skipped_and_reported(B):
    """A level whose pixels fall past num_keys contributes nothing and raises the
    device error word; the kernels read nothing outside value."""
    shapes = ((4, 4), (2, 2))
    K = gen.num_keys(shapes)
    v = torch.randn(1, K, 2, 16, device="cuda")
    loc = torch.rand(1, 5, 2, 2, 3, 2, device="cuda")
    w = torch.rand(1, 5, 2, 2, 3, device="cuda")
    sh = torch.tensor(shapes, device="cuda")
    good = torch.tensor([0, 16], device="cuda")
    bad = torch.tensor([0, 18], device="cuda")      # level 1 would end at key 22 > K = 20
    assert B.msda_last_device_error() == 0
    assert B.msda_check_shapes(sh, good, K) == 0
    assert B.msda_check_shapes(sh, bad, K) == 7
    out_bad = B.msda_forward(v, sh, bad, loc, w)
    assert B.msda_last_device_error() == 8
    assert B.msda_last_device_error() == 0          # cleared by the read
    # the consistent level still contributes exactly as with good indices and
    # level-1 weights zeroed
    w0 = w.clone()
    w0[:, :, :, 1] = 0
    out_ref = B.msda_forward(v, sh, good, loc, w0)
    torch.cuda.synchronize()
    assert torch.equal(out_bad, out_ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_grad_value_accumulate_flag(B, dtype):
    wl = gen.random_workload(31, 2, ((9, 7), (5, 4)), 2, 32, 3, 11, dtype=dtype)
    inp = gen.make_inputs(wl)
    d = to_device(inp, wl)
    args = (d["value"], d["spatial_shapes"], d["level_start_index"], d["sampling_locations"],
            d["attention_weights"], d["grad_output"])
    gv1, _, _ = B.msda_backward(*args)
    gv2 = gv1.clone()
    B.msda_backward(*args, grad_value=gv2, accumulate=True)
    torch.cuda.synchronize()
    rv = oracle.backward(inp["value"], inp["spatial_shapes"], inp["level_start_index"],
                         inp["sampling_locations"], inp["attention_weights"],
                         inp["grad_output"])[0]
    assert_grad_close(host(gv2), 2 * rv, wl.dtype, "accumulated grad_value")


def test_non_default_stream_and_zero_fill(B):
    wl = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(wl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = to_device(inp, wl)
        out = B.msda_forward(d["value"], d["spatial_shapes"], d["level_start_index"],
                             d["sampling_locations"], d["attention_weights"], stream=s)
        buf = torch.ones(1000, 8, device="cuda")
        B.msda_zero_fill(buf, stream=s)
    s.synchronize()
    assert torch.all(buf == 0)
    assert_out_close(host(out), oracle.run_inputs(inp, backward_pass=False)[0], "f32")


def test_autograd_wrapper_matches_direct_calls(B):
    wl = gen.random_workload(41, 2, ((9, 7), (5, 4)), 2, 32, 3, 11)
    inp = gen.make_inputs(wl)
    d = to_device(inp, wl)
    v = d["value"].clone().requires_grad_()
    loc = d["sampling_locations"].clone().requires_grad_()
    w = d["attention_weights"].clone().requires_grad_()
    out = B.MSDeformAttnFunction.apply(v, d["spatial_shapes"], d["level_start_index"], loc, w, 64)
    out.backward(d["grad_output"])
    gv, gl, gw = B.msda_backward(d["value"], d["spatial_shapes"], d["level_start_index"],
                                 d["sampling_locations"], d["attention_weights"],
                                 d["grad_output"])
    torch.cuda.synchronize()
    ref_out, (rv, rl, rw) = oracle.run_inputs(inp)
    assert_out_close(host(out), ref_out, "f32")
    assert_grad_close(host(v.grad), rv, "f32")
    assert_grad_close(host(loc.grad), rl, "f32")
    assert_grad_close(host(w.grad), rw, "f32")
    assert_grad_close(host(gl), rl, "f32")
