"""msda_backward_noalloc: the bf16 backward for callers that cannot allocate.

Some callers of this library may not allocate device memory themselves: a
host framework that owns every allocation, a plug-in with no access to the
allocator, or code that must not call cudaMalloc while work is being captured
or timed.  For them the library offers msda_backward_noalloc, which takes no
workspace and accumulates in a fixed scratch array of its own.  This test
calls it through the C ABI (the ctypes binding) twice in a row on the
decoder shape with different inputs, then on a smaller problem right after a
larger one, with the accumulate flag and with int32 index tensors, and checks
each result against the regular msda_backward with its caller-provided
workspace, within the bf16 gradient tolerance the parity tests use (max|err|
<= 1e-2 * max|ref|): the scratch left by one call does not leak into the next.
It also checks that NULL and misaligned gradient pointers are refused.

The file name makes pytest collect it last.
"""
import numpy as np
import pytest
import torch

from scale_deformable_attention_05_b300 import inputs as gen
from tests.gpu_helpers import assert_grad_close, host, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_05_b300 import binding
    return binding


def _decoder_bf16(seed):
    # decoder cross-attention shape in bf16: the fp32 accumulator (45.5 MB) fits
    # the fixed scratch array
    return gen.WORKLOADS["decoder"].with_(seed=seed, dtype="bf16")


def test_noalloc_backward_matches_regular_backward_twice(B):
    for seed in (2001, 2002):
        wl = _decoder_bf16(seed)
        d = to_device(gen.make_inputs(wl), wl)
        args = (d["value"], d["spatial_shapes"], d["level_start_index"],
                d["sampling_locations"], d["attention_weights"], d["grad_output"])
        ref = B.msda_backward(*args)
        got = tuple(torch.full_like(t, 3.0) for t in ref)
        B.msda_backward_noalloc(*args, *got)
        torch.cuda.synchronize()
        assert B.msda_last_device_error() == 0
        for name, g, r in zip(("grad_value", "grad_sampling_loc", "grad_attn_weight"), got, ref):
            assert_grad_close(host(g), host(r), "bf16", f"{name} (seed {seed})")
        assert torch.count_nonzero(got[0]) > 0


def test_noalloc_rejects_sizes_beyond_its_scratch(B):
    # bs*K*M*D fp32 accumulators above the fixed maximum: refused before any launch
    limit_elems = (64 << 20) // 4
    K = limit_elems // (8 * 32) + 1
    v = torch.zeros(1, K, 8, 32, device="cuda", dtype=torch.bfloat16)
    loc = torch.zeros(1, 2, 8, 1, 1, 2, device="cuda", dtype=torch.bfloat16)
    w = torch.zeros(1, 2, 8, 1, 1, device="cuda", dtype=torch.bfloat16)
    g = torch.zeros(1, 2, 256, device="cuda", dtype=torch.bfloat16)
    sh = torch.tensor([[1, K]], device="cuda")
    lsi = torch.tensor([0], device="cuda")
    with pytest.raises(B.MsdaError) as e:
        B.msda_backward_noalloc(v, sh, lsi, loc, w, g, torch.empty_like(v),
                                torch.empty_like(loc), torch.empty_like(w))
    assert e.value.status == 5
    # fp32 needs no workspace, so it has no allocation-free variant
    with pytest.raises(B.MsdaError) as e:
        f = lambda t: t.float()
        B.msda_backward_noalloc(f(v[:, :4]), torch.tensor([[1, 4]], device="cuda"), lsi,
                                f(loc), f(w), f(g), f(v[:, :4]), f(loc), f(w))
    assert e.value.status == 3


def test_noalloc_smaller_call_after_larger_accumulate_and_int32(B):
    """A smaller problem right after a larger one (the shared array still holds
    the larger call's sums beyond the part the smaller one clears), the
    accumulate flag, and int32 index tensors, each against msda_backward."""
    big = _decoder_bf16(2003)
    d = to_device(gen.make_inputs(big), big)
    args = (d["value"], d["spatial_shapes"], d["level_start_index"], d["sampling_locations"],
            d["attention_weights"], d["grad_output"])
    B.msda_backward_noalloc(*args, *(torch.empty_like(t) for t in
                                    (d["value"], d["sampling_locations"],
                                     d["attention_weights"])))
    small = gen.WORKLOADS["tiny"].with_(seed=2004, dtype="bf16")
    d = to_device(gen.make_inputs(small), small)
    args = (d["value"], d["spatial_shapes"], d["level_start_index"], d["sampling_locations"],
            d["attention_weights"], d["grad_output"])
    ref = B.msda_backward(*args)
    got = tuple(torch.full_like(t, 3.0) for t in ref)
    B.msda_backward_noalloc(*args, *got)
    torch.cuda.synchronize()
    for name, g, r in zip(("grad_value", "grad_sampling_loc", "grad_attn_weight"), got, ref):
        assert_grad_close(host(g), host(r), "bf16", f"{name} (smaller call)")

    # accumulate: both entry points add into the same starting grad_value
    base = torch.randn(d["value"].shape, generator=torch.Generator().manual_seed(7)).to(
        device="cuda", dtype=torch.bfloat16)
    want = B.msda_backward(*args, grad_value=base.clone(), accumulate=True)[0]
    got_v = base.clone()
    B.msda_backward_noalloc(*args, got_v, torch.empty_like(ref[1]), torch.empty_like(ref[2]),
                            accumulate=True)
    torch.cuda.synchronize()
    assert_grad_close(host(got_v), host(want), "bf16", "grad_value (accumulate)")

    # int32 index tensors give the int64 results
    args32 = args[:1] + (args[1].to(torch.int32), args[2].to(torch.int32)) + args[3:]
    got32 = tuple(torch.empty_like(t) for t in ref)
    B.msda_backward_noalloc(*args32, *got32)
    torch.cuda.synchronize()
    for name, g, r in zip(("grad_value", "grad_sampling_loc", "grad_attn_weight"), got32, ref):
        assert_grad_close(host(g), host(r), "bf16", f"{name} (int32 indices)")


def test_noalloc_rejects_null_and_misaligned_pointers(B):
    """Through the C ABI directly: a NULL gradient pointer and a gradient pointer
    off the 16-byte grid are refused before anything is enqueued."""
    wl = gen.WORKLOADS["tiny"].with_(seed=2005, dtype="bf16")
    d = to_device(gen.make_inputs(wl), wl)
    gv = torch.empty(d["value"].numel() + 8, dtype=torch.bfloat16, device="cuda")
    gl, gw = torch.empty_like(d["sampling_locations"]), torch.empty_like(d["attention_weights"])
    dims = (wl.bs, wl.num_keys, wl.num_heads, wl.head_dim, wl.num_levels, wl.num_points,
            wl.num_queries)
    P_ = lambda t: t.data_ptr()
    common = (P_(d["value"]), P_(d["spatial_shapes"]), P_(d["level_start_index"]),
              P_(d["sampling_locations"]), P_(d["attention_weights"]), P_(d["grad_output"]))
    lib = B._LIB
    assert lib.msda_backward_noalloc(*common, None, P_(gl), P_(gw), *dims, 1, 0, None) == 1
    assert lib.msda_backward_noalloc(*common, P_(gv) + 2, P_(gl), P_(gw), *dims, 1, 0, None) == 4
    assert lib.msda_backward_noalloc(*common, P_(gv), P_(gl), P_(gw), *dims, 1, 0, None) == 0
    torch.cuda.synchronize()
