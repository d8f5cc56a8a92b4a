"""The MSDeformAttn layer (projections + fused operator) against an fp64
composition of the same steps: numpy matmuls for the four projections around
the fused oracle (oracle/fused.py), forward and every gradient.

The sampling-offset projection has zero weight (the layer's initial state), so
the offsets are its bias exactly on both sides and both select the same
pixels; the other projections are seeded random.  Tolerance: the fp32 grad
rule, max|err| <= 1e-4 * max|ref|, for the output too -- it passes through
three fp32 GEMMs of depth d_model before and after the operator."""
import numpy as np
import pytest
import torch

from oracle import fused as ofused
from scale_deformable_attention_05_b300 import inputs as gen
from tests.gpu_helpers import assert_grad_close, host

pytestmark = pytest.mark.gpu

TOL = 1e-4


def _oracle(params, q, x, ref, shapes, lsi, mask, g, M, L, P):
    """fp64 forward and gradients of output_proj(msda(value_proj(x), ...))."""
    Wv, bv, Wo, bo, Wa, ba, Wout, bout = (params[k] for k in (
        "value_proj.weight", "value_proj.bias", "sampling_offsets.weight", "sampling_offsets.bias",
        "attention_weights.weight", "attention_weights.bias", "output_proj.weight",
        "output_proj.bias"))
    N, Q, C = q.shape
    K = x.shape[1]
    value = (x @ Wv.T + bv).reshape(N, K, M, C // M)
    off = (q @ Wo.T + bo).reshape(N, Q, M, L, P, 2)
    logits = (q @ Wa.T + ba).reshape(N, Q, M, L * P)
    y = ofused.forward(value, shapes, lsi, ref, off.astype(np.float32), logits,
                       padding_mask=mask)
    out = y @ Wout.T + bout
    gy = g @ Wout
    gv, goff, glog, gref = ofused.backward(value, shapes, lsi, ref, off.astype(np.float32),
                                           logits, gy, padding_mask=mask)
    gv, goff, glog = gv.reshape(N, K, C), goff.reshape(N, Q, -1), glog.reshape(N, Q, -1)
    flat = lambda a: a.reshape(-1, a.shape[-1])
    grads = {
        "output_proj.weight": flat(g).T @ flat(y), "output_proj.bias": flat(g).sum(0),
        "value_proj.weight": flat(gv).T @ flat(x), "value_proj.bias": flat(gv).sum(0),
        "sampling_offsets.weight": flat(goff).T @ flat(q), "sampling_offsets.bias": flat(goff).sum(0),
        "attention_weights.weight": flat(glog).T @ flat(q),
        "attention_weights.bias": flat(glog).sum(0),
        "query": goff @ Wo + glog @ Wa, "input_flatten": gv @ Wv, "reference_points": gref,
    }
    return out, grads


@pytest.mark.parametrize("ref_dim,masked", [(2, True), (4, False)])
def test_module_matches_fp64_composition(ref_dim, masked):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_05_b300.module import MSDeformAttn
    torch.backends.cuda.matmul.allow_tf32 = False
    shapes = ((10, 12), (5, 6), (3, 3))
    C, M, L, P, N, Q = 64, 4, len(shapes), 4, 2, 9
    wl = gen.random_workload(81 + ref_dim, N, shapes, M, C // M, P, Q)
    K = wl.num_keys
    rng = np.random.default_rng(wl.seed)
    layer = MSDeformAttn(C, L, M, P).cuda()
    params = {}
    with torch.no_grad():
        for name, p in layer.named_parameters():
            if name == "sampling_offsets.weight":
                a = np.zeros(tuple(p.shape))
            elif name == "sampling_offsets.bias":
                a = rng.normal(0.0, 2.0, tuple(p.shape))
            else:
                a = rng.normal(0.0, 1.0 / np.sqrt(C), tuple(p.shape))
            a = a.astype(np.float32)
            p.copy_(torch.from_numpy(a))
            params[name] = a.astype(np.float64)
    q = rng.standard_normal((N, Q, C)).astype(np.float32)
    x = rng.standard_normal((N, K, C)).astype(np.float32)
    ref = rng.uniform(0.1, 0.9, (N, Q, L, 2))
    if ref_dim == 4:
        ref = np.concatenate([ref, rng.uniform(0.1, 0.5, (N, Q, L, 2))], -1)
    ref = ref.astype(np.float32)
    g = rng.standard_normal((N, Q, C)).astype(np.float32)
    mask = gen.padding_mask(wl, min_ratio=0.5) if masked else None
    sh = torch.tensor(shapes, dtype=torch.int64, device="cuda")
    lsi = torch.from_numpy(gen.level_start_index(shapes)).cuda()
    tq, tx, tref = (torch.tensor(a, device="cuda", requires_grad=True) for a in (q, x, ref))
    tmask = None if mask is None else torch.from_numpy(mask).cuda()
    out = layer(tq, tref, tx, sh, lsi, tmask)
    out.backward(torch.from_numpy(g).cuda())
    torch.cuda.synchronize()
    want, grads = _oracle(params, q.astype(np.float64), x.astype(np.float64), ref,
                          np.array(shapes), gen.level_start_index(shapes), mask,
                          g.astype(np.float64), M, L, P)
    assert_grad_close(host(out), want, "f32", "output")
    got = {n: p.grad for n, p in layer.named_parameters()}
    got.update(query=tq.grad, input_flatten=tx.grad, reference_points=tref.grad)
    for name, ref_grad in grads.items():
        assert_grad_close(host(got[name]), ref_grad, "f32", name)
    if mask is not None:                       # padded keys pass no gradient to the input
        assert not host(tx.grad)[mask].any()


def _round(a, dtype):
    """Round to bf16 or fp16 (round to nearest even) and widen back to fp64, on the CPU."""
    return torch.from_numpy(np.asarray(a, np.float64)).to(dtype).double().numpy()


def _assert_close(got, ref, tol, what):
    scale = float(np.abs(ref).max())
    err = float(np.abs(got - ref).max())
    assert err <= tol * scale, f"{what}: max|err| {err:.3e} > {tol} * max|ref| ({scale:.3e})"


@pytest.mark.parametrize("dtype,tol", [
    (torch.bfloat16, 1e-2),     # the bf16 gradient rule
    (torch.float16, 4e-3),      # eight fp16 unit roundoffs: the layer stores value, offsets,
                                # logits, the operator's output and every gradient in fp16
])
def test_half_module_on_tensor_cores_matches_fp64_composition(dtype, tol):
    """The layer in bf16 / fp16: its four projections run on the tensor-core
    kernel (msda_linear) forward, and for the input gradients backward; bias
    gradients on msda_linear_bias_grad.  Reference: the fp64 composition, with
    the layer's stored intermediates (value, offsets, logits, the operator's
    output) rounded to the layer's dtype where the layer stores them."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_05_b300.module import MSDeformAttn
    r = lambda a: _round(a, dtype)
    shapes = ((10, 12), (5, 6))
    C, M, L, P, N, Q = 128, 4, len(shapes), 4, 2, 9      # offsets 64 and logits 32 wide
    wl = gen.random_workload(91, N, shapes, M, C // M, P, Q,
                             dtype="bf16" if dtype == torch.bfloat16 else "f16")
    K = wl.num_keys
    rng = np.random.default_rng(wl.seed)
    layer = MSDeformAttn(C, L, M, P).cuda().to(dtype)
    params = {}
    with torch.no_grad():
        for name, p in layer.named_parameters():
            if name == "sampling_offsets.weight":
                a = np.zeros(tuple(p.shape))
            elif name == "sampling_offsets.bias":
                a = rng.normal(0.0, 2.0, tuple(p.shape))
            else:
                a = rng.normal(0.0, 1.0 / np.sqrt(C), tuple(p.shape))
            a = r(a)
            p.copy_(torch.from_numpy(a))
            params[name] = a
    q, x = r(rng.standard_normal((N, Q, C))), r(rng.standard_normal((N, K, C)))
    ref = r(rng.uniform(0.1, 0.9, (N, Q, L, 2)))
    g = r(rng.standard_normal((N, Q, C)))
    sh = torch.tensor(shapes, dtype=torch.int64, device="cuda")
    lsi = torch.from_numpy(gen.level_start_index(shapes)).cuda()
    tq, tx, tref = (torch.tensor(a, device="cuda", dtype=dtype, requires_grad=True)
                    for a in (q, x, ref))
    out = layer(tq, tref, tx, sh, lsi)
    out.backward(torch.from_numpy(g).to(device="cuda", dtype=dtype))
    torch.cuda.synchronize()

    Wv, bv, Wo, bo, Wa, ba, Wout, bout = (params[k] for k in (
        "value_proj.weight", "value_proj.bias", "sampling_offsets.weight", "sampling_offsets.bias",
        "attention_weights.weight", "attention_weights.bias", "output_proj.weight",
        "output_proj.bias"))
    value = r(x @ Wv.T + bv).reshape(N, K, M, C // M)
    off = r(q @ Wo.T + bo).reshape(N, Q, M, L, P, 2)
    logits = r(q @ Wa.T + ba).reshape(N, Q, M, L * P)
    shp, lsin = np.array(shapes), gen.level_start_index(shapes)
    y = r(ofused.forward(value, shp, lsin, ref, off.astype(np.float32), logits))
    want = y @ Wout.T + bout
    _assert_close(host(out), want, tol, "output")
    gy = g @ Wout
    gv, goff, glog, gref = ofused.backward(value, shp, lsin, ref, off.astype(np.float32), logits,
                                           gy)
    gv, goff, glog = gv.reshape(N, K, C), goff.reshape(N, Q, -1), glog.reshape(N, Q, -1)
    flat = lambda a: a.reshape(-1, a.shape[-1])
    grads = {
        "output_proj.weight": flat(g).T @ flat(y), "output_proj.bias": flat(g).sum(0),
        "value_proj.weight": flat(gv).T @ flat(x), "value_proj.bias": flat(gv).sum(0),
        "sampling_offsets.weight": flat(goff).T @ flat(q),
        "sampling_offsets.bias": flat(goff).sum(0),
        "attention_weights.weight": flat(glog).T @ flat(q),
        "attention_weights.bias": flat(glog).sum(0),
        "query": goff @ Wo + glog @ Wa, "input_flatten": gv @ Wv, "reference_points": gref,
    }
    got = {n: p.grad for n, p in layer.named_parameters()}
    got.update(query=tq.grad, input_flatten=tx.grad, reference_points=tref.grad)
    for name, ref_grad in grads.items():
        _assert_close(host(got[name]), ref_grad, tol, name)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_module_step_replays_as_one_cuda_graph(dtype):
    """Forward + backward of the layer captured as one CUDA graph (every entry
    point on the caller's stream, no host synchronisation, workspaces from the
    caller's allocator) and replayed: output and gradients equal the eager
    step's up to the order of the backward's atomic sums."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_05_b300.module import MSDeformAttn
    torch.backends.cuda.matmul.allow_tf32 = False
    shapes = ((16, 20), (8, 10))
    C, M, L, P, N, Q = 128, 4, len(shapes), 4, 2, 300
    wl = gen.random_workload(5, N, shapes, M, C // M, P, Q)
    g = torch.Generator().manual_seed(5)
    layer = MSDeformAttn(C, L, M, P).cuda().to(dtype)
    q = torch.randn(N, Q, C, generator=g).cuda().to(dtype).requires_grad_()
    x = torch.randn(N, wl.num_keys, C, generator=g).cuda().to(dtype).requires_grad_()
    go = torch.randn(N, Q, C, generator=g).cuda().to(dtype)
    ref = torch.rand(N, Q, L, 2, generator=g).cuda().to(dtype)
    sh = torch.tensor(shapes, dtype=torch.int64, device="cuda")
    lsi = torch.from_numpy(gen.level_start_index(shapes)).cuda()

    def run():
        out = layer(q, ref, x, sh, lsi)
        out.backward(go)
        return out

    def clear():
        for p in layer.parameters():
            p.grad = None
        q.grad = x.grad = None

    def grads():
        d = {n: p.grad.detach().clone() for n, p in layer.named_parameters()}
        d.update(query=q.grad.detach().clone(), input_flatten=x.grad.detach().clone())
        return d

    clear()
    want_out = run().detach().clone()
    want = grads()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            clear()
            run()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    clear()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        static_out = run()
    q.grad.zero_()                      # replays must rewrite, not accumulate
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    got = grads()
    tol = 1e-5 if dtype == torch.float32 else 1e-2
    scale = lambda t: t.float().abs().max().item() + 1e-30
    assert (static_out.float() - want_out.float()).abs().max().item() <= tol * scale(want_out)
    for name, w in want.items():
        assert (got[name].float() - w.float()).abs().max().item() <= tol * scale(w), name
