"""The library's calls can be captured into a CUDA graph and replayed: every
launch goes to the caller's stream, nothing is allocated or synchronised
inside a call.  A replay must give the eager call's results (the forward bit
for bit; the backward up to the order of its atomic adds)."""
import numpy as np
import pytest
import torch

from scale_deformable_attention_05_b300 import inputs as gen
from tests.gpu_helpers import assert_grad_close, host

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,fused", [("f32", False), ("bf16", False), ("f32", True)])
def test_graph_replay_matches_eager(dtype, fused):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_05_b300 import binding as B
    wl = gen.random_workload(91, 2, ((12, 10), (6, 5), (3, 3)), 2, 32, 4, 23, dtype=dtype)
    inp = gen.make_fused_inputs(wl, 2) if fused else gen.make_inputs(wl)
    names = (("value", "reference_points", "sampling_offsets", "attention_logits", "grad_output")
             if fused else ("value", "sampling_locations", "attention_weights", "grad_output"))

    def dev(k):
        if dtype == "bf16":
            return torch.from_numpy(inp[k + "_bf16"].view(np.int16).copy()).view(
                torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()

    d = {k: dev(k) for k in names}
    sh = torch.from_numpy(inp["spatial_shapes"]).cuda()
    lsi = torch.from_numpy(inp["level_start_index"]).cuda()
    args = (d["value"], sh, lsi) + tuple(d[k] for k in names[1:-1])
    out = torch.empty(wl.bs, wl.num_queries, wl.num_heads * wl.head_dim, dtype=d["value"].dtype,
                      device="cuda")
    gv = torch.empty_like(d["value"])
    gl, gw = torch.empty_like(d[names[-3]]), torch.empty_like(d[names[-2]])
    code = {"f32": B.MSDA_F32, "bf16": B.MSDA_BF16}[dtype]
    ws = torch.empty(max(16, B.msda_backward_workspace_bytes(wl.bs, wl.num_keys, wl.num_heads,
                                                             wl.head_dim, code)),
                     dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()

    def step():
        if fused:
            B.msda_forward_fused(*args, output=out, stream=side)
            B.msda_backward_fused(*args, d["grad_output"], grad_value=gv,
                                  grad_sampling_offsets=gl, grad_attn_logits=gw,
                                  reference_grad=False, workspace=ws, stream=side)
        else:
            B.msda_forward(*args, output=out, stream=side)
            B.msda_backward(*args, d["grad_output"], gv, gl, gw, workspace=ws, stream=side)

    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        step()                                           # eager (also warms up the library)
    torch.cuda.synchronize()
    eager = [host(x) for x in (out, gv, gl, gw)]
    for x in (out, gv, gl, gw):
        x.fill_(7.0)                                     # the replay must overwrite everything
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step()
    graph.replay()
    torch.cuda.synchronize()
    assert B.msda_last_device_error() == 0
    got = [host(x) for x in (out, gv, gl, gw)]
    np.testing.assert_array_equal(got[0], eager[0])
    np.testing.assert_array_equal(got[2], eager[2])
    np.testing.assert_array_equal(got[3], eager[3])
    assert_grad_close(got[1], eager[1], dtype, "grad_value")
