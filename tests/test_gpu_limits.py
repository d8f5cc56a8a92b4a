"""The operator at the limits of the interface.

* A value tensor of 2.68e9 elements (10.7 GB fp32; byte offsets past 8 GB):
  samples at pixel centres with weight 1 must return their value row exactly,
  and the backward must put exactly a * g into that row of grad_value and the
  exact dot product into grad_attn.  The value field is a small-integer
  pattern, so every expected number is an exact fp32 integer (a closed form,
  no oracle call at this size).
* 16 levels, 16 points per level (L*P = 256) at head_dim 8 and 512, against
  the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from scale_deformable_attention_05_b300 import inputs as gen
from tests.gpu_helpers import assert_grad_close, assert_out_close, empty_cache, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_05_b300 import binding
    return binding


def _pattern(keys, m, d, b):
    """value[b, k, m, d] = (7k + 3m + d + 11b) mod 4093, exact in fp32."""
    return (7 * keys + 3 * m + d + 11 * b) % 4093


def test_value_beyond_two_to_the_31_elements(B):
    bs, H, W, M, D = 2, 2048, 2048, 8, 40
    K = H * W
    assert bs * K * M * D > 2 ** 31
    dev = torch.device("cuda")
    value = torch.empty((bs, K, M, D), dtype=torch.float32, device=dev)
    mm = torch.arange(M, dtype=torch.int32, device=dev).view(1, M, 1)
    dd = torch.arange(D, dtype=torch.int32, device=dev).view(1, 1, D)
    chunk = 1 << 19
    for b in range(bs):
        for k0 in range(0, K, chunk):
            kk = torch.arange(k0, min(K, k0 + chunk), dtype=torch.int32, device=dev).view(-1, 1, 1)
            value[b, k0:k0 + kk.shape[0]] = _pattern(kk, mm, dd, b).to(torch.float32)
    # 24 queries per image on distinct pixels, half of them in the last rows (largest offsets)
    rng = np.random.default_rng(5)
    Q = 24
    xs = rng.choice(W, size=(bs, Q), replace=False)
    ys = np.concatenate([rng.integers(0, 8, (bs, Q // 2)), rng.integers(H - 8, H, (bs, Q // 2))], 1)
    loc = np.empty((bs, Q, M, 1, 1, 2), np.float32)
    loc[..., 0] = ((xs + 0.5) / W)[:, :, None, None, None]       # exact: W is a power of two
    loc[..., 1] = ((ys + 0.5) / H)[:, :, None, None, None]
    attn = np.ones((bs, Q, M, 1, 1), np.float32)
    g = rng.integers(-3, 4, (bs, Q, M * D)).astype(np.float32)
    shapes = torch.tensor([[H, W]], device=dev)
    lsi = torch.tensor([0], device=dev)
    tloc, tattn, tg = (torch.from_numpy(a).to(dev) for a in (loc, attn, g))
    out = B.msda_forward(value, shapes, lsi, tloc, tattn)
    gv = torch.empty_like(value)
    _, gl, gw = B.msda_backward(value, shapes, lsi, tloc, tattn, tg, grad_value=gv)
    torch.cuda.synchronize()
    assert B.msda_last_device_error() == 0
    keys = ys * W + xs                                            # [bs, Q]
    m_ = np.arange(M)[None, None, :, None]
    d_ = np.arange(D)[None, None, None, :]
    b_ = np.arange(bs)[:, None, None, None]
    want = _pattern(keys[:, :, None, None], m_, d_, b_).astype(np.float64)   # [bs, Q, M, D]
    np.testing.assert_array_equal(host(out).reshape(bs, Q, M, D), want)
    # grad_value: exactly g in the sampled rows, nothing in their neighbours
    bidx = torch.arange(bs, device=dev).view(bs, 1).expand(bs, Q)
    kidx = torch.from_numpy(keys).to(dev)
    np.testing.assert_array_equal(host(gv[bidx, kidx]), g.reshape(bs, Q, M, D))
    # ... and nowhere else: the other corners of a pixel-centre sample weigh 0 and send nothing
    assert int(torch.count_nonzero(gv)) == int(np.count_nonzero(g))
    assert float(gv.sum()) == float(g.sum())                     # small integers: exact in any order
    # grad_attn = sum_d g_d v_d, a sum of small-integer products (exact in fp32)
    np.testing.assert_array_equal(host(gw).reshape(bs, Q, M),
                                  (g.reshape(bs, Q, M, D) * want).sum(-1))
    assert np.isfinite(host(gl)).all()
    del value, gv
    empty_cache()


@pytest.mark.parametrize("D", [8, 512])
def test_sixteen_levels_and_256_points(B, D):
    shapes = ((6, 5), (5, 4), (4, 4), (4, 3), (3, 3), (3, 2), (2, 3), (2, 2),
              (2, 1), (1, 2), (1, 1), (3, 1), (1, 3), (2, 4), (4, 2), (1, 1))
    assert len(shapes) == 16
    wl = gen.random_workload(95 + D, 1, shapes, 1, D, 16, 5)
    inp = gen.make_inputs(wl)
    dev = {k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()
           for k in ("value", "spatial_shapes", "level_start_index", "sampling_locations",
                     "attention_weights", "grad_output")}
    args = (dev["value"], dev["spatial_shapes"], dev["level_start_index"],
            dev["sampling_locations"], dev["attention_weights"])
    out = B.msda_forward(*args)
    gv, gl, gw = B.msda_backward(*args, dev["grad_output"])
    torch.cuda.synchronize()
    assert B.msda_last_device_error() == 0
    ref_out, (rv, rl, rw) = oracle.run_inputs(inp)
    assert_out_close(host(out), ref_out, "f32")
    assert_grad_close(host(gv), rv, "f32", "grad_value")
    assert_grad_close(host(gl), rl, "f32", "grad_sampling_loc")
    assert_grad_close(host(gw), rw, "f32", "grad_attn_weight")
