"""GPU results of the fused entry points (msda_forward_fused / msda_backward_fused)
against the fused oracle (oracle/fused.py), through the C ABI, element by
element with the tolerances of the parity tests (tests/gpu_helpers.py).  The
locations select pixels in the same binary32 operations on both sides, so
which value rows receive gradient is compared exactly."""
import numpy as np
import pytest
import torch

from oracle import fused as ofused
from scale_deformable_attention_05_b300 import inputs as gen
from tests.gpu_helpers import TOL, assert_grad_close, assert_out_close, empty_cache, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from scale_deformable_attention_05_b300 import binding
    return binding


def _dev(inp, wl, name):
    if wl.dtype in ("bf16", "f16"):
        tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
        return torch.from_numpy(inp[name + "_" + wl.dtype].view(np.int16).copy()).view(tdt).cuda()
    return torch.from_numpy(np.ascontiguousarray(inp[name])).cuda()


def _mask_for(wl, kind):
    if kind is None:
        return None
    if kind == "detr":
        return gen.padding_mask(wl)                     # padded right / bottom per image
    rng = np.random.default_rng(wl.seed + 90000)
    return rng.random((wl.bs, wl.num_keys)) < 0.3      # scattered padded keys


def _run_and_check(B, wl, ref_dim, sigma=2.0, mask_kind=None):
    inp = gen.make_fused_inputs(wl, ref_dim, offset_sigma=sigma)
    mask = _mask_for(wl, mask_kind)
    names = ("value", "reference_points", "sampling_offsets", "attention_logits", "grad_output")
    d = {k: _dev(inp, wl, k) for k in names}
    sh = torch.from_numpy(inp["spatial_shapes"]).cuda()
    lsi = torch.from_numpy(inp["level_start_index"]).cuda()
    dmask = None if mask is None else torch.from_numpy(mask).cuda()
    args = (d["value"], sh, lsi, d["reference_points"], d["sampling_offsets"],
            d["attention_logits"])
    out = B.msda_forward_fused(*args, dmask)
    gv, goff, glog, gref = B.msda_backward_fused(*args, d["grad_output"], dmask)
    torch.cuda.synchronize()
    assert B.msda_last_device_error() == 0
    oargs = (inp["value"], inp["spatial_shapes"], inp["level_start_index"],
             inp["reference_points"], inp["sampling_offsets"], inp["attention_logits"])
    assert_out_close(host(out), ofused.forward(*oargs, padding_mask=mask), wl.dtype)
    rv, roff, rlog, rref = ofused.backward(*oargs, inp["grad_output"], padding_mask=mask)
    assert_grad_close(host(gv), rv, wl.dtype, "grad_value")
    assert_grad_close(host(goff), roff, wl.dtype, "grad_sampling_offsets")
    assert_grad_close(host(glog), rlog, wl.dtype, "grad_attn_logits")
    assert_grad_close(host(gref), rref, wl.dtype, "grad_reference_points")
    np.testing.assert_array_equal(np.any(host(gv) != 0, -1), np.any(rv != 0, -1))
    empty_cache()


CASES = [
    # (name, seed, bs, shapes, M, D, P, Q, dtype, ref_dim)
    ("one-level", 61, 1, ((12, 10),), 2, 32, 8, 9, "f32", 2),
    ("pyramid", 62, 2, ((9, 7), (5, 4), (3, 2), (2, 1)), 3, 32, 4, 17, "f32", 2),
    ("boxes", 63, 2, ((9, 7), (5, 4), (3, 2), (2, 1)), 3, 32, 4, 17, "f32", 4),
    ("wide-head", 64, 1, ((16, 12), (8, 6)), 2, 256, 16, 7, "f32", 4),
    ("lp64", 65, 1, ((10, 9), (5, 5), (3, 3), (2, 2)), 2, 64, 16, 5, "f32", 2),
    ("bf16", 66, 2, ((9, 7), (5, 4)), 2, 32, 8, 11, "bf16", 2),
    ("f16-boxes", 67, 2, ((9, 7), (5, 4)), 2, 64, 4, 11, "f16", 4),
    ("odd-points", 68, 1, ((7, 5), (4, 3), (2, 2)), 2, 16, 3, 13, "f32", 2),
    # 16-bit rows of 32 bytes in 4-lane groups of 8-byte vectors
    ("bf16-narrow", 69, 2, ((9, 7), (5, 4)), 3, 16, 4, 13, "bf16", 2),
    ("f16-narrow-boxes", 70, 1, ((8, 8), (4, 5)), 2, 16, 2, 9, "f16", 4),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_fused_random_shapes(B, case):
    _, seed, bs, shapes, M, D, P, Q, dtype, ref_dim = case
    wl = gen.random_workload(seed, bs, shapes, M, D, P, Q, dtype=dtype)
    _run_and_check(B, wl, ref_dim)


@pytest.mark.parametrize("ref_dim", [2, 4])
def test_fused_decoder_shape(B, ref_dim):
    _run_and_check(B, gen.WORKLOADS["decoder"], ref_dim)


def test_fused_encoder_shape(B):
    wl = gen.WORKLOADS["encoder"].with_(bs=1, seed=1007)
    _run_and_check(B, wl, 2, sigma=1.5)


EDGE_SHAPES = ((6, 7), (5, 21), (3, 167))          # widths with inexact reciprocals


def _cell(loc, W):
    """Cell column of a binary32 location: floor of fl(loc * W - 0.5) (one rounding)."""
    x = (np.asarray(loc, np.float64) * W - 0.5).astype(np.float32)
    return np.floor(x)


def _edge_case_inputs(ref_dim, seed=81, Q=4, M=2, P=3, D=32):
    """Fused inputs whose every sample lies on a cell edge in x, placed so that
    the module's expression with correctly rounded division (walk-through
    "2.2.4 源码分析": off / (W, H); "2.4": off / P * wh * 0.5) picks one cell and
    the same expression with once-rounded reciprocals picks its neighbour.  The
    bilinear derivative along x jumps between the two cells, so the offset
    gradient tells which form a kernel computed.  Returns the inputs and the
    reciprocal form's cells next to the division form's."""
    f = np.float32
    rng = np.random.default_rng(seed)
    L = len(EDGE_SHAPES)
    ref = np.empty((1, Q, L, ref_dim), f)
    off = np.zeros((1, Q, M, L, P, 2), f)
    cells_div = np.zeros((1, Q, M, L, P))
    cells_rec = np.zeros((1, Q, M, L, P))
    for q in range(Q):
        for l, (H, W) in enumerate(EDGE_SHAPES):
            ref[0, q, l, 1] = (rng.integers(0, H) + 0.5 + 0.3) / H       # mid-cell in y
            if ref_dim == 4:
                ref[0, q, l, 2:] = rng.choice([0.375, 0.6875, 0.9375], 2)
            wh = ref[0, q, l, 2] if ref_dim == 4 else f(1)
            hits = []
            for _ in range(200):            # a reference x that admits at least one edge
                rx = ref[0, q, l, 0] = rng.uniform(0.1, 0.9)
                rx = ref[0, q, l, 0]
                if ref_dim == 2:
                    form = lambda o: (f(rx + f(o / f(W))), f(rx + f(o * f(f(1) / f(W)))))
                    scale = float(W)
                else:
                    form = lambda o: (f(rx + f(f(f(o / f(P)) * wh) * f(0.5))),
                                      f(rx + f(f(o * wh) * f(f(1) / f(2 * P)))))
                    scale = 2.0 * P / float(wh)
                for n in range(1, W - 1):
                    o = f((float(n + 0.5) / W - float(rx)) * scale)
                    for _ in range(24):
                        o = np.nextafter(o, f(np.inf))
                        ld, lr = form(o)
                        if _cell(ld, W) != _cell(lr, W):
                            hits.append((o, _cell(ld, W), _cell(lr, W)))
                            break
                if hits:
                    break
            assert hits, "no edge sample found"
            for i, (m, p) in enumerate(np.ndindex(M, P)):
                o, cd, cr = hits[i % len(hits)]
                off[0, q, m, l, p, 0] = o
                cells_div[0, q, m, l, p] = cd
                cells_rec[0, q, m, l, p] = cr
    value = rng.standard_normal((1, gen.num_keys(EDGE_SHAPES), M, D)).astype(f)
    logits = rng.standard_normal((1, Q, M, L * P)).astype(f)
    g = rng.standard_normal((1, Q, M * D)).astype(f)
    inp = {"value": value, "spatial_shapes": np.array(EDGE_SHAPES, np.int64),
           "level_start_index": gen.level_start_index(EDGE_SHAPES), "reference_points": ref,
           "sampling_offsets": off, "attention_logits": logits, "grad_output": g}
    return inp, cells_div, cells_rec


@pytest.mark.parametrize("ref_dim", [2, 4])
def test_fused_locations_divide_on_cell_edges(B, ref_dim):
    """The kernels form locations with IEEE division, as the oracle does: on
    samples where a reciprocal product would land one cell over, the offset
    gradients still agree."""
    inp, cells_div, cells_rec = _edge_case_inputs(ref_dim)
    assert (cells_div != cells_rec).all()
    oargs = tuple(inp[k] for k in ("value", "spatial_shapes", "level_start_index",
                                   "reference_points", "sampling_offsets", "attention_logits"))
    t = lambda k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()
    args = (t("value"), t("spatial_shapes"), t("level_start_index"), t("reference_points"),
            t("sampling_offsets"), t("attention_logits"))
    out = B.msda_forward_fused(*args)
    gv, goff, glog, gref = B.msda_backward_fused(*args, t("grad_output"))
    torch.cuda.synchronize()
    assert_out_close(host(out), ofused.forward(*oargs), "f32")
    rv, roff, rlog, rref = ofused.backward(*oargs, inp["grad_output"])
    assert_grad_close(host(goff), roff, "f32", "grad_sampling_offsets")
    assert_grad_close(host(glog), rlog, "f32", "grad_attn_logits")
    assert_grad_close(host(gv), rv, "f32", "grad_value")
    np.testing.assert_array_equal(np.any(host(gv) != 0, -1), np.any(rv != 0, -1))
    empty_cache()


MASK_CASES = [
    ("pyramid-scattered", 71, 2, ((9, 7), (5, 4), (3, 2), (2, 1)), 3, 32, 4, 17, "f32", 2,
     "random"),
    ("boxes-detr", 72, 3, ((12, 10), (6, 5), (3, 3)), 2, 32, 4, 15, "f32", 4, "detr"),
    ("bf16-detr", 73, 2, ((9, 7), (5, 4)), 2, 32, 8, 11, "bf16", 2, "detr"),
    ("wide-head-scattered", 74, 2, ((16, 12), (8, 6)), 2, 256, 16, 7, "f32", 2, "random"),
]


@pytest.mark.parametrize("case", MASK_CASES, ids=lambda c: c[0])
def test_fused_padding_mask(B, case):
    _, seed, bs, shapes, M, D, P, Q, dtype, ref_dim, kind = case
    wl = gen.random_workload(seed, bs, shapes, M, D, P, Q, dtype=dtype)
    _run_and_check(B, wl, ref_dim, mask_kind=kind)


def test_fused_encoder_shape_padded_batch(B):
    """bs=2 encoder pyramid, image 1 padded (DETR-style valid region)."""
    wl = gen.WORKLOADS["encoder"].with_(seed=1008)
    _run_and_check(B, wl, 2, sigma=1.5, mask_kind="detr")


def test_fused_padding_mask_accumulate_leaves_padded_rows(B):
    wl = gen.random_workload(75, 2, ((9, 7), (5, 4)), 2, 32, 4, 13)
    inp = gen.make_fused_inputs(wl, 2)
    mask = _mask_for(wl, "random")
    t = lambda k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()
    sh = torch.from_numpy(inp["spatial_shapes"]).cuda()
    lsi = torch.from_numpy(inp["level_start_index"]).cuda()
    args = (t("value"), sh, lsi, t("reference_points"), t("sampling_offsets"),
            t("attention_logits"), t("grad_output"), torch.from_numpy(mask).cuda())
    base = torch.randn(t("value").shape, generator=torch.Generator().manual_seed(5)).cuda()
    gv = base.clone()
    B.msda_backward_fused(*args, grad_value=gv, accumulate=True)
    torch.cuda.synchronize()
    gv, base = host(gv), host(base)
    np.testing.assert_array_equal(gv[mask], base[mask])         # padded rows untouched
    rv = ofused.backward(*[inp[k] for k in ("value", "spatial_shapes", "level_start_index",
                                            "reference_points", "sampling_offsets",
                                            "attention_logits", "grad_output")],
                         padding_mask=mask)[0]
    assert_grad_close(gv - base, rv, "f32", "grad_value")


def test_fused_autograd_wrapper(B):
    wl = gen.random_workload(69, 2, ((9, 7), (5, 4)), 2, 32, 4, 9)
    inp = gen.make_fused_inputs(wl, 2)
    t = lambda k, rg=False: torch.tensor(inp[k], device="cuda", requires_grad=rg)
    v, ref, off, lg = t("value", True), t("reference_points", True), t("sampling_offsets", True), \
        t("attention_logits", True)
    sh = torch.from_numpy(inp["spatial_shapes"]).cuda()
    lsi = torch.from_numpy(inp["level_start_index"]).cuda()
    out = B.ms_deform_attn_fused(v, sh, lsi, ref, off, lg)
    out.backward(t("grad_output"))
    oargs = (inp["value"], inp["spatial_shapes"], inp["level_start_index"],
             inp["reference_points"], inp["sampling_offsets"], inp["attention_logits"])
    rv, roff, rlog, rref = ofused.backward(*oargs, inp["grad_output"])
    for got, want in ((v.grad, rv), (off.grad, roff), (lg.grad, rlog), (ref.grad, rref)):
        assert_grad_close(host(got), want, "f32")


def _fused_tensors(wl, ref_dim=2, mask=None, index=torch.int64):
    inp = gen.make_fused_inputs(wl, ref_dim)
    t = lambda k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()
    sh = torch.from_numpy(inp["spatial_shapes"]).to(index).cuda()
    lsi = torch.from_numpy(inp["level_start_index"]).to(index).cuda()
    args = (t("value"), sh, lsi, t("reference_points"), t("sampling_offsets"),
            t("attention_logits"))
    dmask = None if mask is None else torch.from_numpy(mask).cuda()
    return inp, args, t("grad_output"), dmask


def test_fused_int32_index_tensors_match_int64(B):
    wl = gen.random_workload(76, 2, ((9, 7), (5, 4), (3, 2)), 2, 32, 4, 13)
    mask = _mask_for(wl, "random")
    res = []
    for index in (torch.int64, torch.int32):
        _, args, g, dmask = _fused_tensors(wl, 4, mask, index)
        out = B.msda_forward_fused(*args, dmask)
        grads = B.msda_backward_fused(*args, g, dmask)
        torch.cuda.synchronize()
        res.append([host(out)] + [host(x) for x in grads])
    (o64, gv64, goff64, glog64, gref64), (o32, gv32, goff32, glog32, gref32) = res
    # per-sample results are computed identically; grad_value and the reference
    # gradient are sums by atomics, whose order may differ between launches
    np.testing.assert_array_equal(o32, o64)
    np.testing.assert_array_equal(goff32, goff64)
    np.testing.assert_array_equal(glog32, glog64)
    assert_grad_close(gv32, gv64, "f32", "grad_value")
    assert_grad_close(gref32, gref64, "f32", "grad_reference_points")


def test_fused_every_key_padded_gives_zeros(B):
    wl = gen.random_workload(77, 2, ((9, 7), (5, 4)), 2, 32, 4, 9)
    mask = np.ones((wl.bs, wl.num_keys), dtype=bool)
    _, args, g, dmask = _fused_tensors(wl, 2, mask)
    gv0 = torch.full_like(args[0], 3.0)
    out = B.msda_forward_fused(*args, dmask)
    gv, goff, glog, gref = B.msda_backward_fused(*args, g, dmask, grad_value=gv0,
                                                 accumulate=True)
    torch.cuda.synchronize()
    assert not host(out).any()
    assert (host(gv) == 3.0).all()                     # nothing added to padded rows
    assert not host(goff).any() and not host(glog).any() and not host(gref).any()


def test_fused_offsets_off_the_map_give_zeros(B):
    wl = gen.random_workload(78, 1, ((9, 7), (5, 4)), 2, 16, 4, 6)
    _, args, g, _ = _fused_tensors(wl, 2)
    off = torch.full_like(args[4], 1.0e4)               # every sample far outside every level
    args = args[:4] + (off,) + args[5:]
    out = B.msda_forward_fused(*args)
    gv, goff, glog, gref = B.msda_backward_fused(*args, g)
    torch.cuda.synchronize()
    for x in (out, gv, goff, glog, gref):
        assert not host(x).any()


def test_fused_no_queries(B):
    wl = gen.random_workload(79, 2, ((9, 7), (5, 4)), 2, 32, 4, 5)
    _, args, g, _ = _fused_tensors(wl, 2)
    cut = lambda x: x[:, :0].contiguous()
    args0 = args[:3] + tuple(cut(x) for x in args[3:])
    out = B.msda_forward_fused(*args0)
    gv, goff, glog, gref = B.msda_backward_fused(*args0, cut(g))
    torch.cuda.synchronize()
    assert out.shape == (wl.bs, 0, wl.num_heads * wl.head_dim)
    assert not host(gv).any() and goff.numel() == 0 and glog.numel() == 0 and gref.numel() == 0


def test_fused_f16_with_mask(B):
    wl = gen.random_workload(80, 2, ((9, 7), (5, 4)), 2, 64, 4, 11, dtype="f16")
    _run_and_check(B, wl, 4, mask_kind="detr")


def _sweep_cases(n=12, seed=20260):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        L = int(rng.integers(1, 5))
        P = int(rng.integers(1, 64 // L + 1))
        shapes = tuple((int(rng.integers(1, 10)), int(rng.integers(1, 10))) for _ in range(L))
        cases.append(dict(seed=300 + i, bs=int(rng.integers(1, 3)), shapes=shapes,
                          M=int(rng.integers(1, 4)), D=int(rng.choice([8, 16, 32, 40, 64, 128])),
                          P=P, Q=int(rng.integers(1, 20)),
                          dtype=str(rng.choice(["f32", "bf16", "f16"])),
                          ref_dim=int(rng.choice([2, 4])),
                          mask=[None, "random", "detr"][int(rng.integers(0, 3))],
                          idx32=bool(rng.integers(0, 2))))
    return cases


@pytest.mark.parametrize("c", _sweep_cases(), ids=lambda c: f"seed{c['seed']}")
def test_fused_random_sweep(B, c):
    """Seeded sweep over levels, points (L*P <= 64), head_dim, heads, dtype,
    reference width, padding mask and index width."""
    wl = gen.random_workload(c["seed"], c["bs"], c["shapes"], c["M"], c["D"], c["P"], c["Q"],
                             dtype=c["dtype"])
    inp = gen.make_fused_inputs(wl, c["ref_dim"])
    mask = _mask_for(wl, c["mask"])
    names = ("value", "reference_points", "sampling_offsets", "attention_logits", "grad_output")
    d = {k: _dev(inp, wl, k) for k in names}
    index = torch.int32 if c["idx32"] else torch.int64
    sh = torch.from_numpy(inp["spatial_shapes"]).to(index).cuda()
    lsi = torch.from_numpy(inp["level_start_index"]).to(index).cuda()
    dmask = None if mask is None else torch.from_numpy(mask).cuda()
    args = (d["value"], sh, lsi, d["reference_points"], d["sampling_offsets"],
            d["attention_logits"])
    out = B.msda_forward_fused(*args, dmask)
    gv, goff, glog, gref = B.msda_backward_fused(*args, d["grad_output"], dmask)
    torch.cuda.synchronize()
    assert B.msda_last_device_error() == 0
    oargs = (inp["value"], inp["spatial_shapes"], inp["level_start_index"],
             inp["reference_points"], inp["sampling_offsets"], inp["attention_logits"])
    assert_out_close(host(out), ofused.forward(*oargs, padding_mask=mask), wl.dtype)
    rv, roff, rlog, rref = ofused.backward(*oargs, inp["grad_output"], padding_mask=mask)
    assert_grad_close(host(gv), rv, wl.dtype, "grad_value")
    assert_grad_close(host(goff), roff, wl.dtype, "grad_sampling_offsets")
    assert_grad_close(host(glog), rlog, wl.dtype, "grad_attn_logits")
    assert_grad_close(host(gref), rref, wl.dtype, "grad_reference_points")
    np.testing.assert_array_equal(np.any(host(gv) != 0, -1), np.any(rv != 0, -1))
