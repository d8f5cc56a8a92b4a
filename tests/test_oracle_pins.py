"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each expected value comes from
a closed form, an invariant, a value the pages print, a brute-force
formulation that shares no step with the oracle (tent sums over all pixels),
or the pages' own library formulation (torch grid_sample in fp64).
"""
import numpy as np
import pytest

import oracle
from oracle import grid_sample_ref, tent
from scale_deformable_attention_05_b300 import inputs as gen
from tests.conftest import parse_shapes, read_golden

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _problem(shapes, bs=1, M=2, D=8, P=3, Q=5, seed=0, loc_range=(-0.2, 1.2)):
    wl = gen.random_workload(seed, bs, shapes, M, D, P, Q, loc_range=loc_range)
    return wl, gen.make_inputs(wl)


def _args(inp):
    return (inp["value"], inp["spatial_shapes"], inp["level_start_index"],
            inp["sampling_locations"], inp["attention_weights"])


# ---------------------------------------------------------------- layout pins

def test_level_start_index_matches_printed_example():
    g = read_golden("level_start_index.txt")
    shapes = parse_shapes(g["shapes"])
    lsi = gen.level_start_index(shapes)
    assert lsi.tolist() == [int(t) for t in g["level_start_index"].split()]
    assert gen.num_keys(shapes) == int(g["num_keys"])


def test_ascend_example_bookkeeping():
    g = read_golden("ascend_example.txt")
    shapes = parse_shapes(g["shapes"])
    assert gen.num_keys(shapes) == int(g["num_keys"])
    assert gen.level_start_index(shapes).tolist() == [int(g["level_start_index"])]
    wl = gen.WORKLOADS["tiny"]
    assert (wl.bs, wl.num_heads, wl.num_points, wl.num_queries, wl.head_dim) == (
        int(g["bs"]), int(g["num_heads"]), int(g["num_points"]), int(g["num_queries"]),
        int(g["head_dim"]))
    assert wl.spatial_shapes == shapes


def test_reference_points_match_printed_example():
    g = read_golden("reference_points.txt")
    (H, W), = parse_shapes(g["shape"])
    ref = gen.encoder_reference_points([(H, W)])
    px = ref * np.array([W, H])
    first = np.array([float(t) for t in g["first_pixel_xy"].split()]).reshape(-1, 2)
    np.testing.assert_allclose(px[:3], first, rtol=0, atol=1e-12)
    np.testing.assert_allclose(px[W], [float(t) for t in g["row1_first_pixel_xy"].split()],
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(px[-1], [float(t) for t in g["last_pixel_xy"].split()],
                               rtol=0, atol=1e-9)


# ------------------------------------------------------------- exact pins

def _pixel_centre_problem(shapes, bs=2, M=3, D=8, P=2, Q=7, seed=3):
    """Every sample at a pixel centre of a power-of-two map, weight 1."""
    rng = np.random.default_rng(seed)
    L = len(shapes)
    K = gen.num_keys(shapes)
    lsi = gen.level_start_index(shapes)
    loc = np.empty((bs, Q, M, L, P, 2), np.float32)
    keys = np.empty((bs, Q, M, L, P), np.int64)
    for l, (H, W) in enumerate(shapes):
        ix = rng.integers(0, W, size=(bs, Q, M, P))
        iy = rng.integers(0, H, size=(bs, Q, M, P))
        loc[:, :, :, l, :, 0] = (ix + 0.5) / W
        loc[:, :, :, l, :, 1] = (iy + 0.5) / H
        keys[:, :, :, l, :] = lsi[l] + iy * W + ix
    return K, lsi, loc, keys


@pytest.mark.parametrize("exact", [False, True])
def test_key_index_field_returns_key_exactly(exact):
    """value[b,k,m,d] = k (+ offsets) at pixel centres returns the flattened key bit for bit."""
    shapes = ((16, 32), (8, 16), (4, 8), (2, 4), (1, 1))
    bs, M, D = 2, 3, 8
    K, lsi, loc, keys = _pixel_centre_problem(shapes, bs=bs, M=M, D=D)
    b = np.arange(bs)[:, None, None, None]
    k = np.arange(K)[None, :, None, None]
    m = np.arange(M)[None, None, :, None]
    d = np.arange(D)[None, None, None, :]
    value = (k + 100000 * m + 1000000 * b + 0.25 * d).astype(np.float64)
    L, P = len(shapes), loc.shape[4]
    w = np.zeros(loc.shape[:-1], np.float32)
    rng = np.random.default_rng(1)
    ls = rng.integers(0, L, size=w.shape[:3])
    ps = rng.integers(0, P, size=w.shape[:3])
    for (bb, qq, mm), l in np.ndenumerate(ls):
        w[bb, qq, mm, l, ps[bb, qq, mm]] = 1.0
    out = oracle.forward(value, np.array(shapes), lsi, loc, w, exact_coords=exact)
    out = out.reshape(bs, -1, M, D)
    for (bb, qq, mm), l in np.ndenumerate(ls):
        key = keys[bb, qq, mm, l, ps[bb, qq, mm]]
        want = key + 100000 * mm + 1000000 * bb + 0.25 * np.arange(D)
        assert np.array_equal(out[bb, qq, mm], want)


def test_pixel_centre_identity_non_power_of_two():
    """For any map, loc at a pixel centre returns that pixel within W*ulp(loc)*max|v|."""
    shapes = ((13, 21), (7, 5))
    K, lsi, loc, keys = _pixel_centre_problem(shapes, bs=1, M=2, D=8, P=3, Q=9, seed=5)
    rng = np.random.default_rng(2)
    value = rng.standard_normal((1, K, 2, 8))
    L = len(shapes)
    for l in range(L):
        w = np.zeros(loc.shape[:-1], np.float32)
        w[:, :, :, l, 0] = 1.0
        out = oracle.forward(value, np.array(shapes), lsi, loc, w).reshape(1, -1, 2, 8)
        k = keys[:, :, :, l, 0]
        want = value[0][k[0], np.arange(2)[None, :]]
        tol = max(shapes[l]) * np.finfo(np.float32).eps * np.abs(value).max() * 2
        np.testing.assert_allclose(out[0], want, rtol=0, atol=tol)


def test_out_of_range_contributes_nothing():
    shapes = ((6, 10), (3, 5))
    wl, inp = _problem(shapes, bs=1, M=2, D=8, P=4, Q=6, seed=7)
    loc = inp["sampling_locations"].copy()
    # x_im <= -1  <=> loc_x <= -0.5/W ; x_im >= W <=> loc_x >= 1 + 0.5/W
    loc[..., 0, 0] = -0.5 / 10 - 0.3
    loc[..., 1, 0] = 1.0 + 0.5 / 10 + 0.01
    loc[..., 2, 1] = -0.5 / 6 - 1e-3
    loc[..., 3, 1] = 1.0 + 0.5 / 6
    loc[:, :, :, 1, :, 0] = 2.5
    loc = loc.astype(np.float32)
    args = (inp["value"], inp["spatial_shapes"], inp["level_start_index"], loc,
            inp["attention_weights"])
    out = oracle.forward(*args)
    np.testing.assert_array_equal(out, 0.0)
    gv, gl, gw = oracle.backward(*args, inp["grad_output"])
    np.testing.assert_array_equal(gv, 0.0)
    np.testing.assert_array_equal(gl, 0.0)
    np.testing.assert_array_equal(gw, 0.0)


def _interior(rng, shapes, bs, Q, M, P):
    """Locations whose four pixels all lie on the map: 0 < x_im < W - 1, 0 < y_im < H - 1."""
    L = len(shapes)
    loc = np.empty((bs, Q, M, L, P, 2), np.float64)
    for l, (H, W) in enumerate(shapes):
        xi = rng.uniform(0.01, W - 1 - 0.01, size=(bs, Q, M, P))
        yi = rng.uniform(0.01, H - 1 - 0.01, size=(bs, Q, M, P))
        loc[:, :, :, l, :, 0] = (xi + 0.5) / W
        loc[:, :, :, l, :, 1] = (yi + 0.5) / H
    return loc.astype(np.float32)


def test_constant_field():
    """value == c everywhere, interior samples: out = c * sum(a); sum_k grad_value = sum(a*g)."""
    shapes = ((9, 14), (5, 7), (3, 3))
    bs, Q, M, D, P = 2, 11, 3, 8, 4
    rng = np.random.default_rng(11)
    K = gen.num_keys(shapes)
    c = 1.75
    value = np.full((bs, K, M, D), c)
    loc = _interior(rng, shapes, bs, Q, M, P)
    w = rng.random((bs, Q, M, len(shapes), P)).astype(np.float32)
    g = rng.standard_normal((bs, Q, M * D))
    lsi = gen.level_start_index(shapes)
    out = oracle.forward(value, np.array(shapes), lsi, loc, w).reshape(bs, Q, M, D)
    want = c * w.astype(np.float64).sum(axis=(3, 4))[..., None]
    np.testing.assert_allclose(out, np.broadcast_to(want, out.shape), rtol=1e-13, atol=0)
    gv, gl, gw = oracle.backward(value, np.array(shapes), lsi, loc, w, g)
    gsum = gv.sum(axis=1)                                            # [bs, M, D]
    want_g = np.einsum("bqm,bqmd->bmd", w.astype(np.float64).sum(axis=(3, 4)),
                       g.reshape(bs, Q, M, D))
    np.testing.assert_allclose(gsum, want_g, rtol=1e-12, atol=1e-12)
    # constant field: no gradient with respect to location
    np.testing.assert_allclose(gl, 0.0, atol=1e-11)


def test_linear_field_closed_form():
    """value = alpha_d * x + beta_d * y + gamma_d per level (interior samples).

    Bilinear interpolation reproduces affine functions exactly, so
      out          = sum a (alpha x_im + beta y_im + gamma)
      grad_loc     = a * (W * sum_d g alpha, H * sum_d g beta)
      grad_weight  = sum_d g (alpha x_im + beta y_im + gamma)
    with x_im = fp32(loc_x * W - 0.5) (coordinate contract).
    """
    shapes = ((9, 14), (5, 7), (4, 3))
    bs, Q, M, D, P = 1, 13, 2, 8, 3
    rng = np.random.default_rng(12)
    L = len(shapes)
    K = gen.num_keys(shapes)
    lsi = gen.level_start_index(shapes)
    alpha = rng.standard_normal((L, M, D))
    beta = rng.standard_normal((L, M, D))
    gamma = rng.standard_normal((L, M, D))
    value = np.empty((bs, K, M, D))
    for l, (H, W) in enumerate(shapes):
        yy, xx = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
        f = (alpha[l][None] * xx.reshape(-1, 1, 1) + beta[l][None] * yy.reshape(-1, 1, 1)
             + gamma[l][None])
        value[:, lsi[l]:lsi[l] + H * W] = f[None]
    loc = _interior(rng, shapes, bs, Q, M, P)
    w = rng.random((bs, Q, M, L, P)).astype(np.float32)
    g = rng.standard_normal((bs, Q, M * D))
    gq = g.reshape(bs, Q, M, D)
    W_ = np.array([s[1] for s in shapes], np.float64)
    H_ = np.array([s[0] for s in shapes], np.float64)
    xim = (loc[..., 0].astype(np.float64) * W_[:, None] - 0.5).astype(np.float32).astype(np.float64)
    yim = (loc[..., 1].astype(np.float64) * H_[:, None] - 0.5).astype(np.float32).astype(np.float64)
    # f at each sample: [bs,Q,M,L,P,D]
    fs = (np.einsum("lmd,bqmlp->bqmlpd", alpha, xim) + np.einsum("lmd,bqmlp->bqmlpd", beta, yim)
          + gamma.transpose(1, 0, 2)[None, None, :, :, None, :])
    want = np.einsum("bqmlp,bqmlpd->bqmd", w.astype(np.float64), fs)
    out = oracle.forward(value, np.array(shapes), lsi, loc, w).reshape(bs, Q, M, D)
    np.testing.assert_allclose(out, want, rtol=1e-11, atol=1e-11)
    gv, gl, gw = oracle.backward(value, np.array(shapes), lsi, loc, w, g)
    want_gw = np.einsum("bqmd,bqmlpd->bqmlp", gq, fs)
    np.testing.assert_allclose(gw, want_gw, rtol=1e-11, atol=1e-11)
    ga = np.einsum("bqmd,lmd->bqml", gq, alpha)[..., None] * w * W_[:, None]
    gb = np.einsum("bqmd,lmd->bqml", gq, beta)[..., None] * w * H_[:, None]
    np.testing.assert_allclose(gl[..., 0], ga, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(gl[..., 1], gb, rtol=1e-10, atol=1e-10)


def test_level_separation():
    """A one-hot weight on level l touches grad_value only inside level l's key range."""
    shapes = ((6, 9), (4, 5), (2, 3))
    wl, inp = _problem(shapes, bs=1, M=2, D=8, P=3, Q=8, seed=21)
    lsi = inp["level_start_index"]
    for l, (H, W) in enumerate(shapes):
        w = np.zeros_like(inp["attention_weights"])
        w[:, :, :, l, :] = 1.0
        gv, _, _ = oracle.backward(inp["value"], inp["spatial_shapes"], lsi,
                                   inp["sampling_locations"], w, inp["grad_output"])
        inside = np.zeros(gv.shape[1], bool)
        inside[lsi[l]:lsi[l] + H * W] = True
        assert np.all(gv[:, ~inside] == 0)
        assert np.any(gv[:, inside] != 0)


def test_ascend_example_closed_form():
    """Ascend call example: every sample at loc = 0.005 on one 100x100 level.

    x_im = fp32(0.005f * 100 - 0.5) is a hair below 0, so the cell is
    [-1, 0] in both axes and only pixel (0, 0) is on the map, with weight
    (1 + x_im)(1 + y_im): out[q, m] = sum_p a[q,m,p] * (1 + x_im)^2 * value[0, m].
    grad_output = ones gives grad_weight = sum_d sample_d.
    """
    g = read_golden("ascend_example.txt")
    wl = gen.WORKLOADS["tiny"]
    inp = gen.make_inputs(wl)
    loc = np.full_like(inp["sampling_locations"], np.float32(float(g["location"])))
    xim = float(np.float32(np.float64(np.float32(0.005)) * 100.0 - 0.5))
    assert -1e-6 < xim < 0.0
    wt = (1.0 + xim) ** 2
    a = inp["attention_weights"].astype(np.float64)
    v0 = inp["value"][0, 0].astype(np.float64)                        # [M, D]
    want = a.sum(axis=(3, 4))[..., None] * wt * v0[None, None]
    out = oracle.forward(inp["value"], inp["spatial_shapes"], inp["level_start_index"], loc,
                         inp["attention_weights"]).reshape(want.shape)
    np.testing.assert_allclose(out, want, rtol=1e-14, atol=0)
    _, _, gw = oracle.backward(inp["value"], inp["spatial_shapes"], inp["level_start_index"],
                               loc, inp["attention_weights"], inp["grad_output"])
    want_gw = np.broadcast_to((wt * v0.sum(axis=-1))[None, None, :, None, None], gw.shape)
    np.testing.assert_allclose(gw, want_gw, rtol=1e-14, atol=0)


# ------------------------------------------------ independent formulations

BRUTE_SHAPES = [
    ((5, 7),),
    ((4, 6), (2, 3)),
    ((1, 5), (3, 1), (1, 1)),
    ((7, 4), (3, 2), (2, 2), (1, 3)),
]


@pytest.mark.parametrize("shapes", BRUTE_SHAPES)
@pytest.mark.parametrize("exact", [False, True])
def test_against_brute_force_tent_sums(shapes, exact):
    wl, inp = _problem(shapes, bs=2, M=2, D=8, P=3, Q=6, seed=len(shapes) * 7 + exact)
    out = oracle.forward(*_args(inp), exact_coords=exact)
    want = tent.forward(*_args(inp), fp32_contract=not exact)
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)
    gv, gl, gw = oracle.backward(*_args(inp), inp["grad_output"], exact_coords=exact)
    tv, tl, tw = tent.backward(*_args(inp), inp["grad_output"], fp32_contract=not exact)
    np.testing.assert_allclose(gv, tv, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gw, tw, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(gl, tl, rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("shapes", BRUTE_SHAPES[1:] + [((16, 9), (8, 5), (4, 3))])
def test_against_torch_grid_sample_fp64(shapes):
    wl, inp = _problem(shapes, bs=2, M=3, D=8, P=4, Q=9, seed=40 + len(shapes))
    out = oracle.forward(*_args(inp), exact_coords=True)
    want = grid_sample_ref.forward(*_args(inp))
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)
    gv, gl, gw = oracle.backward(*_args(inp), inp["grad_output"], exact_coords=True)
    tv, tl, tw = grid_sample_ref.backward(*_args(inp), inp["grad_output"])
    np.testing.assert_allclose(gv, tv, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(gw, tw, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(gl, tl, rtol=1e-10, atol=1e-10)


def _near_kink(loc, shapes, tol_px=1e-3):
    """Samples whose pixel coordinate lies within tol of an integer or of -1 / W."""
    bad = np.zeros(loc.shape[:-1], bool)
    for l, (H, W) in enumerate(shapes):
        for ax, size in ((0, W), (1, H)):
            t = loc[:, :, :, l, :, ax].astype(np.float64) * size - 0.5
            bad[:, :, :, l, :] |= np.abs(t - np.round(t)) < tol_px
            bad[:, :, :, l, :] |= (np.abs(t + 1) < tol_px) | (np.abs(t - size) < tol_px)
    return bad


def test_backward_matches_central_differences():
    shapes = ((6, 8), (3, 4))
    wl, inp = _problem(shapes, bs=1, M=2, D=8, P=2, Q=4, seed=77)
    args = list(_args(inp))
    value = args[0].astype(np.float64)
    loc = args[3].astype(np.float64)
    w = args[4].astype(np.float64)
    g = inp["grad_output"].astype(np.float64)
    gv, gl, gw = oracle.backward(value, args[1], args[2], loc, w, g, exact_coords=True)

    def J(v=value, lc=loc, ww=w):
        return float((oracle.forward(v, args[1], args[2], lc, ww, exact_coords=True) * g).sum())

    h = 1e-6
    bad = _near_kink(loc, shapes, tol_px=1e-3)
    rng = np.random.default_rng(0)
    checked = 0
    for idx in zip(*np.nonzero(~bad)):
        for ax in range(2):
            lp, lm = loc.copy(), loc.copy()
            lp[idx + (ax,)] += h
            lm[idx + (ax,)] -= h
            fd = (J(lc=lp) - J(lc=lm)) / (2 * h)
            an = gl[idx + (ax,)]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (idx, ax, fd, an)
            checked += 1
        wp, wm = w.copy(), w.copy()
        wp[idx] += h
        wm[idx] -= h
        fd = (J(ww=wp) - J(ww=wm)) / (2 * h)
        assert abs(fd - gw[idx]) <= 1e-6 * max(1.0, abs(gw[idx]))
    assert checked > 10
    flat = value.reshape(-1)
    for i in rng.choice(flat.size, size=40, replace=False):
        vp, vm = flat.copy(), flat.copy()
        vp[i] += h
        vm[i] -= h
        fd = (J(v=vp.reshape(value.shape)) - J(v=vm.reshape(value.shape))) / (2 * h)
        assert abs(fd - gv.reshape(-1)[i]) <= 1e-6 * max(1.0, abs(gv.reshape(-1)[i]))


def test_fp32_contract_selects_cell_of_single_rounding():
    """coord_mode 0 equals rounding the exact loc*W - 0.5 once to binary32.

    A location whose exact pixel coordinate sits just below an integer in
    fp64 but rounds onto it in fp32 must be sampled from the upper cell.
    """
    W = 3
    # loc*3 - 0.5 = 1 - 2^-30 exactly in fp64 -> rounds to 1.0f in fp32
    loc_x = np.float32((1.5 - 2.0 ** -30) / 3.0)
    t = float(loc_x) * 3 - 0.5
    t32 = float(np.float32(t))
    value = np.zeros((1, W, 1, 8))
    value[0, :, 0, :] = np.array([10.0, 20.0, 30.0])[:, None]
    loc = np.zeros((1, 1, 1, 1, 1, 2), np.float32)
    loc[..., 0] = loc_x
    loc[..., 1] = 0.5
    w = np.ones((1, 1, 1, 1, 1), np.float32)
    out = oracle.forward(value, np.array([[1, W]]), np.array([0]), loc, w)
    fx = t32 - np.floor(t32)
    x0 = int(np.floor(t32))
    want = (1 - fx) * value[0, x0, 0, 0] + fx * (value[0, x0 + 1, 0, 0] if x0 + 1 < W else 0.0)
    assert out[0, 0, 0] == want


def test_workload_generator_is_seeded_and_shaped():
    for name, wl in gen.WORKLOADS.items():
        if name in ("envelope",):
            continue
        a = gen.make_inputs(wl, with_grad=False)
        b = gen.make_inputs(wl, with_grad=False)
        assert np.array_equal(a["sampling_locations"], b["sampling_locations"])
        assert a["value"].shape == (wl.bs, wl.num_keys, wl.num_heads, wl.head_dim)
        assert a["sampling_locations"].shape == (wl.bs, wl.num_queries, wl.num_heads,
                                                 wl.num_levels, wl.num_points, 2)
        if wl.weight_kind == "softmax":
            s = a["attention_weights"].astype(np.float64).sum(axis=(3, 4))
            np.testing.assert_allclose(s, 1.0, atol=1e-2 if wl.dtype in ("bf16", "f16") else 1e-5)
    enc = gen.WORKLOADS["encoder"]
    assert enc.num_keys == enc.num_queries == 22223
    assert gen.level_start_index(enc.spatial_shapes).tolist() == [0, 16700, 20900, 21950]
    assert gen.WORKLOADS["envelope"].num_keys == 53125


def test_bf16_rounding_is_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, 1.0 + 2 ** -9, -2.5, 3.140625],
                 np.float32)
    bits = gen.f32_to_bf16_bits(x)
    back = gen.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 (bf16 has 7 fraction bits): even -> 1.0
    np.testing.assert_array_equal(back, np.array([1.0, 1.0, 1.0 + 2 ** -7, 1.0, -2.5, 3.140625],
                                                 np.float32))


def test_f16_rounding_is_round_to_nearest_even():
    # IEEE half has 10 fraction bits: 1 + 2^-11 is a tie between 1 and 1 + 2^-10 (even -> 1),
    # 1 + 3*2^-11 a tie between 1 + 2^-10 and 1 + 2^-9 (even -> 1 + 2^-9)
    x = np.array([1.0, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, 1.0 + 2 ** -12, -2.5, 65504.0],
                 np.float32)
    bits = gen.f32_to_f16_bits(x)
    assert bits[0] == 0x3C00 and bits[5] == 0x7BFF
    np.testing.assert_array_equal(gen.f16_bits_to_f32(bits),
                                  np.array([1.0, 1.0, 1.0 + 2 ** -9, 1.0, -2.5, 65504.0], np.float32))


@pytest.mark.parametrize("exact", [False, True])
def test_backward_is_the_adjoint_in_value_and_weights(exact):
    """The operator is linear in value and in the attention weights, so its
    gradients with respect to them are its adjoints: <out, G> must equal both
    <value, grad_value> and <weights, grad_weights> for any G (random ragged
    shapes, samples inside and outside the maps)."""
    for seed, shapes in ((31, ((5, 7), (3, 2), (1, 1))), (32, ((9, 4), (4, 6)))):
        wl = gen.random_workload(seed, 2, shapes, 3, 8, 5, 11)
        inp = gen.make_inputs(wl)
        args = (inp["value"], inp["spatial_shapes"], inp["level_start_index"],
                inp["sampling_locations"], inp["attention_weights"])
        out = oracle.forward(*args, exact_coords=exact)
        gv, _, gw = oracle.backward(*args, inp["grad_output"], exact_coords=exact)
        lhs = float((out * inp["grad_output"].astype(np.float64)).sum())
        np.testing.assert_allclose((inp["value"].astype(np.float64) * gv).sum(), lhs, rtol=1e-12)
        np.testing.assert_allclose((inp["attention_weights"].astype(np.float64) * gw).sum(), lhs,
                                   rtol=1e-12)
