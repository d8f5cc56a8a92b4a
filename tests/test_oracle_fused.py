"""Pins of the fused-preparation oracle (oracle/fused.py) against closed forms,
invariants and finite differences; none compares the oracle with itself."""
import numpy as np
import pytest

from oracle import fused
from scale_deformable_attention_05_b300 import inputs as gen

SHAPES = ((16, 32), (8, 16), (4, 8))           # powers of two: pixel centres and /W are exact


def _problem(seed, ref_dim=2, bs=2, M=2, D=8, P=4, Q=5, shapes=SHAPES):
    rng = np.random.default_rng(seed)
    L = len(shapes)
    K = gen.num_keys(shapes)
    value = rng.standard_normal((bs, K, M, D)).astype(np.float32)
    ref = rng.uniform(0.2, 0.8, (bs, Q, L, 2))
    if ref_dim == 4:
        ref = np.concatenate([ref, rng.uniform(0.05, 0.3, (bs, Q, L, 2))], -1)
    off = rng.normal(0.0, 1.5, (bs, Q, M, L, P, 2))
    logits = rng.standard_normal((bs, Q, M, L * P))
    g = rng.standard_normal((bs, Q, M * D))
    f32 = lambda a: np.asarray(a, np.float32)
    return (value, np.array(shapes, np.int64), gen.level_start_index(shapes), f32(ref), f32(off),
            f32(logits), f32(g))


def test_softmax_weights_closed_form():
    z = np.array([[[[0.3, -1.2]]]])
    a = fused.softmax_weights(z, 1, 2)
    s = 1.0 / (1.0 + np.exp(-1.5))                        # sigma(z1 - z2)
    np.testing.assert_allclose(a.reshape(-1), [s, 1.0 - s], rtol=0, atol=1e-15)


@pytest.mark.parametrize("ref_dim", [2, 4])
def test_logit_shift_invariance(ref_dim):
    v, sh, lsi, ref, off, logits, g = _problem(1, ref_dim)
    out = fused.forward(v, sh, lsi, ref, off, logits)
    out2 = fused.forward(v, sh, lsi, ref, off, logits.astype(np.float64) + 7.5)   # exact shift
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-12)
    gl = fused.backward(v, sh, lsi, ref, off, logits, g)[2]
    np.testing.assert_allclose(gl.sum(-1), 0.0, atol=1e-12)   # softmax Jacobian rows sum to 0


def test_integer_offsets_shift_by_whole_pixels():
    """2-d references at pixel centres, integer offsets in pixels, one dominant
    logit: the output is the value row of the shifted pixel."""
    rng = np.random.default_rng(3)
    bs, M, D, P, Q = 1, 2, 8, 3, 6
    shapes = ((16, 32), (8, 16), (8, 8))        # room for +-2 pixel shifts on every level
    L = len(shapes)
    K = gen.num_keys(shapes)
    lsi = gen.level_start_index(shapes)
    value = rng.standard_normal((bs, K, M, D)).astype(np.float32)
    ref = np.empty((bs, Q, L, 2), np.float32)
    off = np.zeros((bs, Q, M, L, P, 2), np.float32)
    logits = np.full((bs, Q, M, L * P), -40.0, np.float32)
    want = np.empty((bs, Q, M, D))
    for q in range(Q):
        px = []
        for l, (H, W) in enumerate(shapes):
            x, y = rng.integers(2, W - 2), rng.integers(2, H - 2)
            ref[0, q, l] = ((x + 0.5) / W, (y + 0.5) / H)
            px.append((x, y))
        for m in range(M):
            l, p = rng.integers(0, L), rng.integers(0, P)
            kx, ky = rng.integers(-2, 3), rng.integers(-2, 3)
            off[0, q, m, l, p] = (kx, ky)
            logits[0, q, m, l * P + p] = 40.0
            H, W = shapes[l]
            key = lsi[l] + (px[l][1] + ky) * W + px[l][0] + kx
            want[0, q, m] = value[0, key, m]
    out = fused.forward(value, np.array(shapes), lsi, ref, off, logits)
    np.testing.assert_allclose(out.reshape(bs, Q, M, D), want, rtol=1e-12, atol=1e-12)


def test_four_d_references_with_matching_box_equal_the_two_d_form():
    """ref_wh = (2P/W, 2P/H) turns off/P * wh * 0.5 into off/(W, H): both forms
    must pick the same locations (bit for bit here) and agree on every gradient."""
    v, sh, lsi, ref2, off, logits, g = _problem(5, 2)
    P = off.shape[4]
    wh = np.stack([2.0 * P / sh[:, 1], 2.0 * P / sh[:, 0]], -1).astype(np.float32)
    ref4 = np.concatenate([ref2, np.broadcast_to(wh, ref2.shape)], -1).astype(np.float32)
    np.testing.assert_array_equal(fused.locations(ref4, off, sh), fused.locations(ref2, off, sh))
    np.testing.assert_array_equal(fused.forward(v, sh, lsi, ref4, off, logits),
                                  fused.forward(v, sh, lsi, ref2, off, logits))
    b2 = fused.backward(v, sh, lsi, ref2, off, logits, g)
    b4 = fused.backward(v, sh, lsi, ref4, off, logits, g)
    for x2, x4 in zip(b2[:3], b4[:3]):
        np.testing.assert_allclose(x4, x2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b4[3][..., :2], b2[3], rtol=1e-12, atol=1e-12)


NPOT_SHAPES = ((7, 21), (5, 13), (3, 9))       # no power of two: 1/W is inexact


def _npot_offsets(ref_dim, seed=17, Q=8, M=2, P=7):
    """Offsets whose quotients in the module's expression are short binary
    fractions: 2-d off = (W, H) * t, 4-d off = P * t, t = k / 64.  The real
    arithmetic of the walk-through's MSDeformAttn.forward ("2.2.4 源码分析": off /
    (W, H); "2.4": off / P * wh * 0.5) then gives loc = ref + t and
    ref_xy + t * wh / 2 exactly, and so must binary32 with correctly rounded
    division."""
    rng = np.random.default_rng(seed)
    L = len(NPOT_SHAPES)
    t = rng.integers(1, 256, (1, Q, M, L, P, 2)) / 64.0
    if ref_dim == 2:
        ref = rng.choice([0.0, 0.125, 0.25], (1, Q, L, 2))
        scale = np.array([[W, H] for H, W in NPOT_SHAPES], np.float64)[None, None, None, :, None]
        want = ref[:, :, None, :, None, :] + t
    else:
        xy = np.zeros((1, Q, L, 2))
        wh = rng.choice([0.375, 0.6875, 0.9375], (1, Q, L, 2))
        ref = np.concatenate([xy, wh], -1)
        scale = np.float64(P)
        want = t * wh[:, :, None, :, None, :] * 0.5
    off = t * scale
    assert np.array_equal(off.astype(np.float32).astype(np.float64), off)   # exact inputs
    return ref.astype(np.float32), off.astype(np.float32), want


@pytest.mark.parametrize("ref_dim", [2, 4])
def test_locations_divide_as_the_module_writes(ref_dim):
    ref, off, want = _npot_offsets(ref_dim)
    loc = fused.locations(ref, off, np.array(NPOT_SHAPES))
    assert loc.dtype == np.float32
    np.testing.assert_array_equal(loc.astype(np.float64), want)
    # the pin discriminates: products with once-rounded reciprocals miss some of them
    f = np.float32
    if ref_dim == 2:
        inv = f(1) / np.array([[W, H] for H, W in NPOT_SHAPES], f)[None, None, None, :, None]
        recip = ref[:, :, None, :, None, :] + off * inv
    else:
        recip = ref[:, :, None, :, None, :2] + (off * ref[:, :, None, :, None, 2:]) * (
            f(1) / f(2 * off.shape[4]))
    assert (recip.astype(np.float64) != want).any()


def _pixel_coords(ref, off, shapes):
    loc = fused.locations(ref, off, shapes, exact=True)
    W = np.asarray(shapes)[:, 1].astype(np.float64)[None, None, None, :, None]
    H = np.asarray(shapes)[:, 0].astype(np.float64)[None, None, None, :, None]
    return loc[..., 0] * W - 0.5, loc[..., 1] * H - 0.5


def _far_from_cell_edges(x, y, tol=2e-3):
    fx, fy = x - np.floor(x), y - np.floor(y)
    return (np.minimum(fx, 1 - fx) > tol) & (np.minimum(fy, 1 - fy) > tol)


@pytest.mark.parametrize("ref_dim", [2, 4])
def test_backward_matches_central_differences(ref_dim):
    v, sh, lsi, ref, off, logits, g = _problem(11 + ref_dim, ref_dim)
    ref, off, logits = (np.asarray(a, np.float64) for a in (ref, off, logits))
    g = np.asarray(g, np.float64)
    f = lambda r, o, z: float((fused.forward(v, sh, lsi, r, o, z, exact=True) * g).sum())
    _, g_off, g_log, g_ref = fused.backward(v, sh, lsi, ref, off, logits, g, exact=True)
    x, y = _pixel_coords(ref, off, sh)
    ok = _far_from_cell_edges(x, y)
    rng = np.random.default_rng(7)
    h = 1e-6
    checked = 0
    for _ in range(40):                                     # offsets
        i = tuple(rng.integers(0, n) for n in off.shape)
        if not ok[i[:5]]:
            continue
        e = np.zeros_like(off); e[i] = h
        fd = (f(ref, off + e, logits) - f(ref, off - e, logits)) / (2 * h)
        np.testing.assert_allclose(g_off[i], fd, rtol=1e-5, atol=1e-7)
        checked += 1
    for _ in range(20):                                     # logits
        i = tuple(rng.integers(0, n) for n in logits.shape)
        e = np.zeros_like(logits); e[i] = h
        fd = (f(ref, off, logits + e) - f(ref, off, logits - e)) / (2 * h)
        np.testing.assert_allclose(g_log[i], fd, rtol=1e-5, atol=1e-7)
    for _ in range(20):                                     # reference points
        i = tuple(rng.integers(0, n) for n in ref.shape)
        if not ok[i[0], i[1], :, i[2]].all():
            continue
        e = np.zeros_like(ref); e[i] = h
        fd = (f(ref + e, off, logits) - f(ref - e, off, logits)) / (2 * h)
        np.testing.assert_allclose(g_ref[i], fd, rtol=1e-5, atol=1e-7)
        checked += 1
    assert checked >= 10


def _mask_problem():
    """Hand-built case: one 8x16 level, one head and point (softmax weight 1),
    value == c everywhere.  Query 0 sits on the centre of pixel (5, 3); query 1
    half-way between pixels (9, 2) and (10, 2).  Batch 1 pads pixels (5, 3) and
    (10, 2); batch 0 pads nothing."""
    H, W, D, c = 8, 16, 4, 3.0
    shapes = np.array([[H, W]])
    lsi = np.array([0])
    value = np.full((2, H * W, 1, D), c)
    ref = np.array([[(5.5 / W, 3.5 / H), (10.0 / W, 2.5 / H)]] * 2, np.float32)[:, :, None, :]
    off = np.zeros((2, 2, 1, 1, 1, 2), np.float32)
    logits = np.zeros((2, 2, 1, 1), np.float32)
    mask = np.zeros((2, H * W), bool)
    mask[1, 3 * W + 5] = mask[1, 2 * W + 10] = True
    g = np.random.default_rng(21).standard_normal((2, 2, D))
    return value, shapes, lsi, ref, off, logits, mask, g, c, W


def test_padding_mask_closed_form():
    value, sh, lsi, ref, off, logits, mask, g, c, W = _mask_problem()
    out = fused.forward(value, sh, lsi, ref, off, logits, padding_mask=mask)
    want = np.array([[c, c], [0.0, 0.5 * c]])[:, :, None] * np.ones(g.shape[-1])
    np.testing.assert_array_equal(out, want)
    gv, goff, glog, gref = fused.backward(value, sh, lsi, ref, off, logits, g, padding_mask=mask)
    gv_want = np.zeros_like(value)
    gv_want[0, 3 * W + 5, 0] = g[0, 0]
    gv_want[0, 2 * W + 9, 0] = gv_want[0, 2 * W + 10, 0] = 0.5 * g[0, 1]
    gv_want[1, 2 * W + 9, 0] = 0.5 * g[1, 1]                  # the padded neighbour gets nothing
    np.testing.assert_allclose(gv, gv_want, rtol=0, atol=1e-15)
    # d out / d x_im between a value-c pixel and a padded (zero) one is -c; offsets are in pixels
    np.testing.assert_allclose(goff[1, 1, 0, 0, 0, 0], -c * g[1, 1].sum(), rtol=1e-12)
    np.testing.assert_allclose(goff[0, 1, 0, 0, 0, 0], 0.0, atol=1e-12)
    # an all-false mask is no mask
    np.testing.assert_array_equal(
        fused.forward(value, sh, lsi, ref, off, logits, padding_mask=np.zeros_like(mask)),
        fused.forward(value, sh, lsi, ref, off, logits))


@pytest.mark.parametrize("ref_dim", [2, 4])
def test_grad_value_is_the_adjoint_with_mask(ref_dim):
    """Linear in value (masked or not): <out, G> = <value, grad_value>."""
    v, sh, lsi, ref, off, logits, g = _problem(41 + ref_dim, ref_dim)
    mask = np.random.default_rng(43).random(v.shape[:2]) < 0.3
    out = fused.forward(v, sh, lsi, ref, off, logits, padding_mask=mask)
    gv = fused.backward(v, sh, lsi, ref, off, logits, g, padding_mask=mask)[0]
    np.testing.assert_allclose((v.astype(np.float64) * gv).sum(),
                               (out * g.astype(np.float64)).sum(), rtol=1e-12)


# ------------------------------------------------ planted mistakes must be caught
def _mutant_locations_swapped(ref, off, shapes, exact=False):
    sh = np.asarray(shapes)[:, ::-1]                      # (H, W) rows read as (W, H)
    return _ORIG_LOCATIONS(ref, off, sh, exact)


def _mutant_locations_no_half(ref, off, shapes, exact=False):
    ref = np.asarray(ref)
    if ref.shape[-1] == 4:
        ref = np.concatenate([ref[..., :2], 2 * ref[..., 2:]], -1)   # drops the 0.5
    return _ORIG_LOCATIONS(ref, off, shapes, exact)


def _mutant_locations_reciprocal(ref, off, shapes, exact=False):
    """Divides by multiplying with once-rounded reciprocals (1/W, 1/H, 1/(2P))."""
    ref = np.asarray(ref)
    f = np.float64 if exact else np.float32
    r = ref.astype(f)[:, :, None, :, None, :]
    o = np.asarray(off).astype(f)
    if ref.shape[-1] == 2:
        sh = np.asarray(shapes)
        inv = f(1) / np.stack([sh[:, 1], sh[:, 0]], -1).astype(f)[None, None, None, :, None, :]
        return r + o * inv
    return r[..., :2] + (o * r[..., 2:]) * (f(1) / f(2 * o.shape[4]))


def _mutant_softmax_wrong_axis(logits, L, P):
    z = np.asarray(logits, np.float64)
    e = np.exp(z - z.max(axis=2, keepdims=True))
    return (e / e.sum(axis=2, keepdims=True)).reshape(*z.shape[:-1], L, P)   # over heads


def _mutant_mask_batch_flipped(value, padding_mask):
    m = None if padding_mask is None else np.asarray(padding_mask)[::-1]
    return _ORIG_KEEP(value, m)


def _mutant_mask_grad_kept(grad_value, keep):
    return grad_value                                     # padded rows keep their gradient


def _npot_locations_exact(ref_dim):
    ref, off, want = _npot_offsets(ref_dim)
    np.testing.assert_array_equal(
        fused.locations(ref, off, np.array(NPOT_SHAPES)).astype(np.float64), want)


_ORIG_LOCATIONS = fused.locations
_ORIG_KEEP = fused.keep_rows


def _battery():
    """True when every pin above passes."""
    try:
        test_softmax_weights_closed_form()
        for rd in (2, 4):
            test_logit_shift_invariance(rd)
        test_integer_offsets_shift_by_whole_pixels()
        test_four_d_references_with_matching_box_equal_the_two_d_form()
        for rd in (2, 4):
            _npot_locations_exact(rd)
        for rd in (2, 4):
            test_backward_matches_central_differences(rd)
        test_padding_mask_closed_form()
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("name,attr,mutant", [
    ("normaliser_transposed", "locations", _mutant_locations_swapped),
    ("box_half_dropped", "locations", _mutant_locations_no_half),
    ("reciprocal_instead_of_division", "locations", _mutant_locations_reciprocal),
    ("softmax_over_heads", "softmax_weights", _mutant_softmax_wrong_axis),
    ("mask_batch_flipped", "keep_rows", _mutant_mask_batch_flipped),
    ("mask_gradient_kept", "masked_fill_grad", _mutant_mask_grad_kept),
])
def test_fused_mutant_is_caught(monkeypatch, name, attr, mutant):
    assert _battery()
    monkeypatch.setattr(fused, attr, mutant)
    assert not _battery(), f"mutation {name} slipped through every pin"
