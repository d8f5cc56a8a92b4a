"""Pins of oracle.touched_rows, the count of distinct value rows one forward
reads with a non-zero weight (the "touched bytes" the benchmark quotes for the
decoder workload).

Closed forms: a sample at a pixel centre reads one pixel; a sample strictly
inside a cell reads four; one with -1 < x_im < 0 reads only column 0; a zero
attention weight reads nothing.  Independent formulation: the tent form of the
bilinear sample (oracle/tent.py), where a pixel (i, j) is read exactly when
max(0, 1 - |x - j|) * max(0, 1 - |y - i|) > 0, brute-forced over every pixel.
Planted mistakes in a copy of the C source must fail these pins.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import tent
from scale_deformable_attention_05_b300 import inputs as gen

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "msda_oracle.c")


def _count(inp, lib=None):
    bs, K, M = inp["value"].shape[:3]
    return oracle.touched_rows(inp["spatial_shapes"], inp["level_start_index"],
                               inp["sampling_locations"], inp["attention_weights"], bs, K, M,
                               lib=lib)


def _brute_force(inp):
    """Rows (b, key, m) whose tent weight is non-zero for some sample with a != 0."""
    loc = np.asarray(inp["sampling_locations"], np.float64)
    a = np.asarray(inp["attention_weights"], np.float64)
    shapes = np.asarray(inp["spatial_shapes"])
    lsi = np.asarray(inp["level_start_index"])
    bs, Q, M, L, P, _ = loc.shape
    seen = set()
    for l, (H, W) in enumerate(shapes.tolist()):
        x = tent._coords(loc[:, :, :, l, :, 0], W, True)
        y = tent._coords(loc[:, :, :, l, :, 1], H, True)
        ii, jj = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
        for b, q, m, p in np.ndindex(bs, Q, M, P):
            if a[b, q, m, l, p] == 0.0:
                continue
            w = tent._tent(x[b, q, m, p] - jj) * tent._tent(y[b, q, m, p] - ii)
            for i, j in zip(*np.nonzero(w)):
                seen.add((b, int(lsi[l] + i * W + j), m))
    return len(seen)


def _centre_inputs(seed=4, bs=2, Q=9, M=3, P=3, shapes=((8, 16), (4, 8))):
    """Samples at pixel centres of power-of-two maps (x_im, y_im exact integers)."""
    rng = np.random.default_rng(seed)
    L = len(shapes)
    lsi = gen.level_start_index(shapes)
    loc = np.empty((bs, Q, M, L, P, 2), np.float32)
    keys = set()
    for b, q, m, l, p in np.ndindex(bs, Q, M, L, P):
        H, W = shapes[l]
        i, j = rng.integers(0, H), rng.integers(0, W)
        loc[b, q, m, l, p] = ((j + 0.5) / W, (i + 0.5) / H)
        keys.add((b, int(lsi[l] + i * W + j), m))
    K = gen.num_keys(shapes)
    return {"value": np.zeros((bs, K, M, 1)), "spatial_shapes": np.array(shapes),
            "level_start_index": lsi, "sampling_locations": loc,
            "attention_weights": np.full((bs, Q, M, L, P), 0.25, np.float32)}, len(keys)


def test_pixel_centres_read_one_pixel_each():
    inp, want = _centre_inputs()
    assert _count(inp) == want


def test_interior_sample_reads_four_rows_and_edge_sample_reads_column_zero():
    shapes = ((4, 8),)
    base = {"value": np.zeros((1, 32, 1, 1)), "spatial_shapes": np.array(shapes),
            "level_start_index": gen.level_start_index(shapes)}
    w = np.ones((1, 1, 1, 1, 1), np.float32)
    inside = dict(base, sampling_locations=np.array([[[[[[0.3, 0.4]]]]]], np.float32),
                  attention_weights=w)
    assert _count(inside) == 4
    # x_im = 0.05 * 8 - 0.5 = -0.1: only column 0 of rows y0 and y0 + 1
    edge = dict(base, sampling_locations=np.array([[[[[[0.05, 0.4]]]]]], np.float32),
                attention_weights=w)
    assert _count(edge) == 2
    # y at a pixel centre as well: a single row
    corner = dict(base, sampling_locations=np.array([[[[[[0.05, 0.375]]]]]], np.float32),
                  attention_weights=w)
    assert _count(corner) == 1
    # zero attention weight reads nothing; a sample past the map reads nothing
    assert _count(dict(inside, attention_weights=0 * w)) == 0
    far = dict(base, sampling_locations=np.array([[[[[[1.2, 0.4]]]]]], np.float32),
               attention_weights=w)
    assert _count(far) == 0


@pytest.mark.parametrize("seed", [31, 32])
def test_matches_brute_force_tent_count(seed):
    wl = gen.random_workload(seed, 2, ((5, 7), (3, 4), (1, 2)), 2, 8, 3, 7)
    inp = gen.make_inputs(wl)
    inp["attention_weights"] = np.where(
        np.random.default_rng(seed).random(inp["attention_weights"].shape) < 0.2, 0.0,
        inp["attention_weights"]).astype(np.float32)
    assert _count(inp) == _brute_force(inp)


MUTATIONS = {
    "zero_corner_weight_counted": (" || f.w[c] == 0.0) continue;", ") continue;"),
    "zero_attention_counted": ("if (!f.in_range || attention_weights[pt] == 0.0) continue;",
                               "if (!f.in_range) continue;"),
    "heads_merged": ("unsigned char* mk = mark + (b * K + f.key[c]) * M + m;",
                     "unsigned char* mk = mark + (b * K + f.key[c]) * M;"),
    "batches_merged": ("unsigned char* mk = mark + (b * K + f.key[c]) * M + m;",
                       "unsigned char* mk = mark + f.key[c] * M + m;"),
    "every_visit_counted": ("if (!*mk) { *mk = 1; ++count; }", "{ *mk = 1; ++count; }"),
}


def _pins_pass(lib):
    inp, want = _centre_inputs()
    if _count(inp, lib) != want:
        return False
    for seed in (31, 32):
        wl = gen.random_workload(seed, 2, ((5, 7), (3, 4), (1, 2)), 2, 8, 3, 7)
        inp = gen.make_inputs(wl)
        inp["attention_weights"] = np.where(
            np.random.default_rng(seed).random(inp["attention_weights"].shape) < 0.2, 0.0,
            inp["attention_weights"]).astype(np.float32)
        if _count(inp, lib) != _brute_force(inp):
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_touched_rows_mutant_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found"
    c_path, so_path = tmp_path / "mutant.c", tmp_path / "mutant.so"
    c_path.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(so_path), str(c_path), "-lm"], check=True)
    assert _pins_pass(oracle.load()), "the unmutated oracle must pass"
    assert not _pins_pass(oracle.load(str(so_path))), f"mutation {name} slipped through"
