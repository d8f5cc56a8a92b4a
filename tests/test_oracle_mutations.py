"""The oracle's pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), builds it, and runs a battery of the pins used in
test_oracle_pins.py against the mutant: brute-force tent sums (forward and
backward, both coordinate modes), the key-index field and the pixel-centre
identity.  A mutant that passes the whole battery means the pins have a blind
spot, and the test fails.
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

MUTATIONS = {
    "fractions_swapped": ("double wx = (c & 1) ? f->fx : 1.0 - f->fx;",
                          "double wx = (c & 1) ? f->fy : 1.0 - f->fy;"),
    "corner_dropped": ("        if (!f.valid[c]) continue;\n                        if (f.key[c] < 0",
                       "        if (!f.valid[c] || c == 3) continue;\n                        if (f.key[c] < 0"),
    "half_pixel_sign_fp32": ("fmaf((float)loc, (float)size, -0.5f)", "fmaf((float)loc, (float)size, 0.5f)"),
    "half_pixel_sign_fp64": ("return loc * (double)size - 0.5;", "return loc * (double)size + 0.5;"),
    "normaliser_transposed": ("double x = pixel_coord(loc_x, W, coord_mode);",
                              "double x = pixel_coord(loc_x, H, coord_mode);"),
    "column_major_keys": ("start + yc * W + xc", "start + xc * H + yc"),
    "level_offset_dropped": ("start + yc * W + xc", "yc * W + xc"),
    "grad_x_sign": ("gx += g[d] * ((1.0 - f.fy) * (v01 - v00)", "gx += g[d] * ((1.0 - f.fy) * (v00 - v01)"),
    "grad_y_fraction": ("gy += g[d] * ((1.0 - f.fx) * (v10 - v00) + f.fx * (v11 - v01));",
                        "gy += g[d] * ((1.0 - f.fy) * (v10 - v00) + f.fy * (v11 - v01));"),
    "grad_value_without_attention": ("const double s = a * f.w[c];\n                        for (int64_t d = 0; d < D; ++d) gv[d]",
                                     "const double s = f.w[c];\n                        for (int64_t d = 0; d < D; ++d) gv[d]"),
    "grad_loc_scale_swapped": ("grad_sampling_loc[2 * pt] = (double)W * a * gx;",
                               "grad_sampling_loc[2 * pt] = (double)H * a * gx;"),
    "range_test_too_narrow": ("f->in_range = (x > -1.0 && x < (double)W",
                              "f->in_range = (x >= 0.0 && x < (double)W"),
    "upper_range_too_narrow": ("y > -1.0 && y < (double)H);", "y > -1.0 && y < (double)(H - 1));"),
    "floor_as_truncation": ("double x0 = floor(x), y0 = floor(y);",
                            "double x0 = (double)(int64_t)x, y0 = (double)(int64_t)y;"),
    "head_stride_wrong": ("const double* v = value + ((b * K + f.key[c]) * M + m) * D;\n                        const double s",
                          "const double* v = value + ((b * K + f.key[c]) * M) * D;\n                        const double s"),
}


def _battery_passes(lib) -> bool:
    """True when the mutant passes every pin in the battery."""
    for shapes, seed in ((((4, 6), (2, 3)), 3), (((7, 4), (3, 2), (2, 2), (1, 3)), 5)):
        wl = gen.random_workload(seed, 2, shapes, 2, 8, 3, 6)
        inp = gen.make_inputs(wl)
        args = (inp["value"], inp["spatial_shapes"], inp["level_start_index"],
                inp["sampling_locations"], inp["attention_weights"])
        for exact in (False, True):
            out = oracle.forward(*args, exact_coords=exact, lib=lib)
            if not np.allclose(out, tent.forward(*args, fp32_contract=not exact), rtol=1e-12,
                               atol=1e-12):
                return False
            got = oracle.backward(*args, inp["grad_output"], exact_coords=exact, lib=lib)
            want = tent.backward(*args, inp["grad_output"], fp32_contract=not exact)
            for a, b in zip(got, want):
                if not np.allclose(a, b, rtol=1e-11, atol=1e-11):
                    return False
    # key-index field at pixel centres
    shapes = ((8, 16), (4, 8), (1, 2))
    lsi = gen.level_start_index(shapes)
    K = gen.num_keys(shapes)
    rng = np.random.default_rng(9)
    M, D = 2, 8
    value = (np.arange(K)[None, :, None, None] + 1000.0 * np.arange(M)[None, None, :, None]
             + np.zeros((1, K, M, D)))
    loc = np.zeros((1, 4, M, 3, 1, 2), np.float32)
    w = np.zeros((1, 4, M, 3, 1), np.float32)
    w[:, :, :, 0, 0] = 1.0
    ix = rng.integers(0, 16, size=(1, 4, M))
    iy = rng.integers(0, 8, size=(1, 4, M))
    loc[:, :, :, 0, 0, 0] = (ix + 0.5) / 16
    loc[:, :, :, 0, 0, 1] = (iy + 0.5) / 8
    out = oracle.forward(value, np.array(shapes), lsi, loc, w, lib=lib).reshape(1, 4, M, D)
    want = (iy * 16 + ix + 1000.0 * np.arange(M)[None, None, :])[..., None]
    if not np.array_equal(out, np.broadcast_to(want, out.shape)):
        return False
    return True


def test_unmutated_oracle_passes_battery():
    assert _battery_passes(oracle.load())


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new)
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "mutant.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(so_path), str(c_path), "-lm"], check=True)
    lib = oracle.load(str(so_path))
    assert not _battery_passes(lib), f"mutation {name} slipped through every pin"
