"""Pins of the oracle's backward (the gradients of the forward definition)
against what calculus and the forward fix, independently of the backward code.

The forward is "TensorRT plugin walkthrough: modulatedDeformConvPlugin"
(trdm.cn), section 5 steps 1-3; that page has no backward, so the backward is
the gradient of sum(grad_out * forward) with the one-sided derivative on cell
edges (the reading stated in the oracle's C source).

  B1 finite differences of the (separately pinned) forward oracle, element by
     element for offset and mask and on sampled elements of x and weight. The
     forward is linear in x, mask, weight and bias, and linear in each single
     offset inside a bilinear cell, so a central difference whose step stays
     inside the cell is exact up to rounding.
  B2 adjoint identities: the forward is linear in x, in mask and in weight, so
     <grad_x, x> = <grad_mask, mask> = <grad_weight, weight>
     = sum(grad_out * (y - bias)); grad_bias is the sum of grad_out.
  B3 zero offsets and a unit mask reduce to an ordinary convolution: grad_x and
     grad_weight equal torch autograd of conv2d in float64, and grad_mask equals
     autograd of the same convolution written with unfold and a per-tap mask.
  B4 hand-worked samples and slopes (tests/golden/bilinear_slopes_2x2.json),
     including the right-hand slope at integer points and the zero border.
  B5 at integer offsets a one-sided forward difference of the forward equals
     the right-hand slope.
Finally, planted slips in the backward C code must each fail a pin.
"""
import json
import os
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F

HERE = os.path.dirname(os.path.abspath(__file__))

GEOMS = [
    dict(N=2, Cin=4, Cout=6, H=6, W=5, kh=3, kw=3, stride=(1, 1), padding=(1, 1), dilation=(1, 1), group=1, dg=2),
    dict(N=1, Cin=6, Cout=4, H=7, W=8, kh=3, kw=2, stride=(2, 1), padding=(2, 1), dilation=(2, 3), group=2, dg=3),
]


def off_grid_offsets(rng, shape, span=3):
    """Offsets whose fractional part lies in [0.1, 0.9]: every sampling point is
    at least 0.1 from a cell edge (anchors are integers)."""
    return rng.integers(-span, span + 1, shape).astype(np.float64) + rng.uniform(0.1, 0.9, shape)


def make_case(rng, geom, integer_offsets=False):
    g = dict(geom)
    N, Cin, Cout, H, W, kh, kw = (g[k] for k in ("N", "Cin", "Cout", "H", "W", "kh", "kw"))
    s, p, d = g["stride"], g["padding"], g["dilation"]
    Ho = (H + 2 * p[0] - d[0] * (kh - 1) - 1) // s[0] + 1
    Wo = (W + 2 * p[1] - d[1] * (kw - 1) - 1) // s[1] + 1
    K, dg, grp = kh * kw, g["dg"], g["group"]
    oshape = (N, 2 * dg * K, Ho, Wo)
    offset = rng.integers(-2, 3, oshape).astype(np.float64) if integer_offsets else off_grid_offsets(rng, oshape)
    return dict(
        x=rng.standard_normal((N, Cin, H, W)),
        offset=offset,
        mask=rng.uniform(0.1, 1.0, (N, dg * K, Ho, Wo)),
        weight=rng.standard_normal((Cout, Cin // grp, kh, kw)) / np.sqrt(Cin * K / grp),
        bias=rng.standard_normal(Cout) * 0.5,
        grad_out=rng.standard_normal((N, Cout, Ho, Wo)),
        attrs=dict(stride=s, padding=p, dilation=d, group=grp, deformable_group=dg),
    )


def loss(o, c, lib=None, **over):
    d = dict(c)
    d.update(over)
    y = o.forward(d["x"], d["offset"], d["mask"], d["weight"], d["bias"], nthreads=1, library=lib, **d["attrs"])
    return float(np.sum(d["grad_out"] * y))


def grads(o, c, lib=None):
    return o.backward(c["x"], c["offset"], c["mask"], c["weight"], c["grad_out"], nthreads=1, library=lib,
                      **c["attrs"])


def fd_check(o, c, g, name, idxs, step, lib=None):
    """Largest |central difference - gradient| over the listed flat indices,
    relative to the largest |gradient| of that input."""
    arr = c[name]
    worst = 0.0
    for e in idxs:
        a, b = arr.copy(), arr.copy()
        a.flat[e] += step
        b.flat[e] -= step
        fd = (loss(o, c, lib, **{name: a}) - loss(o, c, lib, **{name: b})) / (2 * step)
        worst = max(worst, abs(fd - g[name].flat[e]))
    return worst / max(np.max(np.abs(g[name])), 1e-300)


@pytest.mark.parametrize("gi", range(len(GEOMS)))
def test_b1_finite_differences(oracle_mod, gi):
    rng = np.random.default_rng(100 + gi)
    c = make_case(rng, GEOMS[gi])
    g = grads(oracle_mod, c)
    # every offset and mask element; the step 0.05 keeps each point in its cell
    assert fd_check(oracle_mod, c, g, "offset", range(c["offset"].size), 0.05) < 1e-10
    assert fd_check(oracle_mod, c, g, "mask", range(c["mask"].size), 0.05) < 1e-10
    for name in ("x", "weight", "bias"):
        n = c[name].size
        idxs = sorted(set(rng.integers(0, n, min(n, 60)).tolist()))
        assert fd_check(oracle_mod, c, g, name, idxs, 0.5) < 1e-10, name


@pytest.mark.parametrize("gi", range(len(GEOMS)))
def test_b2_adjoint_identities(oracle_mod, gi):
    rng = np.random.default_rng(200 + gi)
    c = make_case(rng, GEOMS[gi])
    g = grads(oracle_mod, c)
    y = oracle_mod.forward(c["x"], c["offset"], c["mask"], c["weight"], None, **c["attrs"])
    ref = float(np.sum(c["grad_out"] * y))
    scale = float(np.sum(np.abs(c["grad_out"] * y))) + 1e-300
    for name in ("x", "mask", "weight"):
        got = float(np.sum(g[name] * c[name]))
        assert abs(got - ref) < 1e-12 * scale, (name, got, ref)
    assert np.allclose(g["bias"], c["grad_out"].sum(axis=(0, 2, 3)), rtol=0, atol=1e-12)
    assert oracle_mod.backward(c["x"], c["offset"], c["mask"], c["weight"], c["grad_out"], with_bias=False,
                               **c["attrs"])["bias"] is None


def unfold_masked_conv(x, mask, weight, stride, padding, dilation, group, dg):
    """An ordinary convolution with a per-(tap, pixel, deformable group) scalar,
    written with torch's unfold (x at the integer tap positions)."""
    N, Cin, H, W = x.shape
    Cout, Cg, kh, kw = weight.shape
    K = kh * kw
    cols = F.unfold(x, (kh, kw), dilation=dilation, padding=padding, stride=stride)  # [N, Cin*K, P]
    P = cols.shape[-1]
    cols = cols.view(N, dg, Cin // dg, K, P) * mask.view(N, dg, 1, K, P)
    cols = cols.reshape(N, group, Cg * K, P)
    wg = weight.reshape(group, Cout // group, Cg * K)
    return torch.einsum("gok,ngkp->ngop", wg, cols).reshape(N, Cout, P)


@pytest.mark.parametrize("gi", range(len(GEOMS)))
def test_b3_zero_offsets_reduce_to_conv2d(oracle_mod, gi):
    rng = np.random.default_rng(300 + gi)
    c = make_case(rng, GEOMS[gi])
    c["offset"][:] = 0.0
    c["mask"][:] = 1.0
    a = c["attrs"]
    g = grads(oracle_mod, c)
    x = torch.from_numpy(c["x"]).requires_grad_()
    w = torch.from_numpy(c["weight"]).requires_grad_()
    b = torch.from_numpy(c["bias"]).requires_grad_()
    y = F.conv2d(x, w, b, stride=a["stride"], padding=a["padding"], dilation=a["dilation"], groups=a["group"])
    y.backward(torch.from_numpy(c["grad_out"]))
    assert np.allclose(g["x"], x.grad.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(g["weight"], w.grad.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(g["bias"], b.grad.numpy(), rtol=0, atol=1e-12)
    m = torch.from_numpy(c["mask"]).requires_grad_()
    y2 = unfold_masked_conv(torch.from_numpy(c["x"]), m, torch.from_numpy(c["weight"]), a["stride"], a["padding"],
                            a["dilation"], a["group"], a["deformable_group"])
    assert np.allclose(y2.detach().numpy().reshape(y.shape), y.detach().numpy() - c["bias"][None, :, None, None],
                       rtol=0, atol=1e-12)
    y2.backward(torch.from_numpy(c["grad_out"]).reshape(y2.shape))
    assert np.allclose(g["mask"], m.grad.numpy(), rtol=0, atol=1e-12)


def golden_slopes():
    return json.load(open(os.path.join(HERE, "golden", "bilinear_slopes_2x2.json")))


def check_golden(o, lib=None):
    """Returns the list of golden cases that fail."""
    gold = golden_slopes()
    x = np.array(gold["x"], dtype=np.float64)[None, None]
    bad = []
    for i, case in enumerate(gold["cases"]):
        off = np.zeros((1, 2, 2, 2))
        msk = np.full((1, 1, 2, 2), 0.7)
        ho, wo = case["ho"], case["wo"]
        off[0, 0, ho, wo], off[0, 1, ho, wo], msk[0, 0, ho, wo] = case["dh"], case["dw"], case["mask"]
        go = np.zeros((1, 1, 2, 2))
        go[0, 0, ho, wo] = 1.0
        g = o.backward(x, off, msk, np.ones((1, 1, 1, 1)), go, nthreads=1, library=lib)
        m = case["mask"]
        ok = (abs(g["mask"][0, 0, ho, wo] - case["v"]) < 1e-12
              and abs(g["offset"][0, 0, ho, wo] - m * case["dvdh"]) < 1e-12
              and abs(g["offset"][0, 1, ho, wo] - m * case["dvdw"]) < 1e-12
              and np.allclose(g["x"][0, 0], np.array(case["grad_x"]), rtol=0, atol=1e-12)
              and abs(g["weight"][0, 0, 0, 0] - m * case["v"]) < 1e-12
              and abs(g["bias"][0] - 1.0) < 1e-12)
        # the other pixels get no gradient (grad_out is 0 there)
        rest = np.ones((2, 2), bool)
        rest[ho, wo] = False
        ok = ok and not np.any(g["offset"][0][:, rest]) and not np.any(g["mask"][0][:, rest])
        if not ok:
            bad.append(i)
    return bad


def test_b4_golden_slopes(oracle_mod):
    assert check_golden(oracle_mod) == []


@pytest.mark.parametrize("gi", range(len(GEOMS)))
def test_b5_right_hand_slope_at_integer_points(oracle_mod, gi):
    rng = np.random.default_rng(500 + gi)
    c = make_case(rng, GEOMS[gi], integer_offsets=True)
    g = grads(oracle_mod, c)
    idxs = sorted(set(rng.integers(0, c["offset"].size, 120).tolist()))
    step = 0.125
    base = loss(oracle_mod, c)
    scale = np.max(np.abs(g["offset"]))
    a_ = c["attrs"]
    kw, K = GEOMS[gi]["kw"], GEOMS[gi]["kh"] * GEOMS[gi]["kw"]
    Ho, Wo = c["offset"].shape[2:]
    for e in idxs:
        # a point exactly on h = -1 or w = -1 is outside the open range, where
        # the sample and its slopes are 0 (the forward's range test), though
        # the sample grows to the right of it: that point is not compared here
        n, ch, ho, wo = np.unravel_index(e, c["offset"].shape)
        k = (ch % (2 * K)) // 2
        base_ch = ch - (ch % 2)
        h = ho * a_["stride"][0] - a_["padding"][0] + (k // kw) * a_["dilation"][0] + c["offset"][n, base_ch, ho, wo]
        w = wo * a_["stride"][1] - a_["padding"][1] + (k % kw) * a_["dilation"][1] + c["offset"][n, base_ch + 1, ho, wo]
        if h == -1 or w == -1:
            assert g["offset"].flat[e] == 0.0
            continue
        a = c["offset"].copy()
        a.flat[e] += step
        fd = (loss(oracle_mod, c, offset=a) - base) / step
        assert abs(fd - g["offset"].flat[e]) < 1e-10 * scale, e


# ----------------------------------------------------------------------------- planted slips
BACKWARD_MUTATIONS = {
    "slope_h_sign": [("*dvdh += (dy ? 1.0 : -1.0) * wx * X;", "*dvdh += (dy ? -1.0 : 1.0) * wx * X;")],
    "slope_w_uses_wx": [("*dvdw += (dx ? 1.0 : -1.0) * wy * X;", "*dvdw += (dx ? 1.0 : -1.0) * wx * X;")],
    "grad_x_without_mask": [("gcol[((n * Cin + c) * K + k) * P + p] * MASK(n, gd, k, p);",
                             "gcol[((n * Cin + c) * K + k) * P + p];")],
    "grad_offset_without_mask": [("s_h += G * m * dvdh;", "s_h += G * dvdh;")],
    "grad_offset_h_w_swapped": [("s_h += G * m * dvdh;", "s_h += G * m * dvdw;"),
                                ("s_w += G * m * dvdw;", "s_w += G * m * dvdh;")],
    "grad_mask_with_mask": [("s_mask += G * v;", "s_mask += G * m * v;")],
    "grad_weight_without_mask": [("col[e] = MASK(n, gd, k, p) * v;", "col[e] = v;")],
    "grad_col_wrong_tap": [("G += weight[(o * Cg + cl) * K + k] * grad_out", "G += weight[(o * Cg + cl) * K] * grad_out")],
    "grad_x_corner_weight_flipped": [("const double wx = dx ? cc.lw : 1.0 - cc.lw;",
                                      "const double wx = dx ? 1.0 - cc.lw : cc.lw;")],
    "closed_range_inside": [("c.inside = !(h <= -1.0 || h >= (double)H || w <= -1.0 || w >= (double)W);",
                             "c.inside = !(h < -1.0 || h > (double)H || w < -1.0 || w > (double)W);")],
}


def backward_pins(o, lib):
    failed = []
    if check_golden(o, lib):
        failed.append("B4")
    rng = np.random.default_rng(77)
    c = make_case(rng, GEOMS[1])
    g = grads(o, c, lib)
    if fd_check(o, c, g, "offset", range(0, c["offset"].size, 3), 0.05) > 1e-10:
        failed.append("B1 offset")
    y = o.forward(c["x"], c["offset"], c["mask"], c["weight"], None, **c["attrs"])
    ref = float(np.sum(c["grad_out"] * y))
    for name in ("x", "mask", "weight"):
        if abs(float(np.sum(g[name] * c[name])) - ref) > 1e-10 * abs(ref):
            failed.append("B2 " + name)
    return failed


def test_unmodified_backward_passes_compact_pins(oracle_mod):
    assert backward_pins(oracle_mod, None) == []


@pytest.mark.parametrize("name", sorted(BACKWARD_MUTATIONS))
def test_planted_backward_slip_is_caught(oracle_mod, name, tmp_path):
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "mdcn_oracle.c")).read()
    for old, new in BACKWARD_MUTATIONS[name]:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    cpath = tmp_path / "mutant.c"
    cpath.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so),
                    str(cpath), "-lm"], check=True)
    lib = oracle_mod.load_library(str(so))
    assert backward_pins(oracle_mod, lib), f"planted slip {name} passed every pin"


# ---------------------------------------------------------- fp32 positions (the kernels' cell decision)
def test_b6_fp32_positions_agree_away_from_edges(oracle_mod):
    """positions="f32" only rounds anchor + offset to fp32: away from cell
    edges it matches finite differences of the forward to fp32 position
    rounding, and on the hand-worked cases (positions exact in fp32) it is
    identical to the exact gradient."""
    rng = np.random.default_rng(600)
    c = make_case(rng, GEOMS[1])
    g32 = oracle_mod.backward(c["x"], c["offset"], c["mask"], c["weight"], c["grad_out"], positions="f32",
                              **c["attrs"])
    g64 = grads(oracle_mod, c)
    for name in ("x", "offset", "mask", "weight", "bias"):
        assert np.abs(g32[name] - g64[name]).max() <= 1e-5 * np.abs(g64[name]).max(), name
    assert fd_check(oracle_mod, c, g32, "offset", range(0, c["offset"].size, 5), 0.05) < 1e-5
    gold = golden_slopes()
    x = np.array(gold["x"], dtype=np.float64)[None, None]
    for case in gold["cases"]:
        off = np.zeros((1, 2, 2, 2))
        off[0, 0, case["ho"], case["wo"]], off[0, 1, case["ho"], case["wo"]] = case["dh"], case["dw"]
        msk = np.full((1, 1, 2, 2), case["mask"])
        go = np.ones((1, 1, 2, 2))
        a = oracle_mod.backward(x, off, msk, np.ones((1, 1, 1, 1)), go, positions="f32")
        b = oracle_mod.backward(x, off, msk, np.ones((1, 1, 1, 1)), go)
        for name in a:
            assert np.array_equal(a[name], b[name]), name


def test_b7_fp32_position_on_a_cell_edge(oracle_mod):
    """Hand-worked: x[y, 0] = y^2 on a 40 x 2 plane, 1x1 weight 1, output pixel
    (38, 0) with offset (-1.4e-6, 0). Exactly, h = 37.9999986 lies in cell 37,
    slope X(38) - X(37) = 1444 - 1369 = 75; in fp32, 38 - 1.4e-6 rounds to 38.0
    (half an ulp there is 1.9e-6), the right-hand slope X(39) - X(38) = 1521 -
    1444 = 77. Both are scaled by the mask 0.5."""
    H, W = 40, 2
    x = np.zeros((1, 1, H, W))
    x[0, 0, :, 0] = np.arange(H, dtype=np.float64) ** 2
    off = np.zeros((1, 2, H, W))
    off[0, 0, 38, 0] = -1.4e-6
    msk = np.full((1, 1, H, W), 0.5)
    go = np.zeros((1, 1, H, W))
    go[0, 0, 38, 0] = 1.0
    g64 = oracle_mod.backward(x, off, msk, np.ones((1, 1, 1, 1)), go)
    g32 = oracle_mod.backward(x, off, msk, np.ones((1, 1, 1, 1)), go, positions="f32")
    assert abs(g64["offset"][0, 0, 38, 0] - 0.5 * 75.0) < 1e-9
    assert abs(g32["offset"][0, 0, 38, 0] - 0.5 * 77.0) < 1e-12
    assert abs(g32["mask"][0, 0, 38, 0] - 1444.0) < 1e-12  # the sample at h = 38 exactly
    with pytest.raises(ValueError):
        oracle_mod.backward(x, off, msk, np.ones((1, 1, 1, 1)), go, positions="f16")
