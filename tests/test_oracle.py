"""Pins of the double-precision oracle against what the operator's definition
fixes, independently of the oracle's own code.

Definition: "TensorRT plugin walkthrough: modulatedDeformConvPlugin"
(trdm.cn), section 2 (layouts, output shape), section 3 (attributes),
section 5 steps 1-3 (deformable im2col with bilinear sampling and mask,
grouped GEMM, bias).

Each pin is chosen so that a plausible slip in the oracle fails it:
  P1 zero offsets + unit mask = ordinary grouped/strided/padded/dilated
     convolution (torch conv2d in float64, and a brute-force loop).
  P2 integer offsets = convolution of a shifted, zero-extended image; per-tap
     integer offsets = plain pixel gathers (fixes the h-then-w order).
  P3 mask = 0 gives the bias; mask scaling; a one-hot mask isolates one tap
     (fixes the mask channel order).
  P4 deformable groups are contiguous channel blocks.
  P5 an independent restatement (bilinear interpolation of a zero-padded
     image, no range tests) agrees on random fractional offsets.
  P6 hand-computed bilinear values (tests/golden/bilinear_2x2.json).
  P7 output shape from x, weight and offset; rejected arguments.
  P8 linearity in x and in weight.
  P9 group = g equals g independent single-group calls.
Finally, broken copies of the C source (planted slips) must each fail a pin.
"""
import json
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch
import torch.nn.functional as F

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def make_case(rng, N=1, Cin=4, Cout=4, H=7, W=6, kh=3, kw=3, stride=(1, 1), padding=(1, 1),
              dilation=(1, 1), group=1, dg=1, bias=True, off_scale=1.5, Ho=None, Wo=None):
    if Ho is None:
        Ho = (H + 2 * padding[0] - dilation[0] * (kh - 1) - 1) // stride[0] + 1
    if Wo is None:
        Wo = (W + 2 * padding[1] - dilation[1] * (kw - 1) - 1) // stride[1] + 1
    K = kh * kw
    return dict(
        x=rnd(rng, N, Cin, H, W),
        offset=rnd(rng, N, 2 * dg * K, Ho, Wo, scale=off_scale),
        mask=rng.uniform(0.0, 1.0, (N, dg * K, Ho, Wo)),
        weight=rnd(rng, Cout, Cin // group, kh, kw, scale=1.0 / math.sqrt(Cin * K / group)),
        bias=rnd(rng, Cout, scale=0.5) if bias else None,
        attrs=dict(stride=stride, padding=padding, dilation=dilation, group=group, deformable_group=dg),
    )


def run(oracle_mod, c, **over):
    d = dict(c)
    d.update(over)
    attrs = d.pop("attrs")
    lib = d.pop("library", None)
    return oracle_mod.forward(d["x"], d["offset"], d["mask"], d["weight"], d["bias"], library=lib, **attrs)


def conv_ref(x, weight, bias, stride, padding, dilation, group):
    y = F.conv2d(torch.from_numpy(x), torch.from_numpy(weight),
                 None if bias is None else torch.from_numpy(bias),
                 stride=stride, padding=padding, dilation=dilation, groups=group)
    return y.numpy()


def zero_extended_restatement(x, offset, mask, weight, bias, stride, padding, dilation, group, dg):
    """Independent restatement: pad x with enough zeros that every sampled
    point and its four corners fall inside, then interpolate bilinearly with no
    range test at all. Vectorised numpy; shares nothing with the C oracle."""
    N, Cin, H, W = x.shape
    Cout, Cg, kh, kw = weight.shape
    Ho, Wo = offset.shape[2:]
    K = kh * kw
    Cd = Cin // dg
    Og = Cout // group
    big = int(np.ceil(np.abs(offset).max())) + 2
    M = big + max(padding) + max(dilation) * (max(kh, kw) - 1) + max(stride) * max(Ho, Wo) + 2
    xp = np.pad(x, ((0, 0), (0, 0), (M, M), (M, M)))
    cols = np.zeros((N, Cin, K, Ho, Wo))
    ho = np.arange(Ho)[:, None]
    wo = np.arange(Wo)[None, :]
    for gd in range(dg):
        for i in range(kh):
            for j in range(kw):
                k = i * kw + j
                hh = ho * stride[0] - padding[0] + i * dilation[0] + offset[:, gd * 2 * K + 2 * k] + M
                ww = wo * stride[1] - padding[1] + j * dilation[1] + offset[:, gd * 2 * K + 2 * k + 1] + M
                h0 = np.floor(hh).astype(np.int64)
                w0 = np.floor(ww).astype(np.int64)
                lh, lw = hh - h0, ww - w0
                m = mask[:, gd * K + k]
                for n in range(N):
                    blk = xp[n, gd * Cd:(gd + 1) * Cd]
                    v = ((1 - lh[n]) * (1 - lw[n]) * blk[:, h0[n], w0[n]]
                         + (1 - lh[n]) * lw[n] * blk[:, h0[n], w0[n] + 1]
                         + lh[n] * (1 - lw[n]) * blk[:, h0[n] + 1, w0[n]]
                         + lh[n] * lw[n] * blk[:, h0[n] + 1, w0[n] + 1])
                    cols[n, gd * Cd:(gd + 1) * Cd, k] = m[n] * v
    y = np.zeros((N, Cout, Ho, Wo))
    for g in range(group):
        wg = weight[g * Og:(g + 1) * Og].reshape(Og, Cg, K)
        cg = cols[:, g * Cg:(g + 1) * Cg]
        y[:, g * Og:(g + 1) * Og] = np.einsum("ock,nckhw->nohw", wg, cg)
    if bias is not None:
        y += bias[None, :, None, None]
    return y


# ----------------------------------------------------------------------------- P6
def test_p6_golden_bilinear(oracle_mod):
    g = json.load(open(os.path.join(HERE, "golden", "bilinear_2x2.json")))
    x = np.array(g["x"], dtype=np.float64)[None, None]
    w = np.full((1, 1, 1, 1), g["weight_1x1"])
    for case in g["cases"]:
        off = np.zeros((1, 2, 2, 2))
        msk = np.ones((1, 1, 2, 2))
        off[0, 0, case["ho"], case["wo"]] = case["dh"]
        off[0, 1, case["ho"], case["wo"]] = case["dw"]
        msk[0, 0, case["ho"], case["wo"]] = case["mask"]
        y = oracle_mod.forward(x, off, msk, w, None, stride=g["stride"], padding=g["padding"],
                               dilation=g["dilation"])
        assert y[0, 0, case["ho"], case["wo"]] == pytest.approx(case["expected"], abs=1e-14), case


# ----------------------------------------------------------------------------- P1
P1_SWEEP = [
    dict(kh=3, kw=3, stride=(1, 1), padding=(1, 1), dilation=(1, 1), group=1, dg=1),
    dict(kh=3, kw=3, stride=(2, 2), padding=(2, 2), dilation=(2, 2), group=4, dg=2),
    dict(kh=1, kw=1, stride=(1, 1), padding=(0, 0), dilation=(1, 1), group=2, dg=1),
    dict(kh=5, kw=3, stride=(2, 1), padding=(2, 1), dilation=(1, 2), group=2, dg=4),
    dict(kh=3, kw=3, stride=(1, 2), padding=(0, 3), dilation=(2, 1), group=1, dg=2),
    dict(kh=2, kw=4, stride=(3, 2), padding=(1, 0), dilation=(1, 1), group=8, dg=8),  # depthwise
]


@pytest.mark.parametrize("p", P1_SWEEP)
@pytest.mark.parametrize("bias", [True, False])
def test_p1_zero_offset_unit_mask_is_conv2d(oracle_mod, p, bias):
    rng = np.random.default_rng(11)
    c = make_case(rng, N=2, Cin=8, Cout=8, H=9, W=11, kh=p["kh"], kw=p["kw"], stride=p["stride"],
                  padding=p["padding"], dilation=p["dilation"], group=p["group"], dg=p["dg"], bias=bias)
    c["offset"][:] = 0.0
    c["mask"][:] = 1.0
    y = run(oracle_mod, c)
    ref = conv_ref(c["x"], c["weight"], c["bias"], p["stride"], p["padding"], p["dilation"], p["group"])
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


def test_p1_brute_force_conv(oracle_mod):
    """A seven-loop direct convolution written here, no library."""
    rng = np.random.default_rng(3)
    c = make_case(rng, N=1, Cin=4, Cout=2, H=5, W=4, stride=(2, 1), padding=(1, 2), dilation=(1, 2), group=2)
    c["offset"][:] = 0.0
    c["mask"][:] = 1.0
    y = run(oracle_mod, c)
    x, wt, b = c["x"], c["weight"], c["bias"]
    N, Cin, H, W = x.shape
    Cout, Cg, kh, kw = wt.shape
    _, _, Ho, Wo = y.shape
    ref = np.zeros_like(y)
    for n in range(N):
        for o in range(Cout):
            g = o // (Cout // 2)
            for ho in range(Ho):
                for wo in range(Wo):
                    s = b[o]
                    for cl in range(Cg):
                        for i in range(kh):
                            for j in range(kw):
                                hh = ho * 2 - 1 + i * 1
                                ww = wo * 1 - 2 + j * 2
                                if 0 <= hh < H and 0 <= ww < W:
                                    s += wt[o, cl, i, j] * x[n, g * Cg + cl, hh, ww]
                    ref[n, o, ho, wo] = s
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- P2
def shifted_conv(x, weight, bias, stride, padding, dilation, group, a, b):
    """conv2d of the zero-extended image shifted by (a, b): out[ho, wo] reads
    x[ho*s - p + i*d + a, wo*s - p + j*d + b] (0 outside)."""
    N, C, H, W = x.shape
    kh, kw = weight.shape[2:]
    Ho = (H + 2 * padding[0] - dilation[0] * (kh - 1) - 1) // stride[0] + 1
    Wo = (W + 2 * padding[1] - dilation[1] * (kw - 1) - 1) // stride[1] + 1
    M = padding[0] + padding[1] + abs(a) + abs(b) + 2
    xp = np.pad(x, ((0, 0), (0, 0), (M, M + H), (M, M + W)))
    h0 = M - padding[0] + a
    w0 = M - padding[1] + b
    crop = np.ascontiguousarray(xp[:, :, h0:, w0:])
    y = conv_ref(crop, weight, bias, stride, (0, 0), dilation, group)
    return y[:, :, :Ho, :Wo]


@pytest.mark.parametrize("ab", [(1, 0), (0, 1), (2, -1), (-3, 2), (1, 3)])
def test_p2_constant_integer_offset_is_shifted_conv(oracle_mod, ab):
    a, b = ab
    rng = np.random.default_rng(5)
    c = make_case(rng, N=2, Cin=6, Cout=4, H=8, W=7, stride=(2, 1), padding=(1, 2), dilation=(1, 2),
                  group=2, dg=3)
    c["offset"][:, 0::2] = a
    c["offset"][:, 1::2] = b
    c["mask"][:] = 1.0
    y = run(oracle_mod, c)
    ref = shifted_conv(c["x"], c["weight"], c["bias"], (2, 1), (1, 2), (1, 2), 2, a, b)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


def test_p2_per_tap_integer_offsets_are_gathers(oracle_mod):
    """Each tap k gets its own integer (a_k, b_k); the output must be the sum
    of plain pixel reads x[ho - p + i + a_k, wo - p + j + b_k] (0 outside)."""
    rng = np.random.default_rng(9)
    c = make_case(rng, N=1, Cin=3, Cout=2, H=6, W=5, bias=False)
    K = 9
    ab = rng.integers(-3, 4, size=(K, 2))
    for k in range(K):
        c["offset"][:, 2 * k] = ab[k, 0]
        c["offset"][:, 2 * k + 1] = ab[k, 1]
    c["mask"][:] = 1.0
    y = run(oracle_mod, c)
    x, wt = c["x"], c["weight"]
    H, W = x.shape[2:]
    ref = np.zeros_like(y)
    for o in range(2):
        for ho in range(y.shape[2]):
            for wo in range(y.shape[3]):
                s = 0.0
                for cc in range(3):
                    for i in range(3):
                        for j in range(3):
                            k = i * 3 + j
                            hh, ww = ho - 1 + i + ab[k, 0], wo - 1 + j + ab[k, 1]
                            if 0 <= hh < H and 0 <= ww < W:
                                s += wt[o, cc, i, j] * x[0, cc, hh, ww]
                ref[0, o, ho, wo] = s
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- P3
def test_p3_zero_mask_gives_bias(oracle_mod):
    rng = np.random.default_rng(1)
    c = make_case(rng, N=2, Cin=4, Cout=6, group=2, dg=2)
    c["mask"][:] = 0.0
    y = run(oracle_mod, c)
    np.testing.assert_array_equal(y, np.broadcast_to(c["bias"][None, :, None, None], y.shape))


def test_p3_mask_scaling(oracle_mod):
    rng = np.random.default_rng(2)
    c = make_case(rng, N=1, Cin=4, Cout=4, dg=2)
    y1 = run(oracle_mod, c)
    y2 = run(oracle_mod, c, mask=c["mask"] * 0.375)
    b = c["bias"][None, :, None, None]
    np.testing.assert_allclose(y2 - b, (y1 - b) * 0.375, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("k", [0, 1, 4, 5, 7])
def test_p3_one_hot_mask_isolates_tap(oracle_mod, k):
    """Zero offsets, mask = 1 on tap k only: equals conv2d with every other tap
    of the weight zeroed. Tap k = i*kw + j (row-major)."""
    rng = np.random.default_rng(4)
    kh, kw = 3, 3
    c = make_case(rng, N=1, Cin=4, Cout=3, H=6, W=8, kh=kh, kw=kw, bias=False)
    c["offset"][:] = 0.0
    c["mask"][:] = 0.0
    c["mask"][:, k] = 1.0
    y = run(oracle_mod, c)
    wk = np.zeros_like(c["weight"])
    wk[:, :, k // kw, k % kw] = c["weight"][:, :, k // kw, k % kw]
    ref = conv_ref(c["x"], wk, None, (1, 1), (1, 1), (1, 1), 1)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


def test_p3_mask_channel_per_deformable_group(oracle_mod):
    """dg = 2: mask = 1 only on group-1 block (channels K..2K-1) -> only input
    channels of the second half contribute."""
    rng = np.random.default_rng(6)
    c = make_case(rng, N=1, Cin=4, Cout=2, dg=2, bias=False)
    K = 9
    c["mask"][:, :K] = 0.0
    y = run(oracle_mod, c)
    x2 = c["x"].copy()
    x2[:, :2] = 0.0
    m2 = c["mask"].copy()
    m2[:, :K] = 1.0  # whatever block 0 does, its channels are zero now
    ref = run(oracle_mod, c, x=x2, mask=m2)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- P4
def test_p4_identical_blocks_equal_single_group(oracle_mod):
    rng = np.random.default_rng(7)
    c1 = make_case(rng, N=2, Cin=8, Cout=4, dg=1)
    dg = 4
    off = np.concatenate([c1["offset"]] * dg, axis=1)
    msk = np.concatenate([c1["mask"]] * dg, axis=1)
    y1 = run(oracle_mod, c1)
    attrs = dict(c1["attrs"], deformable_group=dg)
    y4 = run(oracle_mod, c1, offset=off, mask=msk, attrs=attrs)
    np.testing.assert_allclose(y4, y1, rtol=0, atol=1e-13)


def test_p4_blocks_are_contiguous_channels(oracle_mod):
    """Perturbing the offsets of deformable group gd changes only the
    contribution of input channels [gd*Cd, (gd+1)*Cd)."""
    rng = np.random.default_rng(8)
    dg, Cin = 2, 8
    Cd = Cin // dg
    K = 9
    c = make_case(rng, N=1, Cin=Cin, Cout=3, dg=dg, bias=False)
    gd = 1
    off2 = c["offset"].copy()
    off2[:, gd * 2 * K:(gd + 1) * 2 * K] += rng.standard_normal(off2[:, gd * 2 * K:(gd + 1) * 2 * K].shape)
    diff = run(oracle_mod, c, offset=off2) - run(oracle_mod, c)
    # the same difference through a dg = 1 call on the block's channels alone
    xb = np.zeros_like(c["x"])
    xb[:, gd * Cd:(gd + 1) * Cd] = c["x"][:, gd * Cd:(gd + 1) * Cd]
    a1 = dict(c["attrs"], deformable_group=1)
    blk = slice(gd * 2 * K, (gd + 1) * 2 * K)
    mb = c["mask"][:, gd * K:(gd + 1) * K]
    d1 = (run(oracle_mod, c, x=xb, offset=off2[:, blk], mask=mb, attrs=a1)
          - run(oracle_mod, c, x=xb, offset=c["offset"][:, blk], mask=mb, attrs=a1))
    assert np.abs(diff).max() > 1e-3
    np.testing.assert_allclose(diff, d1, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- P5
P5_SWEEP = [
    dict(N=2, Cin=4, Cout=4, H=7, W=6, kh=3, kw=3, stride=(1, 1), padding=(1, 1), dilation=(1, 1), group=1, dg=1, off_scale=1.5),
    dict(N=1, Cin=8, Cout=4, H=9, W=9, kh=3, kw=3, stride=(2, 2), padding=(2, 2), dilation=(2, 2), group=4, dg=2, off_scale=8.0),
    dict(N=2, Cin=6, Cout=6, H=5, W=8, kh=5, kw=3, stride=(1, 2), padding=(2, 0), dilation=(1, 1), group=3, dg=3, off_scale=3.0),
    dict(N=1, Cin=4, Cout=8, H=4, W=4, kh=1, kw=1, stride=(1, 1), padding=(0, 0), dilation=(1, 1), group=1, dg=4, off_scale=2.0),
    dict(N=1, Cin=2, Cout=2, H=3, W=3, kh=3, kw=3, stride=(1, 1), padding=(1, 1), dilation=(1, 1), group=1, dg=1, off_scale=20.0),
]


@pytest.mark.parametrize("p", P5_SWEEP)
def test_p5_zero_extended_restatement(oracle_mod, p):
    rng = np.random.default_rng(12)
    p = dict(p)
    c = make_case(rng, **p)
    # include exact integer and half-integer points and the -1 / H edges
    c["offset"].flat[::7] = np.round(c["offset"].flat[::7])
    c["offset"].flat[3::11] = np.round(c["offset"].flat[3::11] * 2) / 2
    y = run(oracle_mod, c)
    a = c["attrs"]
    ref = zero_extended_restatement(c["x"], c["offset"], c["mask"], c["weight"], c["bias"], a["stride"],
                                    a["padding"], a["dilation"], a["group"], a["deformable_group"])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_p5_far_outside_is_zero(oracle_mod):
    rng = np.random.default_rng(13)
    c = make_case(rng, N=1, Cin=2, Cout=2, H=4, W=4, bias=True)
    c["offset"][:, 0::2] = 1e6
    y = run(oracle_mod, c)
    np.testing.assert_array_equal(y, np.broadcast_to(c["bias"][None, :, None, None], y.shape))


# ----------------------------------------------------------------------------- P7
def test_p7_output_shape_from_offset(oracle_mod):
    """Ho, Wo come from offset's dims 2 and 3, whatever the convolution formula
    would give; N from x, Cout from weight."""
    rng = np.random.default_rng(14)
    c = make_case(rng, N=3, Cin=4, Cout=5, H=6, W=6, Ho=2, Wo=9)
    y = run(oracle_mod, c)
    assert y.shape == (3, 5, 2, 9)
    a = c["attrs"]
    ref = zero_extended_restatement(c["x"], c["offset"], c["mask"], c["weight"], c["bias"], a["stride"],
                                    a["padding"], a["dilation"], a["group"], a["deformable_group"])
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("bad", [
    dict(stride=(0, 1)), dict(dilation=(1, 0)), dict(padding=(-1, 0)), dict(group=0), dict(deformable_group=0),
])
def test_p7_attribute_ranges(oracle_mod, bad):
    rng = np.random.default_rng(15)
    c = make_case(rng)
    with pytest.raises(ValueError):
        run(oracle_mod, c, attrs=dict(c["attrs"], **bad))


def test_p7_shape_bindings(oracle_mod):
    rng = np.random.default_rng(16)
    c = make_case(rng, N=2, Cin=4, Cout=4, dg=2)
    with pytest.raises(ValueError):  # offset batch != x batch
        run(oracle_mod, c, offset=c["offset"][:1])
    with pytest.raises(ValueError):  # mask spatial != offset spatial
        run(oracle_mod, c, mask=c["mask"][:, :, :-1])
    with pytest.raises(ValueError):  # offset channels != 2*dg*K
        run(oracle_mod, c, offset=c["offset"][:, :-2])
    with pytest.raises(ValueError):  # mask channels != dg*K
        run(oracle_mod, c, mask=c["mask"][:, :-1])
    with pytest.raises(ValueError):  # bias length != Cout
        run(oracle_mod, c, bias=c["bias"][:-1])
    with pytest.raises(ValueError):  # dg does not divide Cin
        run(oracle_mod, c, attrs=dict(c["attrs"], deformable_group=3),
            offset=np.zeros((2, 54, 7, 6)), mask=np.zeros((2, 27, 7, 6)))


# ----------------------------------------------------------------------------- P8
def test_p8_linearity(oracle_mod):
    rng = np.random.default_rng(17)
    c = make_case(rng, N=1, Cin=4, Cout=4, group=2, dg=2)
    b = c["bias"][None, :, None, None]
    x1, x2 = c["x"], rnd(rng, *c["x"].shape)
    y1, y2 = run(oracle_mod, c, x=x1) - b, run(oracle_mod, c, x=x2) - b
    y12 = run(oracle_mod, c, x=2.5 * x1 - 0.75 * x2) - b
    np.testing.assert_allclose(y12, 2.5 * y1 - 0.75 * y2, rtol=1e-12, atol=1e-12)
    w1, w2 = c["weight"], rnd(rng, *c["weight"].shape)
    z1, z2 = run(oracle_mod, c, weight=w1) - b, run(oracle_mod, c, weight=w2) - b
    z12 = run(oracle_mod, c, weight=-1.5 * w1 + 3.0 * w2) - b
    np.testing.assert_allclose(z12, -1.5 * z1 + 3.0 * z2, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------------------- P9
def test_p9_group_decomposition(oracle_mod):
    rng = np.random.default_rng(18)
    g, Cin, Cout = 4, 8, 12
    c = make_case(rng, N=2, Cin=Cin, Cout=Cout, group=g, dg=2)
    y = run(oracle_mod, c)
    Cg, Og = Cin // g, Cout // g
    K = 9
    Cd = Cin // 2
    parts = []
    for gi in range(g):
        chans = slice(gi * Cg, (gi + 1) * Cg)
        gd = (gi * Cg) // Cd  # each group lies inside one deformable group here
        a = dict(c["attrs"], group=1, deformable_group=1)
        parts.append(run(oracle_mod, c, x=c["x"][:, chans], weight=c["weight"][gi * Og:(gi + 1) * Og],
                         bias=c["bias"][gi * Og:(gi + 1) * Og],
                         offset=c["offset"][:, gd * 2 * K:(gd + 1) * 2 * K],
                         mask=c["mask"][:, gd * K:(gd + 1) * K], attrs=a))
    np.testing.assert_allclose(y, np.concatenate(parts, axis=1), rtol=0, atol=1e-13)


# ----------------------------------------------------------------------------- planted slips
MUTATIONS = {
    "swap_h_w_offset": [("const int64_t och_h = gd * 2 * K + 2 * k;", "const int64_t och_h = gd * 2 * K + 2 * k + 1;"),
                        ("const int64_t och_w = och_h + 1;", "const int64_t och_w = och_h - 1;")],
    "swap_bilinear_weight": [("const double wy = dy ? lh : 1.0 - lh;", "const double wy = dy ? 1.0 - lh : lh;")],
    "interleaved_deformable_groups": [("const int64_t gd = c / Cd;", "const int64_t gd = c % deformable_group;")],
    "mask_tap_major": [("const int64_t mch = gd * K + k;", "const int64_t mch = k * deformable_group + gd;")],
    "group_channel_base_dropped": [("const int64_t c = g * Cg + cl;", "const int64_t c = cl;")],
    "bias_dropped": [("if (bias) acc += bias[o];", "(void)bias;")],
    "stride_for_dilation": [("+ i * dil_h", "+ i * stride_h")],
    "replicate_border": [("if (y < 0 || y >= H || xx < 0 || xx >= W) continue;",
                          "const int64_t y2 = y < 0 ? 0 : (y >= H ? H - 1 : y); const int64_t x2 = xx < 0 ? 0 : (xx >= W ? W - 1 : xx); v += (dy ? lh : 1.0 - lh) * (dx ? lw : 1.0 - lw) * plane[y2 * W + x2]; continue;")],
    "offset_dropped_h": [("+ dh;", "+ 0.0 * dh;")],
}


def all_pins(oracle_mod, lib):
    """Re-run a compact set of the pins against a given build; return the
    names of the pins that fail."""
    failed = []
    o = oracle_mod

    def fwd(c, **over):
        return run(o, c, library=lib, **over)

    rng = np.random.default_rng(21)
    # P6
    g = json.load(open(os.path.join(HERE, "golden", "bilinear_2x2.json")))
    x = np.array(g["x"], dtype=np.float64)[None, None]
    for case in g["cases"]:
        off = np.zeros((1, 2, 2, 2))
        msk = np.ones((1, 1, 2, 2))
        off[0, 0, case["ho"], case["wo"]] = case["dh"]
        off[0, 1, case["ho"], case["wo"]] = case["dw"]
        msk[0, 0, case["ho"], case["wo"]] = case["mask"]
        y = o.forward(x, off, msk, np.ones((1, 1, 1, 1)), None, library=lib)
        if abs(y[0, 0, case["ho"], case["wo"]] - case["expected"]) > 1e-12:
            failed.append("P6")
            break
    # P1 (strided, dilated, grouped)
    p = P1_SWEEP[1]
    c = make_case(rng, N=1, Cin=8, Cout=8, H=9, W=11, kh=3, kw=3, stride=p["stride"], padding=p["padding"],
                  dilation=p["dilation"], group=p["group"], dg=p["dg"])
    c["offset"][:] = 0.0
    c["mask"][:] = 1.0
    if not np.allclose(fwd(c), conv_ref(c["x"], c["weight"], c["bias"], p["stride"], p["padding"],
                                        p["dilation"], p["group"]), rtol=0, atol=1e-12):
        failed.append("P1")
    # P2 (a != b)
    c = make_case(rng, N=1, Cin=6, Cout=4, H=8, W=7, stride=(2, 1), padding=(1, 2), dilation=(1, 2), group=2, dg=3)
    c["offset"][:, 0::2] = 2
    c["offset"][:, 1::2] = -1
    c["mask"][:] = 1.0
    if not np.allclose(fwd(c), shifted_conv(c["x"], c["weight"], c["bias"], (2, 1), (1, 2), (1, 2), 2, 2, -1),
                       rtol=0, atol=1e-12):
        failed.append("P2")
    # P4 (contiguous blocks) and P3 (mask block)
    c = make_case(rng, N=1, Cin=8, Cout=3, dg=2, bias=False)
    K, Cd, gd = 9, 4, 1
    off2 = c["offset"].copy()
    off2[:, gd * 2 * K:] += 1.3
    diff = fwd(c, offset=off2) - fwd(c)
    xb = np.zeros_like(c["x"])
    xb[:, gd * Cd:] = c["x"][:, gd * Cd:]
    a1 = dict(c["attrs"], deformable_group=1)
    mb = c["mask"][:, gd * K:]
    d1 = fwd(c, x=xb, offset=off2[:, gd * 2 * K:], mask=mb, attrs=a1) - fwd(c, x=xb, offset=c["offset"][:, gd * 2 * K:],
                                                                            mask=mb, attrs=a1)
    if not np.allclose(diff, d1, rtol=0, atol=1e-12):
        failed.append("P4")
    # P5 on border-heavy offsets
    c = make_case(rng, **P5_SWEEP[1])
    a = c["attrs"]
    if not np.allclose(fwd(c), zero_extended_restatement(c["x"], c["offset"], c["mask"], c["weight"], c["bias"],
                                                         a["stride"], a["padding"], a["dilation"], a["group"],
                                                         a["deformable_group"]), rtol=1e-12, atol=1e-12):
        failed.append("P5")
    return failed


def test_unmodified_oracle_passes_compact_pins(oracle_mod):
    assert all_pins(oracle_mod, None) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_slip_is_caught(oracle_mod, name, tmp_path):
    src = open(os.path.join(os.path.dirname(HERE), "oracle", "mdcn_oracle.c")).read()
    for old, new in MUTATIONS[name]:
        assert old in src, (name, old)
        src = src.replace(old, new)
    cpath = tmp_path / "mutant.c"
    cpath.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so),
                    str(cpath), "-lm"], check=True)
    lib = oracle_mod.load_library(str(so))
    assert all_pins(oracle_mod, lib), f"planted slip {name} passed every pin"


# ---------------------------------------------------------------- the pack front end
# (offset and mask from an ordinary convolution of x; the final sigmoid on the
# mask channels). Pinned against torch's float64 conv2d and sigmoid, and a
# closed form.

def _pack_case(seed=7, N=2, Cin=4, H=7, W=6, Cout=5, k=(3, 3), stride=(1, 1), padding=(1, 1), dilation=(1, 1),
               dg=2, group=1):
    g = torch.Generator().manual_seed(seed)
    kh, kw = k
    K = kh * kw
    x = torch.randn(N, Cin, H, W, generator=g, dtype=torch.float64)
    w_om = 0.3 * torch.randn(3 * dg * K, Cin, kh, kw, generator=g, dtype=torch.float64)
    b_om = 0.2 * torch.randn(3 * dg * K, generator=g, dtype=torch.float64)
    w = torch.randn(Cout, Cin // group, kh, kw, generator=g, dtype=torch.float64)
    b = torch.randn(Cout, generator=g, dtype=torch.float64)
    return x, w_om, b_om, w, b, dict(stride=stride, padding=padding, dilation=dilation, group=group,
                                     deformable_group=dg)


@pytest.mark.parametrize("geom", [dict(), dict(stride=(2, 1), padding=(2, 0), dilation=(1, 2)),
                                  dict(k=(1, 3), dg=1, padding=(0, 1))])
def test_pack_front_end_is_conv2d_then_sigmoid(oracle_mod, geom):
    x, w_om, b_om, w, b, a = _pack_case(**geom)
    off, msk = oracle_mod.offset_mask_front_end(x.numpy(), w_om.numpy(), b_om.numpy(), a["stride"], a["padding"],
                                                a["dilation"], a["deformable_group"])
    om = torch.nn.functional.conv2d(x, w_om, b_om, a["stride"], a["padding"], a["dilation"])
    c = off.shape[1]
    assert c == 2 * a["deformable_group"] * w_om.shape[2] * w_om.shape[3]
    np.testing.assert_allclose(off, om[:, :c].numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(msk, torch.sigmoid(om[:, c:]).numpy(), rtol=0, atol=1e-12)


def test_pack_zero_front_end_is_half_conv(oracle_mod):
    """weight_om = 0, bias_om = 0: offset 0 and mask 1/2 everywhere, so the
    output is half an ordinary convolution plus the bias."""
    x, w_om, b_om, w, b, a = _pack_case(seed=8)
    out, off, msk = oracle_mod.forward_pack(x.numpy(), np.zeros_like(w_om.numpy()), np.zeros_like(b_om.numpy()),
                                            w.numpy(), b.numpy(), **a)
    assert np.all(off == 0) and np.all(msk == 0.5)
    ref = 0.5 * torch.nn.functional.conv2d(x, w, None, a["stride"], a["padding"], a["dilation"], a["group"]) \
        + b[None, :, None, None]
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)


def test_pack_mask_channels_follow_the_offset_channels(oracle_mod):
    """Only the mask channel of tap k of deformable group 0 is switched on
    (bias +40, every other mask channel -40, zero offset weights): the output
    is the convolution restricted to that tap on group 0's input channels."""
    x, w_om, b_om, w, b, a = _pack_case(seed=9, dg=2)
    K = 9
    w_om0 = np.zeros_like(w_om.numpy())
    b_om0 = np.full(b_om.shape, -40.0)
    b_om0[: 2 * 2 * K] = 0.0                   # offsets 0
    k = 4
    b_om0[2 * 2 * K + k] = 40.0                # mask of (group 0, tap k) ~ 1
    out, off, msk = oracle_mod.forward_pack(x.numpy(), w_om0, b_om0, w.numpy(), None, **a)
    wk = torch.zeros_like(w)
    wk[:, : w.shape[1] // 2, k // 3, k % 3] = w[:, : w.shape[1] // 2, k // 3, k % 3]
    ref = torch.nn.functional.conv2d(x, wk, None, a["stride"], a["padding"], a["dilation"], a["group"])
    np.testing.assert_allclose(out, ref.numpy(), rtol=0, atol=1e-12)
