"""GPU parity of the backward (mdcn_backward through the C ABI) against the
fp64 CPU oracle's backward on the same seeded inputs.

The oracle's backward is pinned in tests/test_oracle_backward.py (finite
differences of the forward, adjoint identities, conv2d autograd, hand-worked
slopes). Gate per gradient tensor: max |gpu - ref| <= tol * max |ref|, tol =
1e-4 for float32 I/O and 2e-2 for float16 / bfloat16 I/O (fp32 arithmetic
inside, as for the forward). The oracle consumes the inputs and grad_out
already rounded to the I/O dtype, widened exactly to float64.
"""
import numpy as np
import pytest
import torch

import modulated_deformable_convolution_gb300 as mdcn
from modulated_deformable_convolution_gb300.workloads import (CONFIG_ORDER, CONFIGS, Case, make_grad_out,
                                                             make_inputs)

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "f16": 2e-2, "bf16": 2e-2}
NAMES = ("x", "offset", "mask", "weight", "bias")


def np64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def gpu_backward(case, inp, go, poison=True):
    dev = torch.device("cuda", 0)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    god = go.to(dev)
    h = mdcn.Handle(**case.attrs())
    gb = torch.full((case.Cout,), float("nan"), dtype=d["x"].dtype, device=dev) if case.bias else None
    need = mdcn.mdcn_backward_workspace_size(h, d["x"], d["offset"], d["mask"], d["weight"], gb)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=dev)  # garbage workspace: nothing may rely on zeros
    fill = float("nan") if poison else 0.0
    g = {k: torch.full_like(d[k], fill) for k in ("x", "offset", "mask", "weight")}
    mdcn.mdcn_backward(h, d["x"], d["offset"], d["mask"], d["weight"], god, g["x"], g["offset"], g["mask"],
                       g["weight"], gb, ws)
    torch.cuda.synchronize()
    s, bits = mdcn.mdcn_query_status(ws)  # no bounded wait of the tensor-core GEMMs gave up
    assert s == mdcn.MDCN_OK, f"device status {bits:#x}"
    g["bias"] = gb
    return {k: np64(v) for k, v in g.items()}


def oracle_backward(oracle_mod, case, inp, go):
    # The slope of the bilinear sample jumps across a cell edge, and the cell
    # is a floor of the position: the oracle takes that decision in the
    # kernels' precision (anchor + offset rounded to fp32). Exactly formed
    # positions differ at points within half an fp32 ulp of an edge, e.g. a
    # bf16 offset of -1.4e-6 from anchor 38 (multi-deformable-group workload).
    return oracle_mod.backward(np64(inp["x"]), np64(inp["offset"]), np64(inp["mask"]), np64(inp["weight"]),
                               np64(go), with_bias=case.bias, positions="f32", **case.attrs())


def compare_all(gpu, ref, dtype, label):
    for k in NAMES:
        if ref[k] is None:
            assert gpu[k] is None
            continue
        g = gpu[k]
        assert np.isfinite(g).all(), f"{label} grad_{k}: non-finite (unwritten) elements"
        err = np.abs(g - ref[k]).max()
        scale = np.abs(ref[k]).max()
        ratio = err / max(scale, 1e-30)
        print(f"[{label}] grad_{k}: max|err|/max|ref| = {ratio:.3e} (tol {TOL[dtype]:.0e})")
        assert ratio <= TOL[dtype], f"{label} grad_{k}: {ratio:.3e} > {TOL[dtype]}"


SWEEP = [
    Case("b_f32_small", "f32", N=2, Cin=8, Cout=8, H=9, W=11, bias=True, seed=60, offset_dist=("normal", 1.5)),
    Case("b_f16_ragged", "f16", N=3, Cin=64, Cout=48, H=13, W=13, bias=True, seed=61, offset_dist=("normal", 1.5)),
    Case("b_bf16_g2_dg4_s2", "bf16", N=2, Cin=128, Cout=96, H=11, W=17, stride=(2, 2), group=2, deformable_group=4,
         bias=True, seed=62, offset_dist=("normal", 2.0)),
    Case("b_f32_k5x3_dg2", "f32", N=1, Cin=32, Cout=40, H=15, W=15, kh=5, kw=3, padding=(2, 1), deformable_group=2,
         bias=False, seed=63, offset_dist=("uniform", -2.0, 2.0)),
    Case("b_f16_depthwise", "f16", N=2, Cin=16, Cout=16, H=9, W=9, group=16, deformable_group=16, bias=True,
         seed=64),
    Case("b_f32_1x1_dg3_far", "f32", N=2, Cin=24, Cout=20, H=7, W=9, kh=1, kw=1, padding=(0, 0), deformable_group=3,
         bias=True, seed=65, offset_dist=("uniform", -8.0, 8.0), mask_dist="uniform"),
    Case("b_f16_s2p2d2_g4_dg2", "f16", N=1, Cin=64, Cout=64, H=21, W=21, stride=(2, 2), padding=(2, 2),
         dilation=(2, 2), group=4, deformable_group=2, bias=True, seed=66, offset_dist=("normal", 3.0)),
    Case("b_bf16_1x5_free_hw", "bf16", N=3, Cin=48, Cout=32, H=6, W=31, kh=1, kw=5, padding=(0, 2), bias=True,
         seed=67, Ho=4, Wo=29),
    Case("b_f32_cin3", "f32", N=2, Cin=3, Cout=5, H=8, W=8, bias=True, seed=68, offset_dist=("normal", 1.0)),
    Case("b_f16_cd6_g3", "f16", N=2, Cin=18, Cout=9, H=10, W=7, group=3, deformable_group=3, bias=False, seed=69,
         offset_dist=("normal", 1.0)),
    # the tensor-core GEMMs (P and K*Cg multiples of 8): pixels not a multiple of 128, K*Cg = 4.5 tiles,
    # Og < 64 (one zero-padded contraction chunk)
    Case("b_f16_tc_ragged", "f16", N=3, Cin=64, Cout=48, H=12, W=10, deformable_group=2, bias=True, seed=71,
         offset_dist=("normal", 1.5)),
    # groups with several deformable groups each
    Case("b_bf16_tc_g2_dg4", "bf16", N=2, Cin=128, Cout=96, H=20, W=20, group=2, deformable_group=4, bias=True,
         seed=72, offset_dist=("normal", 2.0)),
    # Cd = 16, strided 5x3 taps
    Case("b_f16_tc_cd16_s2_k5x3", "f16", N=2, Cin=64, Cout=40, H=16, W=16, kh=5, kw=3, stride=(2, 2),
         padding=(2, 1), deformable_group=4, bias=False, seed=77, offset_dist=("normal", 1.5)),
    # Cd = 8 (lanes of 2 per sampling point)
    Case("b_f16_tc_cd8_s2_k5x3", "f16", N=2, Cin=32, Cout=40, H=16, W=16, kh=5, kw=3, stride=(2, 2),
         padding=(2, 1), deformable_group=4, bias=False, seed=73, offset_dist=("normal", 1.5)),
    # Og = 256 (four 64-wide contraction chunks), Cd = 128, dilated, border-heavy offsets
    Case("b_f16_tc_og256_dil2", "f16", N=1, Cin=128, Cout=256, H=24, W=24, padding=(2, 2), dilation=(2, 2),
         bias=False, seed=74, offset_dist=("uniform", -4.0, 4.0), mask_dist="uniform"),
    # Cd = 4: one lane per sampling point
    Case("b_bf16_tc_cd4", "bf16", N=2, Cin=8, Cout=8, H=8, W=8, deformable_group=2, bias=True, seed=75,
         offset_dist=("normal", 1.0)),
    # a deformable group of 32 channels over two groups of 16
    Case("b_f16_tc_g4_dg2", "f16", N=2, Cin=64, Cout=64, H=16, W=16, group=4, deformable_group=2,
         bias=True, seed=76, offset_dist=("normal", 1.5)),
]

# Two image chunks (about 140 MB of per-chunk buffers per image: one image per chunk).
CHUNKED = Case("b_f16_tc_chunks", "f16", N=2, Cin=16, Cout=16, H=384, W=384, bias=False, seed=70,
               offset_dist=("normal", 1.5))


@pytest.mark.parametrize("case", SWEEP, ids=[c.name for c in SWEEP])
def test_backward_sweep(oracle_mod, case):
    inp = make_inputs(case)
    go = make_grad_out(case)
    compare_all(gpu_backward(case, inp, go), oracle_backward(oracle_mod, case, inp, go), case.dtype, case.name)


def test_backward_two_chunks(oracle_mod):
    """Images in two chunks (each chunk's channels-last x, columns and grad_x
    buffers reused), every element of every gradient."""
    case = CHUNKED
    inp = make_inputs(case)
    h = mdcn.Handle(**case.attrs())
    dev = torch.device("cuda", 0)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    launches = mdcn.mdcn_backward_launches(h, d["x"], d["offset"], d["mask"], d["weight"], None)
    # weight re-layout; per chunk: transpose (clearing grad_x), column-gradient GEMM, sampling,
    # weight-gradient GEMM and its split sum, transpose; the weight gradient's layout
    assert launches == 1 + 2 * 6 + 1
    go = make_grad_out(case)
    compare_all(gpu_backward(case, inp, go), oracle_backward(oracle_mod, case, inp, go), case.dtype, case.name)


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_backward_named_workloads(oracle_mod, name):
    """The five named workloads at full size, every element of every
    gradient; large-channel runs in two image chunks."""
    case = CONFIGS[name]
    inp = make_inputs(case)
    go = make_grad_out(case)
    compare_all(gpu_backward(case, inp, go), oracle_backward(oracle_mod, case, inp, go), case.dtype, name)


def test_backward_zero_grad_out_gives_zero():
    case = SWEEP[1]
    inp = make_inputs(case)
    go = torch.zeros_like(make_grad_out(case))
    g = gpu_backward(case, inp, go)
    for k in NAMES:
        assert not np.any(g[k]), k


def test_backward_repeatable_except_grad_x():
    """Two calls agree bit for bit on every gradient but grad_x (whose fp32
    atomic sums may round differently), and closely on grad_x."""
    case = SWEEP[2]
    inp = make_inputs(case)
    go = make_grad_out(case)
    a, b = gpu_backward(case, inp, go), gpu_backward(case, inp, go)
    for k in ("offset", "mask", "weight", "bias"):
        assert np.array_equal(a[k], b[k]), k
    assert np.abs(a["x"] - b["x"]).max() <= 1e-2 * np.abs(a["x"]).max()


def test_backward_rejects_before_launch():
    case = SWEEP[0]
    dev = torch.device("cuda", 0)
    inp = {k: v.to(dev) for k, v in make_inputs(case).items()}
    go = make_grad_out(case).to(dev)
    h = mdcn.Handle(**case.attrs())
    need = mdcn.mdcn_backward_workspace_size(h, inp["x"], inp["offset"], inp["mask"], inp["weight"], inp["bias"])
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    g = {k: torch.full_like(inp[k], 7.0) for k in ("x", "offset", "mask", "weight", "bias")}
    with pytest.raises(mdcn.MdcnError) as e:  # workspace one byte short
        mdcn.mdcn_backward(h, inp["x"], inp["offset"], inp["mask"], inp["weight"], go, g["x"], g["offset"], g["mask"],
                           g["weight"], g["bias"], ws[: need - 1])
    assert e.value.status == mdcn.MDCN_ERR_WORKSPACE
    with pytest.raises(mdcn.MdcnError) as e:  # grad_out of the wrong dims is caught by the Python shape check of dims
        mdcn.mdcn_backward(h, inp["x"], inp["offset"], inp["mask"], inp["weight"][:, :4].contiguous(), go, g["x"], g["offset"],
                           g["mask"], g["weight"], g["bias"], ws)
    assert e.value.status == mdcn.MDCN_ERR_SHAPE
    torch.cuda.synchronize()
    for k in g:
        assert torch.all(g[k] == 7.0), k
