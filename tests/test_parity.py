"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle
on the same seeded inputs.

Gate (per case): max |gpu - ref| <= tol * max |ref|, tol = 1e-4 for float32
I/O and 2e-2 for float16 / bfloat16 I/O with fp32 accumulation. The oracle
consumes the inputs already rounded to the I/O dtype, widened exactly to
float64. Informational columns (printed): the per-element relative error
|gpu - ref| / max(|ref|, 1e-6) (max, mean, share above 1e-5).
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import modulated_deformable_convolution_gb300 as mdcn
from modulated_deformable_convolution_gb300.workloads import CONFIG_ORDER, CONFIGS, Case, make_inputs

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "f16": 2e-2, "bf16": 2e-2}


def np64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


_REF_CACHE = {}


def oracle_out(oracle_mod, case, inp, ho_range=None):
    """The oracle's output for a case. Full outputs of the named workloads
    (inputs untouched) are computed once per session."""
    key = (case.name, case.seed) if ho_range is None and case.name in CONFIGS and case == CONFIGS[case.name] else None
    if key is not None and key in _REF_CACHE:
        return _REF_CACHE[key]
    ref = oracle_mod.forward(np64(inp["x"]), np64(inp["offset"]), np64(inp["mask"]), np64(inp["weight"]),
                              np64(inp["bias"]), ho_range=ho_range, **case.attrs())
    if key is not None:
        _REF_CACHE[key] = ref
    return ref


def gpu_out(case, inp, algo="fused", check_status=True, tuning=None):
    dev = torch.device("cuda", 0)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    h = mdcn.Handle(**case.attrs(), tuning=tuning)
    if algo == "fused":
        need = mdcn.mdcn_workspace_size(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"])
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
    else:
        need = mdcn.mdcn_im2col_gemm_workspace_size(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"])
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
    shape = mdcn.mdcn_output_dims(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"])
    out = torch.full(shape, float("nan"), dtype=d["x"].dtype, device=dev)  # poison: every element must be written
    if algo == "fused":
        mdcn.mdcn_forward(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"], out, ws)
        if check_status:
            s, bits = mdcn.mdcn_query_status(ws)
            assert s == mdcn.MDCN_OK, f"device status {bits:#x}"
    else:
        mdcn.mdcn_forward_im2col_gemm(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"], out, ws)
    torch.cuda.synchronize()
    return out


def compare(gpu, ref, dtype, label):
    g = gpu.astype(np.float64)
    assert np.isfinite(g).all(), f"{label}: non-finite output"
    err = np.abs(g - ref)
    scale = np.abs(ref).max()
    ratio = err.max() / max(scale, 1e-30)
    rel = err / np.maximum(np.abs(ref), 1e-6)
    print(f"[{label}] max|err|/max|ref| = {ratio:.3e} (tol {TOL[dtype]:.0e}); rel: max {rel.max():.2e} "
          f"mean {rel.mean():.2e} >1e-5 {np.mean(rel > 1e-5) * 100:.1f}%")
    assert ratio <= TOL[dtype], f"{label}: {ratio:.3e} > {TOL[dtype]}"


@pytest.mark.parametrize("name", CONFIG_ORDER)
def test_named_workloads(oracle_mod, name):
    """The five named workloads at full size, in the launch configuration the
    benchmark times: every element of the output against the oracle."""
    case = CONFIGS[name]
    inp = make_inputs(case)
    gpu = np64(gpu_out(case, inp))
    ref = oracle_out(oracle_mod, case, inp)
    compare(gpu, ref, case.dtype, name)


SWEEP = [
    Case("f16_ragged", "f16", N=3, Cin=64, Cout=48, H=13, W=13, bias=True, seed=10, offset_dist=("normal", 1.5)),
    Case("bf16_g2_dg4_s2", "bf16", N=2, Cin=128, Cout=96, H=11, W=17, stride=(2, 2), group=2, deformable_group=4,
         bias=True, seed=11, offset_dist=("normal", 2.0)),
    Case("f32_k5x3_dg2", "f32", N=1, Cin=32, Cout=40, H=15, W=15, kh=5, kw=3, padding=(2, 1), deformable_group=2,
         bias=True, seed=12, offset_dist=("uniform", -2.0, 2.0)),
    Case("f16_depthwise", "f16", N=2, Cin=16, Cout=16, H=9, W=9, group=16, deformable_group=16, bias=True, seed=13),
    Case("f16_cout320", "f16", N=1, Cin=64, Cout=320, H=12, W=12, bias=False, seed=14),
    Case("bf16_cout544", "bf16", N=1, Cin=32, Cout=544, H=10, W=10, bias=True, seed=15),
    Case("f32_1x1_dg3_far", "f32", N=2, Cin=24, Cout=20, H=7, W=9, kh=1, kw=1, padding=(0, 0), deformable_group=3,
         bias=False, seed=16, offset_dist=("uniform", -8.0, 8.0), mask_dist="uniform"),
    Case("f16_s2p2d2_g4_dg2", "f16", N=1, Cin=64, Cout=64, H=21, W=21, stride=(2, 2), padding=(2, 2),
         dilation=(2, 2), group=4, deformable_group=2, bias=True, seed=17, offset_dist=("normal", 3.0)),
    Case("bf16_1x5_free_hw", "bf16", N=3, Cin=48, Cout=32, H=6, W=31, kh=1, kw=5, padding=(0, 2), bias=True,
         seed=18, Ho=4, Wo=29),
    Case("f32_tiny_cin3", "f32", N=2, Cin=3, Cout=5, H=8, W=8, bias=True, seed=19, offset_dist=("normal", 1.0)),
    Case("f16_k7_dil3", "f16", N=1, Cin=16, Cout=16, H=20, W=20, kh=7, kw=7, padding=(9, 9), dilation=(3, 3),
         bias=False, seed=20, offset_dist=("normal", 2.0)),
]


@pytest.mark.parametrize("case", SWEEP, ids=[c.name for c in SWEEP])
def test_sweep_full_compare(oracle_mod, case):
    inp = make_inputs(case)
    gpu = np64(gpu_out(case, inp))
    ref = oracle_out(oracle_mod, case, inp)
    compare(gpu, ref, case.dtype, case.name)


TUNED = [
    # 2-D tiles with ragged right edge, TMA-store epilogue (Wo*2 bytes % 16 == 0, Og % 16 == 0)
    (Case("f16_2d_ragged_tma", "f16", N=2, Cin=64, Cout=32, H=40, W=40, bias=True, seed=40,
          offset_dist=("normal", 2.0)), dict(tile_mode=1, stages=4)),
    # grouped, 2-D tiles, TMA-store epilogue with a group channel offset, bf16
    (Case("bf16_2d_g2_tma", "bf16", N=1, Cin=64, Cout=96, H=24, W=32, group=2, deformable_group=2, bias=True,
          seed=41), dict(tile_mode=1, stages=2)),
    # ragged bottom edge (Ho = 20 not a multiple of 8), fp32, 2-D tiles, TMA-store epilogue
    (Case("f32_2d_bottom_tma", "f32", N=1, Cin=32, Cout=16, H=20, W=16, bias=False, seed=42), dict(tile_mode=1)),
    # 2-D tiles without the TMA epilogue (Og = 40 not a multiple of 16)
    (Case("f16_2d_scalar_epi", "f16", N=1, Cin=32, Cout=40, H=16, W=32, bias=True, seed=43), dict(tile_mode=1)),
    # linear tiles forced on a shape the planner would tile in 2-D, several CTAs per SM count capped
    (Case("f16_linear_forced", "f16", N=2, Cin=64, Cout=64, H=16, W=16, bias=False, seed=44),
     dict(tile_mode=0, stages=6, max_ctas=3)),
    # Cout = 512 in one tile (two MMAs, one TMEM accumulator), 2-D tiles
    (Case("f16_cout512_2d", "f16", N=1, Cin=64, Cout=512, H=16, W=16, deformable_group=2, bias=False, seed=45),
     dict(tile_mode=1)),
    # one k-tile at a time across all 8 gather warps; two tap blocks (K = 15) of two channel chunks
    (Case("bf16_k5x3_kg1", "bf16", N=2, Cin=128, Cout=64, H=12, W=12, kh=5, kw=3, padding=(2, 1), bias=True,
          seed=46, offset_dist=("normal", 2.0)), dict(kgroups=1, stages=2)),
    # four k-tiles at once; 1x1 kernel with 3 deformable groups: groups of one k-tile, most warps skip most groups
    (Case("f16_1x1_dg3_kg4", "f16", N=2, Cin=96, Cout=32, H=9, W=11, kh=1, kw=1, padding=(0, 0),
          deformable_group=3, bias=True, seed=47, offset_dist=("uniform", -3.0, 3.0)), dict(kgroups=4, stages=4)),
    # fp32, 10 tiles of 9 k-tiles over 4 CTAs: 23 k-tiles each, tiles split at three points
    (Case("f32_split4", "f32", N=1, Cin=64, Cout=48, H=24, W=24, group=2, deformable_group=2, bias=True, seed=48,
          offset_dist=("normal", 2.0)), dict(max_ctas=4)),
    # A stages in tensor memory: bf16, 2 groups x 2 deformable groups, 8 stages, tiles split over 5 CTAs
    (Case("bf16_tmemA_g2_split", "bf16", N=2, Cin=64, Cout=96, H=20, W=24, group=2, deformable_group=2, bias=True,
          seed=49, offset_dist=("normal", 2.0)), dict(a_operand=2, stages=8, max_ctas=5)),
    # A stages in tensor memory with one accumulator (Cout = 256 leaves no room for two), linear tiles, f16
    (Case("f16_tmemA_cout256", "f16", N=1, Cin=128, Cout=256, H=13, W=27, bias=True, seed=50), dict(a_operand=2)),
    # the same shape with A in shared memory
    (Case("f16_smemA_cout256", "f16", N=1, Cin=128, Cout=256, H=13, W=27, bias=True, seed=50), dict(a_operand=1)),
]


@pytest.mark.parametrize("case,tuning", TUNED, ids=[c.name for c, _ in TUNED])
def test_tuned_plans(oracle_mod, case, tuning):
    inp = make_inputs(case)
    gpu = np64(gpu_out(case, inp, tuning=tuning))
    ref = oracle_out(oracle_mod, case, inp)
    compare(gpu, ref, case.dtype, case.name)


def test_tunings_agree_bitwise():
    """With the A stages in one place (shared or tensor memory), the stage count
    and the number of k-tiles produced at once do not change which sums are
    formed nor their order: outputs are bitwise equal."""
    case = CONFIGS["neck_f16"]
    inp = make_inputs(case)
    smem = gpu_out(case, inp, tuning=dict(a_operand=1))
    for tuning in (dict(a_operand=1, stages=2), dict(stages=4, kgroups=4), dict(stages=4, kgroups=1),
                   dict(stages=2, kgroups=1)):
        assert torch.equal(gpu_out(case, inp, tuning=tuning), smem), tuning
    tmem = gpu_out(case, inp)
    for tuning in (dict(stages=2), dict(a_operand=2, stages=8), dict(stages=6)):
        assert torch.equal(gpu_out(case, inp, tuning=tuning), tmem), tuning


@pytest.mark.parametrize("name", ["neck_f16", "multidg_bf16"])
def test_a_operand_places_agree(oracle_mod, name):
    """A in tensor memory (one accumulator where two do not fit beside the
    stages, as on multi-dg) and in shared memory: both within the tolerance of
    the oracle on every element, and within one rounding of each other."""
    case = CONFIGS[name]
    inp = make_inputs(case)
    ref = oracle_out(oracle_mod, case, inp)
    outs = [np64(gpu_out(case, inp, tuning=dict(a_operand=a))) for a in (1, 2)]
    for a, g in zip((1, 2), outs):
        compare(g, ref, case.dtype, f"{name} a_operand={a}")
    # the two differ only in fp32 rounding inside the accumulation, which can
    # move an output by at most one unit in the last place of its 16-bit type
    ulp = {"f16": 2.0 ** -10, "bf16": 2.0 ** -7}[case.dtype]
    assert np.abs(outs[0] - outs[1]).max() <= ulp * np.abs(outs[0]).max()


@pytest.mark.parametrize("tuning", [dict(max_ctas=40), dict(max_ctas=7), dict(max_ctas=151), dict(tile_mode=0)],
                         ids=["ctas40_whole_tiles", "ctas7", "ctas151", "linear_tiles"])
def test_split_points_move(oracle_mod, tuning):
    """Other CTA counts and tile shapes split other tiles between CTAs (and
    max_ctas=40 splits none on this shape): every element stays within the
    tolerance."""
    case = CONFIGS["neck_f16"]
    inp = make_inputs(case)
    gpu = np64(gpu_out(case, inp, tuning=tuning))
    ref = oracle_out(oracle_mod, case, inp)
    compare(gpu, ref, case.dtype, f"neck {tuning}")


@pytest.mark.parametrize("case", [SWEEP[0], SWEEP[1], SWEEP[2], SWEEP[3]], ids=lambda c: c.name)
def test_im2col_gemm_ablation(oracle_mod, case):
    inp = make_inputs(case)
    gpu = np64(gpu_out(case, inp, algo="im2col_gemm"))
    ref = oracle_out(oracle_mod, case, inp)
    compare(gpu, ref, case.dtype, "im2col_" + case.name)


def test_im2col_gemm_neck_f16(oracle_mod):
    case = CONFIGS["neck_f16"]
    inp = make_inputs(case)
    gpu = np64(gpu_out(case, inp, algo="im2col_gemm"))
    ref = oracle_out(oracle_mod, case, inp)
    compare(gpu, ref, case.dtype, "im2col neck")


def test_query_plan_split_choice():
    """The planner splits tiles between CTAs where that evens out the work
    (neck: 200 tiles over one CTA per SM) and keeps whole tiles where the
    split would not pay (largec: 2 tiles of 72 k-tiles per CTA)."""
    dev = torch.device("cuda", 0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    for name, split, a_operand in (("neck_f16", 1, 2), ("largec_f16", 0, 1), ("multidg_bf16", 1, 2)):
        case = CONFIGS[name]
        d = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(case).items()}
        h = mdcn.Handle(**case.attrs())
        plan = mdcn.mdcn_query_plan(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"])
        assert plan["split"] == split, (name, plan)
        assert plan["a_operand"] == a_operand, (name, plan)
        assert plan["launches"] == 2  # one prep launch (transpose + pack), the fused kernel
        assert plan["ctas"] <= sms and plan["ctas"] * plan["ktiles_per_cta"] >= plan["tiles"] * plan["ktiles_per_tile"]
        if not split:
            assert plan["ktiles_per_cta"] % plan["ktiles_per_tile"] == 0


def test_zero_mask_gives_bias():
    case = dataclasses.replace(SWEEP[2], name="f32_mask0", seed=30)
    inp = make_inputs(case)
    inp["mask"] = torch.zeros_like(inp["mask"])
    gpu = gpu_out(case, inp).cpu()
    expect = inp["bias"][None, :, None, None].expand_as(gpu)
    assert torch.equal(gpu, expect)


def test_huge_offsets_read_nothing():
    """Offsets far outside the image (and NaN-free huge values) give bias only."""
    case = dataclasses.replace(SWEEP[0], name="f16_far", seed=31)
    inp = make_inputs(case)
    inp["offset"] = torch.full_like(inp["offset"], 3.0e4)
    gpu = gpu_out(case, inp).cpu()
    expect = inp["bias"][None, :, None, None].expand_as(gpu)
    assert torch.equal(gpu, expect)


def test_deterministic_bitwise():
    case = CONFIGS["multidg_bf16"]
    inp = make_inputs(case)
    a = gpu_out(case, inp)
    b = gpu_out(case, inp)
    assert torch.equal(a, b)


def test_wait_timeout_selftest_then_gpu_still_works():
    """The bounded wait gives up on a barrier nothing signals, reports a
    timeout, and the context stays usable."""
    buf = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert mdcn.mdcn_selftest_wait_timeout(buf, 2000) == mdcn.MDCN_ERR_TIMEOUT
    bits = int(buf[0].item())
    assert bits & 1 and bits & (1 << 14) and not bits & (1 << 31)
    case = SWEEP[9]
    inp = make_inputs(case)
    out = gpu_out(case, inp)
    assert torch.isfinite(out).all()


def test_rejected_calls_leave_out_untouched():
    """Calls that fail validation on real device buffers (workspace too small,
    a misaligned pointer, dims that break a binding) return their error and
    launch nothing: the canary in out survives."""
    case = CONFIGS["neck_f16"]
    dev = torch.device("cuda", 0)
    d = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(case).items()}
    h = mdcn.Handle(**case.attrs())
    x, off, m, w = d["x"], d["offset"], d["mask"], d["weight"]
    dims = mdcn.make_dims(x.shape, off.shape, m.shape, w.shape, 0)
    nbytes = mdcn.mdcn_workspace_size(h, x, off, m, w, None)
    ws = torch.zeros(nbytes + 64, dtype=torch.uint8, device=dev)
    out = torch.full(mdcn.mdcn_output_dims(h, x, off, m, w, None), 7.0, dtype=x.dtype, device=dev)
    lib = mdcn._lib()
    vp = lambda t, add=0: ctypes.c_void_p(t.data_ptr() + add)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def fwd(out_add=0, ws_bytes=nbytes, dd=dims):
        return lib.mdcn_forward(h.value, vp(x), vp(off), vp(m), vp(w), None, vp(out, out_add), vp(ws), ws_bytes,
                                ctypes.byref(dd), mdcn._abi.MDCN_F16, st)

    assert fwd(ws_bytes=nbytes - 256) == mdcn.MDCN_ERR_WORKSPACE
    assert fwd(out_add=2) == mdcn._abi.MDCN_ERR_ALIGN
    bad = mdcn.make_dims(x.shape, off.shape, m.shape, w.shape, 0)
    bad.mask[1] = 4
    assert fwd(dd=bad) == mdcn._abi.MDCN_ERR_SHAPE
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    assert fwd() == mdcn.MDCN_OK  # and the same buffers work
    torch.cuda.synchronize()
    assert not torch.all(out == 7.0)


# Shapes with little contraction per output, for the direct CUDA-core kernel:
# depthwise with a channel multiplier, small groups, the largest direct group
# (32 outputs), strides, dilations, 5x3 taps, far offsets. Each runs on both
# paths (tuning path=2 and path=1).
DIRECT = [
    Case("f16_dw_mult2_dg8", "f16", N=2, Cin=32, Cout=64, H=23, W=19, group=32, deformable_group=8, bias=True,
         seed=70, offset_dist=("normal", 2.0)),
    Case("bf16_g8_s2d2", "bf16", N=2, Cin=64, Cout=64, H=30, W=30, stride=(2, 2), padding=(2, 2), dilation=(2, 2),
         group=8, deformable_group=4, bias=True, seed=71, offset_dist=("uniform", -4.0, 4.0)),
    Case("f32_g4_k5x3_far", "f32", N=1, Cin=16, Cout=16, H=17, W=21, kh=5, kw=3, padding=(2, 1), group=4,
         deformable_group=2, bias=False, seed=72, offset_dist=("uniform", -6.0, 6.0), mask_dist="uniform"),
    Case("f16_og32_cg2", "f16", N=1, Cin=4, Cout=64, H=12, W=12, group=2, deformable_group=2, bias=True, seed=73),
]


@pytest.mark.parametrize("case", DIRECT, ids=[c.name for c in DIRECT])
def test_direct_path(oracle_mod, case):
    """The direct kernel (one launch) and the fused kernel, each forced on the
    same shape, both meet the tolerance on every element; the automatic plan is
    direct exactly where (Cin/group) * (Cout/group) <= 16."""
    dev = torch.device("cuda", 0)
    inp = make_inputs(case)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    for tuning, path in ((None, 2 if (case.Cin // case.group) * (case.Cout // case.group) <= 16 else 1),
                         (dict(path=2), 2), (dict(path=1), 1)):
        h = mdcn.Handle(**case.attrs(), tuning=tuning)
        plan = mdcn.mdcn_query_plan(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"])
        assert plan["path"] == path and (path == 1 or plan["launches"] == 1), (tuning, plan)
    ref = oracle_out(oracle_mod, case, inp)
    compare(np64(gpu_out(case, inp, tuning=dict(path=2))), ref, case.dtype, case.name + " direct")
    compare(np64(gpu_out(case, inp, tuning=dict(path=1))), ref, case.dtype, case.name + " fused")


@pytest.mark.parametrize("case", SWEEP, ids=[c.name for c in SWEEP])
def test_sweep_fused_forced(oracle_mod, case):
    """Every sweep shape on the fused kernel, whichever path the planner picks
    for it (the small ones plan as direct)."""
    inp = make_inputs(case)
    compare(np64(gpu_out(case, inp, tuning=dict(path=1))), oracle_out(oracle_mod, case, inp), case.dtype,
            case.name + " fused")


# Depthwise layers (one input and one output channel per group) whose
# deformable groups hold whole 4-channel chunks: the automatic plan is the
# direct kernel's channels-last form (a copy of x, then the kernel: two
# launches); forced path=2 keeps the plain direct kernel on x in place.
DIRECT_CL = [
    Case("f16_dw_dg1", "f16", N=2, Cin=64, Cout=64, H=20, W=21, group=64, bias=True, seed=75,
         offset_dist=("normal", 1.5)),
    Case("bf16_dw_dg16_s2", "bf16", N=2, Cin=64, Cout=64, H=19, W=17, stride=(2, 2), group=64,
         deformable_group=16, bias=False, seed=76, offset_dist=("normal", 2.0)),
    Case("f32_dw_k5x3_far", "f32", N=1, Cin=8, Cout=8, H=13, W=15, kh=5, kw=3, padding=(2, 1), group=8,
         deformable_group=2, bias=True, seed=77, offset_dist=("uniform", -6.0, 6.0), mask_dist="uniform"),
    # bfloat16 with one deformable group (the shared-points kernel), 96 channels: lanes 24-31 idle
    Case("bf16_dw_dg1_c96", "bf16", N=2, Cin=96, Cout=96, H=14, W=18, group=96, bias=True, seed=79,
         offset_dist=("normal", 2.0)),
    # 132 channels: a second block of channels with one lane group in it; 63 pixels per image
    Case("f16_dw_c132_dil2", "f16", N=3, Cin=132, Cout=132, H=7, W=9, padding=(2, 2), dilation=(2, 2),
         group=132, deformable_group=33, bias=True, seed=78, Ho=7, Wo=9),
]


@pytest.mark.parametrize("case", DIRECT_CL, ids=[c.name for c in DIRECT_CL])
def test_direct_channels_last(oracle_mod, case):
    """The depthwise channels-last form (automatic plan: two launches, x
    copied channels-last into the workspace after the status header) and the
    plain direct kernel (forced, one launch) both meet the tolerance on every
    element, and give the same bits: the same fp32 sums in the same order."""
    dev = torch.device("cuda", 0)
    inp = make_inputs(case)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    h = mdcn.Handle(**case.attrs())
    plan = mdcn.mdcn_query_plan(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"])
    assert plan["path"] == 2 and plan["launches"] == 2, plan
    es = torch.empty((), dtype=d["x"].dtype).element_size()
    need = mdcn.mdcn_workspace_size(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"])
    assert need >= 1024 + (case.N * case.H * case.W + 1) * case.Cin * es
    hp = mdcn.Handle(**case.attrs(), tuning=dict(path=2))
    assert mdcn.mdcn_query_plan(hp, d["x"], d["offset"], d["mask"], d["weight"], d["bias"])["launches"] == 1
    ref = oracle_out(oracle_mod, case, inp)
    a = gpu_out(case, inp)
    b = gpu_out(case, inp, tuning=dict(path=2))
    compare(np64(a), ref, case.dtype, case.name + " channels-last")
    compare(np64(b), ref, case.dtype, case.name + " direct")
    assert torch.equal(a, b)


def test_direct_neck_depthwise_vs_forced_direct():
    """A neck-sized depthwise layer (128 channels, one deformable group):
    automatic (the channels-last form) and forced-direct plans give the same
    bits; the step-wise calls refuse a direct plan and launch nothing."""
    case = dataclasses.replace(CONFIGS["neck_f16"], name="neck_dw", group=128, seed=74)
    inp = make_inputs(case)
    a = gpu_out(case, inp)
    b = gpu_out(case, inp, tuning=dict(path=2))
    assert torch.equal(a, b)
    dev = torch.device("cuda", 0)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    h = mdcn.Handle(**case.attrs())
    ws = torch.empty(mdcn.mdcn_workspace_size(h, d["x"], d["offset"], d["mask"], d["weight"], None),
                     dtype=torch.uint8, device=dev)
    # the status header, then x channels-last with one zero pixel
    assert ws.numel() == 1024 + (4 * 80 * 80 + 1) * 128 * 2
    hp = mdcn.Handle(**case.attrs(), tuning=dict(path=2))
    assert mdcn.mdcn_workspace_size(hp, d["x"], d["offset"], d["mask"], d["weight"], None) == 1024
    with pytest.raises(mdcn.MdcnError) as e:
        mdcn.mdcn_prepare_input(h, d["x"], d["offset"], d["mask"], d["weight"], None, ws, torch.cuda.current_stream())
    assert e.value.status == mdcn._abi.MDCN_ERR_UNSUPPORTED
