"""The pack form (offset and mask from an ordinary convolution of x in front
of the deformable one), with the tolerances of the main parity tests:

- end to end: the GPU's output against the oracle's pack form run on the
  original inputs (its front end in fp64, no rounding of offset or mask), so
  the gate includes the error the front end carries into the deformable
  convolution;
- stage by stage: the GPU's offset and mask against the oracle's front end,
  and the GPU's output against the oracle's forward on the GPU's own offset and
  mask (the rounded tensors the deformable kernel consumed).

Every element of every output is compared."""
import dataclasses

import numpy as np
import pytest
import torch

import modulated_deformable_convolution_gb300 as mdcn

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.float16: 2e-2, torch.bfloat16: 2e-2}


@dataclasses.dataclass
class PackCase:
    name: str
    dtype: torch.dtype
    N: int
    Cin: int
    Cout: int
    H: int
    W: int
    k: tuple = (3, 3)
    stride: tuple = (1, 1)
    padding: tuple = (1, 1)
    dilation: tuple = (1, 1)
    group: int = 1
    dg: int = 1
    bias: bool = True
    seed: int = 0


CASES = [
    PackCase("f16_basic", torch.float16, 2, 64, 64, 24, 24, seed=1),
    PackCase("bf16_dg4", torch.bfloat16, 2, 128, 64, 20, 20, dg=4, seed=2),
    PackCase("f32_s2p2d2_g2_dg2", torch.float32, 1, 32, 48, 17, 17, stride=(2, 2), padding=(2, 2),
             dilation=(2, 2), group=2, dg=2, seed=3),
    PackCase("f16_1x5_odd", torch.float16, 1, 16, 24, 9, 13, k=(1, 5), padding=(0, 2), dg=2, bias=False, seed=4),
    PackCase("f16_neck_shape", torch.float16, 4, 128, 128, 80, 80, seed=5),
    # depthwise deformable convolutions: the direct kernel's channels-last form after the front end
    PackCase("f16_depthwise", torch.float16, 2, 64, 64, 20, 20, group=64, seed=6),
    PackCase("bf16_depthwise_dg16", torch.bfloat16, 1, 64, 64, 15, 17, group=64, dg=16, seed=7),
]


def _inputs(c: PackCase):
    g = torch.Generator().manual_seed(c.seed)
    kh, kw = c.k
    K = kh * kw
    x = torch.randn(c.N, c.Cin, c.H, c.W, generator=g)
    # offsets ~ N(0, 1) and masks spread over (0, 1)
    w_om = torch.randn(3 * c.dg * K, c.Cin, kh, kw, generator=g) / (c.Cin * K) ** 0.5
    b_om = 0.5 * torch.randn(3 * c.dg * K, generator=g)
    w = torch.randn(c.Cout, c.Cin // c.group, kh, kw, generator=g) / (c.Cin // c.group * K) ** 0.5
    b = 0.1 * torch.randn(c.Cout, generator=g) if c.bias else None
    cast = lambda t: None if t is None else t.to(c.dtype)
    return cast(x), cast(w_om), cast(b_om), cast(w), cast(b)


def _f64(t):
    return None if t is None else t.double().cpu().numpy()


@pytest.mark.parametrize("c", CASES, ids=[c.name for c in CASES])
def test_pack_matches_oracle(oracle_mod, c):
    x, w_om, b_om, w, b = _inputs(c)
    dev = torch.device("cuda", 0)
    h = mdcn.Handle(c.stride, c.padding, c.dilation, c.group, c.dg)
    oshape, mshape = mdcn.pack_dims(h, x, w)
    d = {k: (None if v is None else v.to(dev)) for k, v in dict(x=x, w_om=w_om, b_om=b_om, w=w, b=b).items()}
    off = torch.full(oshape, float("nan"), dtype=c.dtype, device=dev)
    msk = torch.full(mshape, float("nan"), dtype=c.dtype, device=dev)
    out = torch.full(mdcn.mdcn_output_dims(h, d["x"], off, msk, d["w"], d["b"]), float("nan"), dtype=c.dtype,
                     device=dev)
    ws = torch.empty(mdcn.mdcn_pack_workspace_size(h, d["x"], off, msk, d["w"], d["b"]), dtype=torch.uint8,
                     device=dev)
    mdcn.mdcn_forward_pack(h, d["x"], d["w_om"], d["b_om"], d["w"], d["b"], off, msk, out, ws)
    torch.cuda.synchronize()
    assert mdcn.mdcn_query_status(ws)[0] == mdcn.MDCN_OK
    # front end
    ref_off, ref_msk = oracle_mod.offset_mask_front_end(_f64(x), _f64(w_om), _f64(b_om), c.stride, c.padding,
                                                        c.dilation, c.dg)
    tol = TOL[c.dtype]
    g_off, g_msk = _f64(off), _f64(msk)
    assert np.isfinite(g_off).all() and np.isfinite(g_msk).all()
    scale = np.abs(ref_off).max()
    assert np.abs(g_off - ref_off).max() <= tol * scale, "offset"
    # the sigmoid is 1/4-Lipschitz: the convolution's error bound, scaled, plus the output rounding
    eps = {torch.float32: 1e-6, torch.float16: 2 ** -10, torch.bfloat16: 2 ** -7}[c.dtype]
    assert np.abs(g_msk - ref_msk).max() <= 0.25 * tol * max(scale, 1.0) + eps, "mask"
    # the deformable convolution on the GPU's own offset and mask
    g_out = _f64(out)
    assert np.isfinite(g_out).all()
    ref = oracle_mod.forward(_f64(x), g_off, g_msk, _f64(w), _f64(b), c.stride, c.padding, c.dilation, c.group,
                             c.dg)
    err = np.abs(g_out - ref).max()
    assert err <= tol * np.abs(ref).max(), f"stage-wise output: {err}"
    # end to end: the oracle's pack form on the original inputs
    ref_e2e, _, _ = oracle_mod.forward_pack(_f64(x), _f64(w_om), _f64(b_om), _f64(w), _f64(b), c.stride, c.padding,
                                            c.dilation, c.group, c.dg)
    err = np.abs(g_out - ref_e2e).max()
    ratio = err / np.abs(ref_e2e).max()
    print(f"[pack {c.name}] end to end max|err|/max|ref| = {ratio:.3e} (tol {tol:.0e})")
    assert ratio <= tol, f"end to end: {ratio:.3e} > {tol}"
