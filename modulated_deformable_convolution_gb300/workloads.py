"""Seeded synthetic workloads for the DCNv2 forward.

This module only draws random inputs; it holds none of the operator's
arithmetic, so both the CUDA path's tests and the CPU oracle can take their
inputs from it. Inputs are drawn in fp32 on the CPU with one
``torch.Generator`` per case, in the order x, offset, mask (logits or
uniform), weight, bias, and then rounded to the case's storage dtype.

The named configurations are detection-neck shapes of the kind OCDNet uses
(the network that "TensorRT plugin walkthrough: modulatedDeformConvPlugin",
sections 1 and 7, names as the operator's consumer); no dataset or trained
weights are involved.
"""
from __future__ import annotations

import dataclasses
import math

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Case:
    name: str
    dtype: str  # "f32" | "f16" | "bf16"
    N: int
    Cin: int
    Cout: int
    H: int
    W: int
    kh: int = 3
    kw: int = 3
    stride: tuple = (1, 1)
    padding: tuple = (1, 1)
    dilation: tuple = (1, 1)
    group: int = 1
    deformable_group: int = 1
    bias: bool = False
    seed: int = 0
    # value distributions: ("normal", std) or ("uniform", lo, hi)
    offset_dist: tuple = ("normal", 1.0)
    mask_dist: str = "sigmoid"  # "sigmoid" of N(0,1) logits, or "uniform" U(0,1)
    weight_std: float | None = None  # default 1/sqrt(Cin*kh*kw)
    bias_std: float = 0.1
    Ho: int | None = None  # default: the convolution formula
    Wo: int | None = None

    @property
    def out_hw(self):
        Ho = self.Ho if self.Ho is not None else conv_out(self.H, self.kh, self.stride[0], self.padding[0], self.dilation[0])
        Wo = self.Wo if self.Wo is not None else conv_out(self.W, self.kw, self.stride[1], self.padding[1], self.dilation[1])
        return Ho, Wo

    @property
    def flops(self) -> int:
        """Contraction flops 2*N*Cout*Ho*Wo*(Cin/group)*kh*kw."""
        Ho, Wo = self.out_hw
        return 2 * self.N * self.Cout * Ho * Wo * (self.Cin // self.group) * self.kh * self.kw

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def io_bytes(self) -> int:
        """x + offset + mask + weight + bias + out, each once (algorithmic bytes)."""
        Ho, Wo = self.out_hw
        K = self.kh * self.kw
        n = (self.N * self.Cin * self.H * self.W
             + self.N * 3 * self.deformable_group * K * Ho * Wo
             + self.Cout * (self.Cin // self.group) * K
             + (self.Cout if self.bias else 0)
             + self.N * self.Cout * Ho * Wo)
        return n * self.elem_bytes

    def attrs(self) -> dict:
        return dict(stride=tuple(self.stride), padding=tuple(self.padding), dilation=tuple(self.dilation),
                    group=self.group, deformable_group=self.deformable_group)


def conv_out(size: int, k: int, s: int, p: int, d: int) -> int:
    return (size + 2 * p - d * (k - 1) - 1) // s + 1


# The five named workloads (tiny, OCDNet-like neck, multi-deformable-group,
# grouped/strided/dilated with border-heavy offsets, large-channel).
CONFIGS = {
    "tiny_f32": Case("tiny_f32", "f32", N=1, Cin=8, Cout=8, H=16, W=16, bias=True, seed=0,
                     offset_dist=("uniform", -2.0, 2.0)),
    "neck_f16": Case("neck_f16", "f16", N=4, Cin=128, Cout=128, H=80, W=80, bias=False, seed=1,
                     offset_dist=("normal", 1.5)),
    "multidg_bf16": Case("multidg_bf16", "bf16", N=8, Cin=256, Cout=256, H=40, W=40,
                         deformable_group=4, bias=True, seed=2, offset_dist=("normal", 2.0)),
    "grouped_f32": Case("grouped_f32", "f32", N=2, Cin=256, Cout=256, H=100, W=100,
                        stride=(2, 2), padding=(2, 2), dilation=(2, 2), group=4, deformable_group=2,
                        bias=True, seed=3, offset_dist=("uniform", -8.0, 8.0), mask_dist="uniform",
                        weight_std=1.0 / math.sqrt(64 * 9)),
    "largec_f16": Case("largec_f16", "f16", N=16, Cin=512, Cout=512, H=32, W=32,
                       deformable_group=8, bias=False, seed=4, offset_dist=("normal", 1.0)),
}
CONFIG_ORDER = ["tiny_f32", "neck_f16", "multidg_bf16", "grouped_f32", "largec_f16"]

# Context beside the named workloads: the neck shape as a depthwise layer (one
# group per channel, one deformable group), the case for the direct kernel.
CONFIGS["depthwise_f16"] = Case("depthwise_f16", "f16", N=4, Cin=128, Cout=128, H=80, W=80, group=128, bias=False,
                                seed=5, offset_dist=("normal", 1.5))
EXTRA_ORDER = ["depthwise_f16"]


def make_inputs(case: Case, device="cpu"):
    """Draw the case's inputs. Returns a dict of tensors in the case's dtype:
    x, offset, mask, weight, bias (None when the case has no bias)."""
    g = torch.Generator().manual_seed(int(case.seed))
    Ho, Wo = case.out_hw
    K = case.kh * case.kw
    dg = case.deformable_group
    x = torch.randn(case.N, case.Cin, case.H, case.W, generator=g)
    od = case.offset_dist
    if od[0] == "normal":
        offset = torch.randn(case.N, 2 * dg * K, Ho, Wo, generator=g) * float(od[1])
    elif od[0] == "uniform":
        offset = torch.rand(case.N, 2 * dg * K, Ho, Wo, generator=g) * (od[2] - od[1]) + od[1]
    else:
        raise ValueError(od)
    if case.mask_dist == "sigmoid":
        mask = torch.sigmoid(torch.randn(case.N, dg * K, Ho, Wo, generator=g))
    elif case.mask_dist == "uniform":
        mask = torch.rand(case.N, dg * K, Ho, Wo, generator=g)
    else:
        raise ValueError(case.mask_dist)
    wstd = case.weight_std if case.weight_std is not None else 1.0 / math.sqrt(case.Cin * K)
    weight = torch.randn(case.Cout, case.Cin // case.group, case.kh, case.kw, generator=g) * wstd
    bias = torch.randn(case.Cout, generator=g) * case.bias_std if case.bias else None
    dt = DTYPES[case.dtype]
    out = dict(x=x, offset=offset, mask=mask, weight=weight, bias=bias)
    return {k: (None if v is None else v.to(dt).contiguous().to(device)) for k, v in out.items()}


def make_grad_out(case: Case, device="cpu"):
    """The output gradient of the case for the backward pass: N(0, 1) of the
    output's shape in the case's dtype, from its own seeded stream (seed + 1000)."""
    g = torch.Generator().manual_seed(int(case.seed) + 1000)
    Ho, Wo = case.out_hw
    go = torch.randn(case.N, case.Cout, Ho, Wo, generator=g)
    return go.to(DTYPES[case.dtype]).contiguous().to(device)
