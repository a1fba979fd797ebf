"""Double-precision CPU oracle for the modulated deformable convolution forward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the product path never
does. It shares no code with the CUDA library and never imports it.

The arithmetic lives in ``mdcn_oracle.c`` (plain C, fp64), which follows
"TensorRT plugin walkthrough: modulatedDeformConvPlugin" (trdm.cn), section 5
steps 1-3, with the layouts of section 2 and the attributes of section 3. This
module compiles it with gcc, checks arguments the way the page's plugin does
(section 2 shape rule, section 3 attribute ranges, section 4 dimension
bindings) and marshals numpy float64 arrays.

``backward`` gives the gradients of the same definition (the pages have no
backward; the reading is stated in the C source), pinned in
``tests/test_oracle_backward.py`` by finite differences of the forward,
adjoint identities, the ordinary-convolution special case and hand-worked
slopes.

Parity status: every part of the definition is pinned by tests in
``tests/test_oracle.py`` (ordinary and shifted convolution, hand-computed
bilinear values, mask and deformable-group invariants, a zero-extended
restatement, linearity, group decomposition). Unpinned: nothing of the
definition; the GPU's low-precision rounding pattern is bounded only by the
tolerance.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mdcn_oracle.c")
_LIB = os.path.join(_HERE, "libmdcn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``mdcn_oracle.c`` into ``libmdcn_oracle.so`` next to it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str):
    """Load a compiled oracle library and declare its entry points."""
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.mdcn_oracle_forward_f64.argtypes = [p, p, p, p, p, p] + [i64] * 19 + [ctypes.c_int]
    lib.mdcn_oracle_forward_f64.restype = ctypes.c_int
    lib.mdcn_oracle_backward_f64.argtypes = [p] * 10 + [i64] * 17 + [ctypes.c_int, ctypes.c_int]
    lib.mdcn_oracle_backward_f64.restype = ctypes.c_int
    lib.mdcn_oracle_num_threads.argtypes = []
    lib.mdcn_oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = load_library(_LIB)
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle runs on by default."""
    return int(_load().mdcn_oracle_num_threads())


def _pair(v, name):
    if isinstance(v, (int, np.integer)):
        return (int(v), int(v))
    v = tuple(int(t) for t in v)
    if len(v) != 2:
        raise ValueError(f"{name} must have two components")
    return v


def check_attrs(stride, padding, dilation, group, deformable_group):
    """Attribute ranges of section 3: stride, dilation > 0; padding >= 0; group, dg > 0."""
    stride, padding, dilation = _pair(stride, "stride"), _pair(padding, "padding"), _pair(dilation, "dilation")
    if min(stride) < 1 or min(dilation) < 1:
        raise ValueError("stride and dilation components must be >= 1")
    if min(padding) < 0:
        raise ValueError("padding components must be >= 0")
    if int(group) < 1 or int(deformable_group) < 1:
        raise ValueError("group and deformable_group must be >= 1")
    return stride, padding, dilation, int(group), int(deformable_group)


def output_shape(x_shape, offset_shape, mask_shape, weight_shape, bias_shape=None,
                 deformable_group=1, group=1):
    """Output dims per section 2 (getOutputShapes): N from x, Cout from weight,
    Ho and Wo from offset. Also checks the section-4 dimension bindings
    (offset/mask batch = x batch, mask spatial = offset spatial, bias length =
    Cout) and the channel counts that the layouts imply."""
    N, Cin, H, W = (int(t) for t in x_shape)
    Cout, Cg, kh, kw = (int(t) for t in weight_shape)
    No, Co, Ho, Wo = (int(t) for t in offset_shape)
    Nm, Cm, Hm, Wm = (int(t) for t in mask_shape)
    K = kh * kw
    if min(N, Cin, H, W, Cout, Cg, kh, kw, Ho, Wo) < 1:
        raise ValueError("every dimension must be >= 1")
    if No != N or Nm != N:
        raise ValueError("offset and mask batch must equal x batch")
    if (Hm, Wm) != (Ho, Wo):
        raise ValueError("mask spatial dims must equal offset spatial dims")
    if Co != 2 * deformable_group * K:
        raise ValueError("offset channels must be 2*deformable_group*kh*kw")
    if Cm != deformable_group * K:
        raise ValueError("mask channels must be deformable_group*kh*kw")
    if Cin % group or Cout % group or Cg != Cin // group:
        raise ValueError("weight must be [Cout, Cin/group, kh, kw] with group | Cin, Cout")
    if Cin % deformable_group:
        raise ValueError("deformable_group must divide Cin")
    if bias_shape is not None and tuple(int(t) for t in bias_shape) != (Cout,):
        raise ValueError("bias must be [Cout]")
    return (N, Cout, Ho, Wo)


def forward(x, offset, mask, weight, bias=None, stride=1, padding=0, dilation=1, group=1,
            deformable_group=1, ho_range=None, nthreads: int = 0, library=None):
    """Oracle forward. Array arguments are converted to contiguous float64.

    ``ho_range=(a, b)`` computes only output rows a..b-1 (the rest of the
    returned array is zero); used to time a bounded slice of a workload.
    ``library`` runs another build of the C source (the tests use it to
    check that deliberately broken copies fail the pins).
    """
    stride, padding, dilation, group, deformable_group = check_attrs(
        stride, padding, dilation, group, deformable_group)
    x = np.ascontiguousarray(x, dtype=np.float64)
    offset = np.ascontiguousarray(offset, dtype=np.float64)
    mask = np.ascontiguousarray(mask, dtype=np.float64)
    weight = np.ascontiguousarray(weight, dtype=np.float64)
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float64)
    shape = output_shape(x.shape, offset.shape, mask.shape, weight.shape,
                         None if bias is None else bias.shape, deformable_group, group)
    N, Cin, H, W = x.shape
    Cout, _, kh, kw = weight.shape
    Ho, Wo = shape[2], shape[3]
    a, b = (0, Ho) if ho_range is None else (int(ho_range[0]), int(ho_range[1]))
    out = np.zeros(shape, dtype=np.float64)
    lib = library if library is not None else _load()
    ptr = lambda arr: None if arr is None else arr.ctypes.data_as(ctypes.c_void_p)
    rc = lib.mdcn_oracle_forward_f64(
        ptr(x), ptr(offset), ptr(mask), ptr(weight), ptr(bias), ptr(out),
        N, Cin, H, W, Cout, kh, kw, Ho, Wo,
        stride[0], stride[1], padding[0], padding[1], dilation[0], dilation[1],
        group, deformable_group, a, b, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return out


def conv_output_hw(H, W, kh, kw, stride, padding, dilation):
    """Spatial size of an ordinary convolution: floor((H + 2p - d(k-1) - 1)/s) + 1."""
    stride, padding, dilation = _pair(stride, "stride"), _pair(padding, "padding"), _pair(dilation, "dilation")
    Ho = (H + 2 * padding[0] - dilation[0] * (kh - 1) - 1) // stride[0] + 1
    Wo = (W + 2 * padding[1] - dilation[1] * (kw - 1) - 1) // stride[1] + 1
    return Ho, Wo


def offset_mask_front_end(x, weight_om, bias_om, stride=1, padding=0, dilation=1, deformable_group=1,
                          kernel_size=None, nthreads: int = 0):
    """The offset/mask front end of the "pack" form of the modulated
    deformable convolution (mmcv ModulatedDeformConv2dPack semantics, which
    the pages name but do not spell out; reading in the design notes): an
    ordinary convolution of x with weight_om [3*dg*kh*kw, Cin, kh, kw] and
    bias_om [3*dg*kh*kw] (group 1, the layer's stride, padding and dilation),
    whose first 2*dg*kh*kw output channels are the offset and whose last
    dg*kh*kw channels, through the logistic sigmoid, are the mask.

    The convolution is this oracle's own forward with zero offsets and a unit
    mask, which the P1 pins prove equal to an ordinary convolution. Returns
    (offset, mask) as float64 arrays."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    weight_om = np.ascontiguousarray(weight_om, dtype=np.float64)
    bias_om = np.ascontiguousarray(bias_om, dtype=np.float64)
    N, Cin, H, W = x.shape
    Com, Cin_w, kh, kw = weight_om.shape
    K = kh * kw
    if Cin_w != Cin:
        raise ValueError("weight_om must be [3*dg*kh*kw, Cin, kh, kw]")
    if Com != 3 * deformable_group * K:
        raise ValueError("weight_om must have 3*deformable_group*kh*kw output channels")
    if bias_om.shape != (Com,):
        raise ValueError("bias_om must be [3*dg*kh*kw]")
    Ho, Wo = conv_output_hw(H, W, kh, kw, stride, padding, dilation)
    if Ho < 1 or Wo < 1:
        raise ValueError("the convolution has an empty output")
    zero_off = np.zeros((N, 2 * K, Ho, Wo))
    unit_mask = np.ones((N, K, Ho, Wo))
    om = forward(x, zero_off, unit_mask, weight_om, bias_om, stride, padding, dilation, 1, 1, nthreads=nthreads)
    c = 2 * deformable_group * K
    offset = np.ascontiguousarray(om[:, :c])
    mask = 1.0 / (1.0 + np.exp(-om[:, c:]))
    return offset, np.ascontiguousarray(mask)


def forward_pack(x, weight_om, bias_om, weight, bias=None, stride=1, padding=0, dilation=1, group=1,
                 deformable_group=1, nthreads: int = 0):
    """The pack form end to end: offset and mask from the front end above,
    then this oracle's forward. Returns (out, offset, mask)."""
    offset, mask = offset_mask_front_end(x, weight_om, bias_om, stride, padding, dilation, deformable_group,
                                         nthreads=nthreads)
    out = forward(x, offset, mask, weight, bias, stride, padding, dilation, group, deformable_group,
                  nthreads=nthreads)
    return out, offset, mask


def backward(x, offset, mask, weight, grad_out, stride=1, padding=0, dilation=1, group=1, deformable_group=1,
             with_bias=True, positions: str = "f64", nthreads: int = 0, library=None):
    """Oracle backward: the gradients of sum(grad_out * forward(...)) with
    respect to x, offset, mask, weight and (if ``with_bias``) the bias.

    The pages describe the forward only; this is the gradient of that
    definition (the one-sided derivative on cell edges, 0 outside the
    sampling range; the reading is spelled out in ``mdcn_oracle.c``).
    Returns a dict of float64 arrays with the shapes of the inputs; the bias
    gradient is None when ``with_bias`` is false.

    ``positions``: "f64" forms each sampling position exactly (the gradient of
    the forward); "f32" rounds anchor + offset to fp32 first, as the kernels
    do, so that the cell (a floor, across which the slope jumps) is decided
    in the kernels' precision. Only positions within half an fp32 ulp of a
    cell edge differ."""
    if positions not in ("f64", "f32"):
        raise ValueError("positions must be 'f64' or 'f32'")
    stride, padding, dilation, group, deformable_group = check_attrs(
        stride, padding, dilation, group, deformable_group)
    x = np.ascontiguousarray(x, dtype=np.float64)
    offset = np.ascontiguousarray(offset, dtype=np.float64)
    mask = np.ascontiguousarray(mask, dtype=np.float64)
    weight = np.ascontiguousarray(weight, dtype=np.float64)
    grad_out = np.ascontiguousarray(grad_out, dtype=np.float64)
    shape = output_shape(x.shape, offset.shape, mask.shape, weight.shape, None, deformable_group, group)
    if tuple(grad_out.shape) != tuple(shape):
        raise ValueError(f"grad_out must have the output's shape {shape}")
    N, Cin, H, W = x.shape
    Cout, _, kh, kw = weight.shape
    Ho, Wo = shape[2], shape[3]
    g = {"x": np.zeros_like(x), "offset": np.zeros_like(offset), "mask": np.zeros_like(mask),
         "weight": np.zeros_like(weight), "bias": np.zeros(Cout) if with_bias else None}
    lib = library if library is not None else _load()
    ptr = lambda arr: None if arr is None else arr.ctypes.data_as(ctypes.c_void_p)
    rc = lib.mdcn_oracle_backward_f64(
        ptr(x), ptr(offset), ptr(mask), ptr(weight), ptr(grad_out),
        ptr(g["x"]), ptr(g["offset"]), ptr(g["mask"]), ptr(g["weight"]), ptr(g["bias"]),
        N, Cin, H, W, Cout, kh, kw, Ho, Wo,
        stride[0], stride[1], padding[0], padding[1], dilation[0], dilation[1],
        group, deformable_group, int(positions == "f32"), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle backward failed with code {rc}")
    return g
