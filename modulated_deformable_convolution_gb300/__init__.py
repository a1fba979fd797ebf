"""GB300 (sm_103a) modulated deformable convolution (DCNv2): forward and backward.

Thin Python binding of libmdcn.so (C ABI in include/mdcn.h): the functions
named ``mdcn_*`` here mirror the C entry points one to one and only marshal
arguments (torch tensors -> device pointers, dims, dtype, the current CUDA
stream). Every step of the computation runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback, and a missing library raises.

The operator follows "TensorRT plugin walkthrough: modulatedDeformConvPlugin"
(section 2 inputs/outputs, section 3 attributes, section 5 algorithm).
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import (MDCN_BF16, MDCN_ERR_ALIGN, MDCN_ERR_ARCH, MDCN_ERR_ATTR, MDCN_ERR_CUDA, MDCN_ERR_DTYPE,  # noqa: F401
                   MDCN_ERR_NULL, MDCN_ERR_SHAPE, MDCN_ERR_TIMEOUT, MDCN_ERR_UNSUPPORTED, MDCN_ERR_WORKSPACE,
                   MDCN_F16, MDCN_F32, MDCN_OK)

__all__ = ["Handle", "MdcnError", "forward", "mdcn_create", "mdcn_destroy", "mdcn_output_dims",
           "mdcn_workspace_size", "mdcn_forward", "mdcn_prepare_input", "mdcn_pack_weight",
           "mdcn_forward_prepared", "mdcn_im2col_gemm_workspace_size", "mdcn_forward_im2col_gemm",
           "mdcn_query_plan", "mdcn_query_status", "mdcn_selftest_wait_timeout", "mdcn_status_string",
           "library_path", "backward", "mdcn_backward_workspace_size", "mdcn_backward_launches",
           "mdcn_backward"]

_DTYPES = {torch.float32: MDCN_F32, torch.float16: MDCN_F16, torch.bfloat16: MDCN_BF16}


def library_path() -> str:
    return _abi.LIB_PATH


def _lib():
    return _abi.load()


class MdcnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        msg = _lib().mdcn_status_string(self.status).decode()
        extra = ""
        if self.status == MDCN_ERR_CUDA:
            extra = f" (cudaError {_lib().mdcn_last_cuda_error()})"
        super().__init__(f"{what}: status {self.status}: {msg}{extra}")


def _check(status: int, what: str):
    if status != MDCN_OK:
        raise MdcnError(status, what)


def mdcn_status_string(status: int) -> str:
    return _lib().mdcn_status_string(int(status)).decode()


def _pair(v):
    if isinstance(v, int):
        return (v, v)
    v = tuple(int(t) for t in v)
    assert len(v) == 2
    return v


def mdcn_create(stride=1, padding=0, dilation=1, group=1, deformable_group=1, tuning=None):
    """mdcn_create (or mdcn_create_tuned when ``tuning`` is a dict with keys
    stages, tile_mode, max_ctas, kgroups, a_operand, ntile, path): returns the opaque handle
    (an int) or raises MdcnError."""
    a = _abi.mdcn_attrs()
    a.stride[:] = _pair(stride)
    a.padding[:] = _pair(padding)
    a.dilation[:] = _pair(dilation)
    a.group = int(group)
    a.deformable_group = int(deformable_group)
    h = ctypes.c_void_p()
    if tuning is None:
        _check(_lib().mdcn_create(ctypes.byref(a), ctypes.byref(h)), "mdcn_create")
    else:
        t = _abi.mdcn_tuning(int(tuning.get("stages", 0)), int(tuning.get("tile_mode", -1)),
                             int(tuning.get("max_ctas", 0)), int(tuning.get("kgroups", 0)),
                             int(tuning.get("a_operand", 0)), int(tuning.get("ntile", 0)),
                             int(tuning.get("path", 0)))
        _check(_lib().mdcn_create_tuned(ctypes.byref(a), ctypes.byref(t), ctypes.byref(h)), "mdcn_create_tuned")
    return h.value


def mdcn_destroy(handle) -> None:
    _check(_lib().mdcn_destroy(handle), "mdcn_destroy")


class Handle:
    """Owns one library handle (the five section-3 attributes)."""

    def __init__(self, stride=1, padding=0, dilation=1, group=1, deformable_group=1, tuning=None):
        self.attrs = dict(stride=_pair(stride), padding=_pair(padding), dilation=_pair(dilation), group=int(group),
                          deformable_group=int(deformable_group))
        self.value = mdcn_create(**self.attrs, tuning=tuning)

    def close(self):
        if getattr(self, "value", None):
            mdcn_destroy(self.value)
            self.value = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _hval(handle):
    return handle.value if isinstance(handle, Handle) else handle


def make_dims(x_shape, offset_shape, mask_shape, weight_shape, bias_len: int = 0):
    d = _abi.mdcn_dims()
    d.x[:] = tuple(int(t) for t in x_shape)
    d.offset[:] = tuple(int(t) for t in offset_shape)
    d.mask[:] = tuple(int(t) for t in mask_shape)
    d.weight[:] = tuple(int(t) for t in weight_shape)
    d.bias = int(bias_len)
    return d


def _dims(x, offset, mask, weight, bias):
    for name, t in (("x", x), ("offset", offset), ("mask", mask), ("weight", weight)):
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D")
    if bias is not None and bias.dim() != 1:
        raise ValueError("bias must be 1-D")
    return make_dims(x.shape, offset.shape, mask.shape, weight.shape, 0 if bias is None else bias.shape[0])


def _dtype(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return _DTYPES[t.dtype]


def mdcn_output_dims(handle, x, offset, mask, weight, bias=None):
    out = (ctypes.c_int64 * 4)()
    _check(_lib().mdcn_output_dims(_hval(handle), ctypes.byref(_dims(x, offset, mask, weight, bias)), out),
           "mdcn_output_dims")
    return tuple(int(v) for v in out)


def mdcn_workspace_size(handle, x, offset, mask, weight, bias=None, dtype=None) -> int:
    n = ctypes.c_size_t()
    dt = _dtype(x) if dtype is None else dtype
    _check(_lib().mdcn_workspace_size(_hval(handle), ctypes.byref(_dims(x, offset, mask, weight, bias)), dt,
                                      ctypes.byref(n)), "mdcn_workspace_size")
    return int(n.value)


def mdcn_query_plan(handle, x, offset, mask, weight, bias=None, dtype=None) -> dict:
    """The fused path's execution plan on the current device, as a dict."""
    info = _abi.mdcn_plan_info()
    dt = _dtype(x) if dtype is None else dtype
    with torch.cuda.device(x.device):
        _check(_lib().mdcn_query_plan(_hval(handle), ctypes.byref(_dims(x, offset, mask, weight, bias)), dt,
                                      ctypes.byref(info)), "mdcn_query_plan")
    return {name: int(getattr(info, name)) for name, _ in info._fields_}


def mdcn_im2col_gemm_workspace_size(handle, x, offset, mask, weight, bias=None, dtype=None) -> int:
    n = ctypes.c_size_t()
    dt = _dtype(x) if dtype is None else dtype
    _check(_lib().mdcn_im2col_gemm_workspace_size(_hval(handle), ctypes.byref(_dims(x, offset, mask, weight, bias)),
                                                  dt, ctypes.byref(n)), "mdcn_im2col_gemm_workspace_size")
    return int(n.value)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_tensors(x, offset, mask, weight, bias, out):
    ts = [x, offset, mask, weight, out] + ([bias] if bias is not None else [])
    for t in ts:
        if not t.is_cuda:
            raise ValueError("every tensor must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("every tensor must be contiguous (NCHW)")
        if t.dtype != x.dtype:
            raise TypeError("every tensor must have the dtype of x")


def _stream(dev, stream):
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def mdcn_forward(handle, x, offset, mask, weight, bias, out, workspace, stream=None) -> None:
    """mdcn_forward on torch tensors (device memory) and the current stream."""
    _check_tensors(x, offset, mask, weight, bias, out)
    d = _dims(x, offset, mask, weight, bias)
    with torch.cuda.device(x.device):
        st = _stream(x.device, stream)
        _check(_lib().mdcn_forward(_hval(handle), _ptr(x), _ptr(offset), _ptr(mask), _ptr(weight), _ptr(bias),
                                   _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                   ctypes.byref(d), _dtype(x), st), "mdcn_forward")


def pack_dims(handle, x, weight) -> tuple:
    """Offset and mask shapes of the pack form for x and weight: the
    convolution's spatial size with the handle's attributes."""
    N, Cin, H, W = x.shape
    _, _, kh, kw = weight.shape
    a = handle.attrs
    Ho = (H + 2 * a["padding"][0] - a["dilation"][0] * (kh - 1) - 1) // a["stride"][0] + 1
    Wo = (W + 2 * a["padding"][1] - a["dilation"][1] * (kw - 1) - 1) // a["stride"][1] + 1
    K = kh * kw
    dg = a["deformable_group"]
    return (N, 2 * dg * K, Ho, Wo), (N, dg * K, Ho, Wo)


def mdcn_pack_workspace_size(handle, x, offset, mask, weight, bias=None, dtype=None) -> int:
    n = ctypes.c_size_t()
    dt = _dtype(x) if dtype is None else dtype
    _check(_lib().mdcn_pack_workspace_size(_hval(handle), ctypes.byref(_dims(x, offset, mask, weight, bias)), dt,
                                           ctypes.byref(n)), "mdcn_pack_workspace_size")
    return int(n.value)


def mdcn_forward_pack(handle, x, weight_om, bias_om, weight, bias, offset_out, mask_out, out, workspace,
                      stream=None) -> None:
    """mdcn_forward_pack on torch tensors (device memory): offset_out and
    mask_out receive the front end's offset and mask, out the layer's output."""
    _check_tensors(x, offset_out, mask_out, weight, bias, out)
    for t in (weight_om, bias_om):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != x.dtype:
            raise ValueError("weight_om and bias_om must be contiguous CUDA tensors of x's dtype")
    d = _dims(x, offset_out, mask_out, weight, bias)
    with torch.cuda.device(x.device):
        _check(_lib().mdcn_forward_pack(_hval(handle), _ptr(x), _ptr(weight_om), _ptr(bias_om), _ptr(weight),
                                        _ptr(bias), _ptr(offset_out), _ptr(mask_out), _ptr(out), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), ctypes.byref(d), _dtype(x),
                                        _stream(x.device, stream)), "mdcn_forward_pack")


def mdcn_host_buffer_size(handle, x, offset, mask, weight, bias=None, dtype=None) -> int:
    """Device-buffer bytes of mdcn_forward_host (tensors give only shapes and dtype)."""
    n = ctypes.c_size_t()
    dt = _dtype(x) if dtype is None else dtype
    _check(_lib().mdcn_host_buffer_size(_hval(handle), ctypes.byref(_dims(x, offset, mask, weight, bias)), dt,
                                        ctypes.byref(n)), "mdcn_host_buffer_size")
    return int(n.value)


def mdcn_forward_host(handle, x, offset, mask, weight, bias, out, device_buffer, stream=None) -> None:
    """mdcn_forward_host: x, offset, mask, weight, bias and out are HOST (CPU)
    tensors, page-locked for asynchronous copies; device_buffer is a uint8 CUDA
    tensor of at least mdcn_host_buffer_size bytes. Asynchronous on the stream."""
    for t in [x, offset, mask, weight, out] + ([bias] if bias is not None else []):
        if t.is_cuda:
            raise ValueError("mdcn_forward_host takes host tensors")
        if not t.is_contiguous():
            raise ValueError("every tensor must be contiguous (NCHW)")
        if t.dtype != x.dtype:
            raise TypeError("every tensor must have the dtype of x")
    if not device_buffer.is_cuda:
        raise ValueError("device_buffer must be a CUDA tensor")
    d = _dims(x, offset, mask, weight, bias)
    with torch.cuda.device(device_buffer.device):
        _check(_lib().mdcn_forward_host(_hval(handle), _ptr(x), _ptr(offset), _ptr(mask), _ptr(weight), _ptr(bias),
                                        _ptr(out), _ptr(device_buffer),
                                        device_buffer.numel() * device_buffer.element_size(), ctypes.byref(d),
                                        _dtype(x), _stream(device_buffer.device, stream)), "mdcn_forward_host")


def mdcn_prepare_input(handle, x, offset, mask, weight, bias, workspace, stream=None) -> None:
    """Step 1 of mdcn_forward: x -> channels-last copy in workspace."""
    d = _dims(x, offset, mask, weight, bias)
    with torch.cuda.device(x.device):
        _check(_lib().mdcn_prepare_input(_hval(handle), _ptr(x), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), ctypes.byref(d), _dtype(x),
                                         _stream(x.device, stream)), "mdcn_prepare_input")


def mdcn_pack_weight(handle, x, offset, mask, weight, bias, workspace, stream=None) -> None:
    """Step 2 of mdcn_forward: weight -> packed copy in workspace."""
    d = _dims(x, offset, mask, weight, bias)
    with torch.cuda.device(x.device):
        _check(_lib().mdcn_pack_weight(_hval(handle), _ptr(weight), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), ctypes.byref(d), _dtype(x),
                                       _stream(x.device, stream)), "mdcn_pack_weight")


def mdcn_forward_prepared(handle, x, offset, mask, weight, bias, out, workspace, stream=None) -> None:
    """Step 3 of mdcn_forward: the fused kernel on the prepared workspace,
    sampling from offset and mask (x and weight only supply dims and dtype)."""
    _check_tensors(x, offset, mask, weight, bias, out)
    d = _dims(x, offset, mask, weight, bias)
    with torch.cuda.device(x.device):
        _check(_lib().mdcn_forward_prepared(_hval(handle), _ptr(offset), _ptr(mask), _ptr(bias), _ptr(out),
                                            _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), ctypes.byref(d), _dtype(x),
                                            _stream(x.device, stream)), "mdcn_forward_prepared")


def mdcn_forward_im2col_gemm(handle, x, offset, mask, weight, bias, out, workspace, stream=None) -> None:
    _check_tensors(x, offset, mask, weight, bias, out)
    d = _dims(x, offset, mask, weight, bias)
    with torch.cuda.device(x.device):
        st = _stream(x.device, stream)
        _check(_lib().mdcn_forward_im2col_gemm(_hval(handle), _ptr(x), _ptr(offset), _ptr(mask), _ptr(weight),
                                               _ptr(bias), _ptr(out), _ptr(workspace),
                                               workspace.numel() * workspace.element_size(), ctypes.byref(d),
                                               _dtype(x), st), "mdcn_forward_im2col_gemm")


def mdcn_query_status(workspace, stream=None):
    """Returns (status, raw device bits) and clears the word."""
    bits = ctypes.c_uint32()
    with torch.cuda.device(workspace.device):
        s = _lib().mdcn_query_status(_ptr(workspace), _stream(workspace.device, stream), ctypes.byref(bits))
    return int(s), int(bits.value)


def mdcn_selftest_wait_timeout(status_buf, limit_us: int, stream=None) -> int:
    with torch.cuda.device(status_buf.device):
        return int(_lib().mdcn_selftest_wait_timeout(_ptr(status_buf), int(limit_us),
                                                     _stream(status_buf.device, stream)))


def forward(x, offset, mask, weight, bias=None, stride=1, padding=0, dilation=1, group=1, deformable_group=1,
            algo: str = "fused", out=None, workspace=None, handle=None):
    """DCNv2 forward: allocates the output (and workspace) with torch and
    runs the library on the current stream. ``algo`` = "fused" (default) or
    "im2col_gemm" (the two-stage ablation)."""
    h = handle if handle is not None else Handle(stride, padding, dilation, group, deformable_group)
    dims = mdcn_output_dims(h, x, offset, mask, weight, bias)
    if out is None:
        out = torch.empty(dims, dtype=x.dtype, device=x.device)
    if algo == "fused":
        need = mdcn_workspace_size(h, x, offset, mask, weight, bias)
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
        mdcn_forward(h, x, offset, mask, weight, bias, out, workspace)
    elif algo == "im2col_gemm":
        need = mdcn_im2col_gemm_workspace_size(h, x, offset, mask, weight, bias)
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
        mdcn_forward_im2col_gemm(h, x, offset, mask, weight, bias, out, workspace)
    else:
        raise ValueError(f"unknown algo {algo!r}")
    return out


def mdcn_backward_workspace_size(handle, x, offset, mask, weight, bias=None, dtype=None) -> int:
    n = ctypes.c_size_t()
    dt = _dtype(x) if dtype is None else dtype
    _check(_lib().mdcn_backward_workspace_size(_hval(handle), ctypes.byref(_dims(x, offset, mask, weight, bias)), dt,
                                               ctypes.byref(n)), "mdcn_backward_workspace_size")
    return int(n.value)


def mdcn_backward_launches(handle, x, offset, mask, weight, bias=None, dtype=None) -> int:
    n = ctypes.c_int32()
    dt = _dtype(x) if dtype is None else dtype
    _check(_lib().mdcn_backward_launches(_hval(handle), ctypes.byref(_dims(x, offset, mask, weight, bias)), dt,
                                         ctypes.byref(n)), "mdcn_backward_launches")
    return int(n.value)


def mdcn_backward(handle, x, offset, mask, weight, grad_out, grad_x, grad_offset, grad_mask, grad_weight, grad_bias,
                  workspace, stream=None) -> None:
    """mdcn_backward on torch tensors (device memory) and the current stream.
    grad_bias may be None (no bias gradient)."""
    _check_tensors(x, offset, mask, weight, grad_bias, grad_out)
    for t in (grad_x, grad_offset, grad_mask, grad_weight):
        _check_tensors(x, offset, mask, weight, None, t)
    d = _dims(x, offset, mask, weight, grad_bias)
    with torch.cuda.device(x.device):
        st = _stream(x.device, stream)
        _check(_lib().mdcn_backward(_hval(handle), _ptr(x), _ptr(offset), _ptr(mask), _ptr(weight), _ptr(grad_out),
                                    _ptr(grad_x), _ptr(grad_offset), _ptr(grad_mask), _ptr(grad_weight),
                                    _ptr(grad_bias), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    ctypes.byref(d), _dtype(x), st), "mdcn_backward")


def backward(x, offset, mask, weight, grad_out, with_bias=True, stride=1, padding=0, dilation=1, group=1,
             deformable_group=1, workspace=None, handle=None):
    """Gradients of sum(grad_out * forward(...)): allocates the gradient
    tensors (and workspace) with torch and runs the library on the current
    stream. Returns a dict with x, offset, mask, weight and bias (None when
    ``with_bias`` is false)."""
    h = handle if handle is not None else Handle(stride, padding, dilation, group, deformable_group)
    Cout = weight.shape[0]
    gb = torch.empty(Cout, dtype=x.dtype, device=x.device) if with_bias else None
    need = mdcn_backward_workspace_size(h, x, offset, mask, weight, gb)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    g = {"x": torch.empty_like(x), "offset": torch.empty_like(offset), "mask": torch.empty_like(mask),
         "weight": torch.empty_like(weight), "bias": gb}
    mdcn_backward(h, x, offset, mask, weight, grad_out, g["x"], g["offset"], g["mask"], g["weight"], gb, workspace)
    return g
