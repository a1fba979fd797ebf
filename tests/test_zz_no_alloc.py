"""The allocation-free forward, mdcn_forward_noalloc, against mdcn_forward.

mdcn_forward_noalloc exists for callers that cannot allocate device memory on
their execution path (for example a serving loop that reserves all memory at
start-up, or a runtime whose execute step must not call cudaMalloc). Its
scratch is a fixed 64 MiB array inside the library, shared by every call on a
device. These checks call it twice in a row through the C ABI and compare each
result with the ordinary forward (which gets a caller-allocated workspace):
both run the same plan and kernels on the same inputs, so the outputs must be
bitwise equal. They also read the array's status word through
mdcn_noalloc_query_status after the calls, and check that a workload needing
more scratch is refused before anything runs.

This file is collected last on purpose, and it does its own set-up, so it runs
the same alone in a fresh process or after every other test.
"""
import ctypes
import dataclasses

import pytest
import torch

from modulated_deformable_convolution_gb300 import _abi, build
from modulated_deformable_convolution_gb300.workloads import CONFIGS, make_inputs

import modulated_deformable_convolution_gb300 as mdcn

pytestmark = pytest.mark.gpu

def _lib():
    build.build()
    return _abi.load()


def _noalloc_fn():
    f = _lib().mdcn_forward_noalloc
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(_abi.mdcn_dims), ctypes.c_int, vp]
    f.restype = ctypes.c_int
    return f


def _noalloc_status():
    """Reads and clears the fixed array's status word on the current device."""
    f = _lib().mdcn_noalloc_query_status
    f.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    f.restype = ctypes.c_int
    bits = ctypes.c_uint32(0xFFFFFFFF)
    s = f(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), ctypes.byref(bits))
    return s, bits.value


def _inputs(name, **replace):
    case = dataclasses.replace(CONFIGS[name], **replace) if replace else CONFIGS[name]
    dev = torch.device("cuda", 0)
    d = {k: (None if v is None else v.to(dev)) for k, v in make_inputs(case).items()}
    return case, d


def _call_noalloc(f, h, d, out):
    dims = mdcn.make_dims(d["x"].shape, d["offset"].shape, d["mask"].shape, d["weight"].shape,
                          0 if d["bias"] is None else d["bias"].shape[0])
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    dt = {torch.float32: _abi.MDCN_F32, torch.float16: _abi.MDCN_F16, torch.bfloat16: _abi.MDCN_BF16}[d["x"].dtype]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return f(h.value, ptr(d["x"]), ptr(d["offset"]), ptr(d["mask"]), ptr(d["weight"]), ptr(d["bias"]), ptr(out),
             ctypes.byref(dims), dt, stream)


@pytest.mark.parametrize("name", ["neck_f16", "tiny_f32", "multidg_bf16", "largec_f16", "depthwise_f16"])
def test_noalloc_matches_forward_on_two_calls(name):
    f = _noalloc_fn()
    case, d = _inputs(name)
    h = mdcn.Handle(**case.attrs())
    ref = mdcn.forward(d["x"], d["offset"], d["mask"], d["weight"], d["bias"], handle=h)
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _call_noalloc(f, h, d, out) == mdcn.MDCN_OK
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all(), f"call {call}: unwritten output"
        # same plan, same kernels, same inputs: the outputs are identical
        assert torch.equal(out, ref), f"call {call}: max diff {(out.float() - ref.float()).abs().max().item()}"
        s, bits = _noalloc_status()
        assert s == mdcn.MDCN_OK and bits == 0, f"call {call}: status {s}, bits {bits:#x}"


def test_noalloc_refuses_workloads_beyond_its_scratch():
    f = _noalloc_fn()
    case, d = _inputs("largec_f16", N=64)  # its channels-last x alone is 67 MB
    h = mdcn.Handle(**case.attrs())
    out = torch.zeros(mdcn.mdcn_output_dims(h, d["x"], d["offset"], d["mask"], d["weight"], d["bias"]),
                      dtype=d["x"].dtype, device=d["x"].device)
    assert _call_noalloc(f, h, d, out) == mdcn.MDCN_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0  # nothing was launched
