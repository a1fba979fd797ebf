"""mdcn_forward_host (the forward from and to host memory) against
mdcn_forward on device copies of the same inputs: the same kernels run on the
same data, so the outputs must be bitwise equal. Also two streams with two
device buffers, their calls alternating so that the copies of one call overlap
the kernels of the other: every output must still be the one its own inputs
give."""
import dataclasses

import pytest
import torch

from modulated_deformable_convolution_gb300.workloads import CONFIGS, make_inputs

import modulated_deformable_convolution_gb300 as mdcn

pytestmark = pytest.mark.gpu


def _device_reference(case, inp):
    dev = torch.device("cuda", 0)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    h = mdcn.Handle(**case.attrs())
    return mdcn.forward(d["x"], d["offset"], d["mask"], d["weight"], d["bias"], handle=h).cpu()


def _pinned(inp):
    return {k: (None if v is None else v.contiguous().pin_memory()) for k, v in inp.items()}


@pytest.mark.parametrize("name", ["tiny_f32", "neck_f16", "multidg_bf16"])
def test_forward_host_equals_device_forward(name):
    case = CONFIGS[name]
    inp = make_inputs(case)
    ref = _device_reference(case, inp)
    p = _pinned(inp)
    h = mdcn.Handle(**case.attrs())
    out = torch.full(ref.shape, float("nan"), dtype=ref.dtype).pin_memory()
    nbytes = mdcn.mdcn_host_buffer_size(h, p["x"], p["offset"], p["mask"], p["weight"], p["bias"])
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    mdcn.mdcn_forward_host(h, p["x"], p["offset"], p["mask"], p["weight"], p["bias"], out, buf)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_two_streams_pipeline_calls():
    """Calls alternate between two streams and two device buffers (the copies
    of one overlap the kernels of the other); each output matches its inputs."""
    base = CONFIGS["neck_f16"]
    cases = [dataclasses.replace(base, name=f"neck_seed{s}", seed=100 + s) for s in range(4)]
    inps = [make_inputs(c) for c in cases]
    refs = [_device_reference(c, i) for c, i in zip(cases, inps)]
    pins = [_pinned(i) for i in inps]
    h = mdcn.Handle(**base.attrs())
    p0 = pins[0]
    nbytes = mdcn.mdcn_host_buffer_size(h, p0["x"], p0["offset"], p0["mask"], p0["weight"], p0["bias"])
    bufs = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    outs = [torch.full(r.shape, float("nan"), dtype=r.dtype).pin_memory() for r in refs]
    for k, p in enumerate(pins):
        mdcn.mdcn_forward_host(h, p["x"], p["offset"], p["mask"], p["weight"], p["bias"], outs[k], bufs[k % 2],
                               streams[k % 2])
    torch.cuda.synchronize()
    for k in range(len(cases)):
        assert torch.equal(outs[k], refs[k]), f"call {k}"
