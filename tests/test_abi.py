"""Host-side tests of the C ABI (no GPU needed): the library loads and
exports everything include/mdcn.h declares, attribute validation (section 3),
the output-shape rule and dimension bindings (sections 2 and 4), workspace
sizing, and argument checks that must reject a call before anything is
launched. Fake device pointers are only ever passed to calls that fail
validation first."""
import ctypes

import pytest
import torch

from modulated_deformable_convolution_gb300 import _abi

import modulated_deformable_convolution_gb300 as mdcn


@pytest.fixture(scope="module")
def lib():
    from modulated_deformable_convolution_gb300 import build

    build.build()
    return _abi.load()


def attrs(stride=(1, 1), padding=(1, 1), dilation=(1, 1), group=1, dg=1):
    a = _abi.mdcn_attrs()
    a.stride[:] = stride
    a.padding[:] = padding
    a.dilation[:] = dilation
    a.group = group
    a.deformable_group = dg
    return a


def handle(lib, **kw):
    h = ctypes.c_void_p()
    assert lib.mdcn_create(ctypes.byref(attrs(**kw)), ctypes.byref(h)) == 0
    return h


def dims(N=2, Cin=8, H=10, W=12, Cout=6, kh=3, kw=3, Ho=10, Wo=12, dg=1, group=1, bias=True):
    K = kh * kw
    return mdcn.make_dims((N, Cin, H, W), (N, 2 * dg * K, Ho, Wo), (N, dg * K, Ho, Wo), (Cout, Cin // group, kh, kw),
                          Cout if bias else 0)


def test_every_declared_symbol_is_exported(lib):
    names = _abi.declared_functions()
    assert "mdcn_forward" in names and "mdcn_create" in names
    raw = ctypes.CDLL(_abi.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings(lib):
    for s in range(0, 11):
        assert lib.mdcn_status_string(s)
    assert lib.mdcn_status_string(999) == b"unknown status"


@pytest.mark.parametrize("bad", [
    dict(stride=(0, 1)), dict(stride=(1, -2)), dict(dilation=(0, 1)), dict(padding=(0, -1)), dict(group=0),
    dict(dg=0), dict(dg=-3),
])
def test_create_rejects_out_of_range_attrs(lib, bad):
    h = ctypes.c_void_p(1234)
    assert lib.mdcn_create(ctypes.byref(attrs(**bad)), ctypes.byref(h)) == _abi.MDCN_ERR_ATTR
    assert h.value == 1234  # untouched on error


@pytest.mark.parametrize("tuning,ok", [
    ((0, -1, 0, 0, 0, 0, 0), True), ((4, 1, 8, 4, 1, 256, 1), True), ((2, 0, 0, 1, 0, 16, 2), True),
    ((6, -1, 0, 2, 2, 512, 0), True), ((0, -1, 0, 3, 0, 0, 0), False), ((0, -1, 0, 8, 0, 0, 0), False),
    ((1, -1, 0, 0, 0, 0, 0), False), ((10, -1, 0, 0, 0, 0, 0), False), ((0, 2, 0, 0, 0, 0, 0), False),
    ((0, -1, -1, 0, 0, 0, 0), False), ((0, -1, 0, 0, 3, 0, 0), False), ((0, -1, 0, 0, -1, 0, 0), False),
    ((0, -1, 0, 0, 0, 24, 0), False), ((0, -1, 0, 0, 0, 528, 0), False), ((0, -1, 0, 0, 0, -16, 0), False),
    ((0, -1, 0, 0, 0, 0, 3), False), ((0, -1, 0, 0, 0, 0, -1), False),
])
def test_create_tuned_validates(lib, tuning, ok):
    h = ctypes.c_void_p()
    t = _abi.mdcn_tuning(*tuning)
    s = lib.mdcn_create_tuned(ctypes.byref(attrs()), ctypes.byref(t), ctypes.byref(h))
    assert s == (0 if ok else _abi.MDCN_ERR_ATTR)
    if ok:
        assert lib.mdcn_destroy(h) == 0


def test_create_null(lib):
    h = ctypes.c_void_p()
    assert lib.mdcn_create(None, ctypes.byref(h)) == _abi.MDCN_ERR_NULL
    assert lib.mdcn_create(ctypes.byref(attrs()), None) == _abi.MDCN_ERR_NULL
    assert lib.mdcn_destroy(None) == 0


def out_dims(lib, h, d):
    o = (ctypes.c_int64 * 4)()
    s = lib.mdcn_output_dims(h, ctypes.byref(d), o)
    return s, tuple(o)


def test_output_dims_rule(lib):
    """N from x, Cout from weight, Ho and Wo from offset, even when they do
    not follow the convolution formula."""
    h = handle(lib)
    s, o = out_dims(lib, h, dims(N=3, Cout=5, Ho=4, Wo=17))
    assert s == 0 and o == (3, 5, 4, 17)
    lib.mdcn_destroy(h)


@pytest.mark.parametrize("mut", ["offset_batch", "mask_batch", "mask_spatial", "offset_channels", "mask_channels",
                                 "weight_cg", "bias_len", "group_cout", "dg_cin", "zero_dim"])
def test_output_dims_bindings(lib, mut):
    h = handle(lib, group=2, dg=2)
    d = dims(Cin=8, Cout=6, group=2, dg=2)
    assert out_dims(lib, h, d)[0] == 0
    if mut == "offset_batch":
        d.offset[0] = 3
    elif mut == "mask_batch":
        d.mask[0] = 1
    elif mut == "mask_spatial":
        d.mask[3] = 11
    elif mut == "offset_channels":
        d.offset[1] = 2 * 9
    elif mut == "mask_channels":
        d.mask[1] = 9
    elif mut == "weight_cg":
        d.weight[1] = 8
    elif mut == "bias_len":
        d.bias = 5
    elif mut == "group_cout":
        d.weight[0] = 7
    elif mut == "dg_cin":
        h2 = handle(lib, group=1, dg=3)
        d = dims(Cin=8, Cout=6, dg=3)
        assert out_dims(lib, h2, d)[0] == _abi.MDCN_ERR_SHAPE
        return
    elif mut == "zero_dim":
        d.x[2] = 0
    assert out_dims(lib, h, d)[0] == _abi.MDCN_ERR_SHAPE
    lib.mdcn_destroy(h)


def test_output_dims_too_large(lib):
    h = handle(lib)
    d = dims()
    d.x[2] = 1 << 31
    assert out_dims(lib, h, d)[0] == _abi.MDCN_ERR_UNSUPPORTED


def ws_size(lib, h, d, dt):
    n = ctypes.c_size_t()
    s = lib.mdcn_workspace_size(h, ctypes.byref(d), dt, ctypes.byref(n))
    return s, n.value


def test_workspace_size(lib):
    h = handle(lib)
    d = dims(N=4, Cin=128, H=80, W=80, Cout=128, Ho=80, Wo=80, bias=False)
    s, n = ws_size(lib, h, d, _abi.MDCN_F16)
    # status header + channels-last x + packed weight, each 256-aligned
    assert s == 0 and n >= 1024 + 4 * 80 * 80 * 128 * 2 + 128 * 128 * 9 * 2
    s, n32 = ws_size(lib, h, d, _abi.MDCN_F32)
    assert s == 0 and n32 >= 1024 + 4 * 80 * 80 * 128 * 4 + 2 * 128 * 128 * 9 * 4
    assert ws_size(lib, h, d, 7)[0] == _abi.MDCN_ERR_DTYPE


def fwd(lib, h, ptrs, d, dt=_abi.MDCN_F16, ws_bytes=1 << 30):
    x, off, m, w, b, out, ws = ptrs
    return lib.mdcn_forward(h, x, off, m, w, b, out, ws, ws_bytes, ctypes.byref(d), dt, None)


FAKE = 0x7f0000000000  # never dereferenced: each call below fails validation first


def test_forward_rejects_before_launch(lib):
    h = handle(lib)
    d = dims(bias=True)
    p = [FAKE + 256 * i for i in range(7)]
    # NULL pointers
    for i in (0, 1, 2, 3, 5, 6):
        q = list(p)
        q[i] = None
        assert fwd(lib, h, q, d) == _abi.MDCN_ERR_NULL
    # bias pointer given but dims say no bias, and the reverse
    q = list(p)
    q[4] = None
    assert fwd(lib, h, q, d) == _abi.MDCN_ERR_NULL
    d0 = dims(bias=False)
    assert fwd(lib, h, p, d0) == _abi.MDCN_ERR_SHAPE
    # misaligned pointer
    q = list(p)
    q[1] = FAKE + 8
    assert fwd(lib, h, q, d) == _abi.MDCN_ERR_ALIGN
    # inconsistent dims
    bad = dims(bias=True)
    bad.mask[1] = 3
    assert fwd(lib, h, p, bad) == _abi.MDCN_ERR_SHAPE
    # workspace too small
    assert fwd(lib, h, p, d, ws_bytes=16) == _abi.MDCN_ERR_WORKSPACE
    # dtype
    assert fwd(lib, h, p, d, dt=5) == _abi.MDCN_ERR_DTYPE
    assert lib.mdcn_forward(None, *p, 1 << 30, ctypes.byref(d), 1, None) == _abi.MDCN_ERR_NULL
    lib.mdcn_destroy(h)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_forward_without_device_reports_cuda_error(lib):
    """With valid arguments and no usable GPU the call stops at the device
    check (nothing is dereferenced) and reports a CUDA error."""
    h = handle(lib)
    d = dims(bias=True)
    p = [FAKE + 256 * i for i in range(7)]
    assert fwd(lib, h, p, d) in (_abi.MDCN_ERR_CUDA, _abi.MDCN_ERR_ARCH)
    info = _abi.mdcn_plan_info()
    assert lib.mdcn_query_plan(h, ctypes.byref(d), _abi.MDCN_F16, ctypes.byref(info)) in (
        _abi.MDCN_ERR_CUDA, _abi.MDCN_ERR_ARCH)
    assert lib.mdcn_query_plan(h, ctypes.byref(d), _abi.MDCN_F16, None) == _abi.MDCN_ERR_NULL
    lib.mdcn_destroy(h)


def test_python_binding_rejects_cpu_tensors(lib):
    x = torch.zeros(1, 8, 4, 4)
    off = torch.zeros(1, 18, 4, 4)
    m = torch.zeros(1, 9, 4, 4)
    w = torch.zeros(8, 8, 3, 3)
    h = mdcn.Handle(1, 1, 1, 1, 1)
    assert mdcn.mdcn_output_dims(h, x, off, m, w) == (1, 8, 4, 4)
    with pytest.raises(ValueError):
        mdcn.mdcn_forward(h, x, off, m, w, None, torch.zeros(1, 8, 4, 4), torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(mdcn.MdcnError):
        mdcn.Handle(stride=0)


def test_host_buffer_size_covers_every_part(lib):
    """mdcn_host_buffer_size: the device copies of the five inputs, the output
    and the forward's workspace, each rounded up to 256 bytes."""
    h = handle(lib)
    d = dims(N=4, Cin=128, H=80, W=80, Cout=128, Ho=80, Wo=80, bias=True)
    n = ctypes.c_size_t()
    assert lib.mdcn_host_buffer_size(h, ctypes.byref(d), _abi.MDCN_F16, ctypes.byref(n)) == 0
    s, ws = ws_size(lib, h, d, _abi.MDCN_F16)
    parts = [4 * 128 * 80 * 80, 4 * 18 * 80 * 80, 4 * 9 * 80 * 80, 128 * 128 * 9, 128, 4 * 128 * 80 * 80]
    up = lambda v: (v + 255) // 256 * 256
    assert n.value == sum(up(2 * p) for p in parts) + up(ws)
    assert lib.mdcn_host_buffer_size(h, ctypes.byref(d), 9, ctypes.byref(n)) == _abi.MDCN_ERR_DTYPE
    assert lib.mdcn_host_buffer_size(h, ctypes.byref(d), _abi.MDCN_F16, None) == _abi.MDCN_ERR_NULL
    lib.mdcn_destroy(h)


def test_forward_host_rejects_before_any_copy(lib):
    """Argument checks of mdcn_forward_host come before its first copy: fake
    host and device pointers are never touched."""
    h = handle(lib)
    d = dims(bias=True)
    p = [FAKE + 256 * i for i in range(8)]  # x, offset, mask, weight, bias, out (host), device buffer, spare

    def call(q, dd=d, nbytes=1 << 30, dt=_abi.MDCN_F16):
        return lib.mdcn_forward_host(h, *q[:7], nbytes, ctypes.byref(dd), dt, None)

    for i in (0, 1, 2, 3, 5, 6):
        q = list(p)
        q[i] = None
        assert call(q) == _abi.MDCN_ERR_NULL
    q = list(p)
    q[4] = None
    assert call(q) == _abi.MDCN_ERR_NULL               # dims say bias, none given
    assert call(p, dd=dims(bias=False)) == _abi.MDCN_ERR_SHAPE
    q = list(p)
    q[6] = FAKE + 8
    assert call(q) == _abi.MDCN_ERR_ALIGN              # device buffer misaligned
    q = list(p)
    q[0] = FAKE + 2                                    # host pointers need no alignment
    assert call(q, nbytes=16) == _abi.MDCN_ERR_WORKSPACE
    assert call(p, dt=4) == _abi.MDCN_ERR_DTYPE
    bad = dims(bias=True)
    bad.offset[1] = 5
    assert call(p, dd=bad) == _abi.MDCN_ERR_SHAPE
    lib.mdcn_destroy(h)


def _pack_dims(N=2, Cin=8, H=10, W=12, Cout=6, kh=3, kw=3, stride=1, pad=1, dil=1, dg=1, bias=True):
    Ho = (H + 2 * pad - dil * (kh - 1) - 1) // stride + 1
    Wo = (W + 2 * pad - dil * (kw - 1) - 1) // stride + 1
    return dims(N=N, Cin=Cin, H=H, W=W, Cout=Cout, kh=kh, kw=kw, Ho=Ho, Wo=Wo, dg=dg, bias=bias)


def test_pack_workspace_size_and_shape_rule(lib):
    h = handle(lib, stride=(2, 2), padding=(1, 1), dg=2)
    d = _pack_dims(stride=2, pad=1, dg=2)
    n = ctypes.c_size_t()
    assert lib.mdcn_pack_workspace_size(h, ctypes.byref(d), _abi.MDCN_F16, ctypes.byref(n)) == 0
    s, ws = ws_size(lib, h, d, _abi.MDCN_F16)
    assert s == 0 and n.value >= ws
    bad = _pack_dims(stride=2, pad=1, dg=2)
    bad.offset[2] += 1                               # not the convolution's output height
    bad.mask[2] += 1
    assert lib.mdcn_pack_workspace_size(h, ctypes.byref(bad), _abi.MDCN_F16, ctypes.byref(n)) == _abi.MDCN_ERR_SHAPE
    lib.mdcn_destroy(h)


def test_forward_pack_rejects_before_launch(lib):
    h = handle(lib)
    d = _pack_dims()
    # x, weight_om, bias_om, weight, bias, offset_out, mask_out, out, workspace
    p = [FAKE + 256 * i for i in range(9)]

    def call(q, dd=d, nbytes=1 << 30):
        return lib.mdcn_forward_pack(h, *q, nbytes, ctypes.byref(dd), _abi.MDCN_F16, None)

    for i in (0, 1, 2, 3, 5, 6, 7, 8):
        q = list(p)
        q[i] = None
        assert call(q) == _abi.MDCN_ERR_NULL
    for i in (0, 1, 2, 5, 6):
        q = list(p)
        q[i] = FAKE + 8
        assert call(q) == _abi.MDCN_ERR_ALIGN
    bad = _pack_dims()
    bad.offset[3] = 5
    bad.mask[3] = 5
    assert call(p, dd=bad) == _abi.MDCN_ERR_SHAPE
    assert call(p, nbytes=64) == _abi.MDCN_ERR_WORKSPACE
    lib.mdcn_destroy(h)


def _meta(shape, dtype):
    return torch.empty(shape, dtype=dtype, device="meta")


def _bwd_problem(N, Cin, Cout, H, W, group=1, dg=1, k=3, bias=False, dtype=torch.float16):
    K = k * k
    t = dict(x=_meta((N, Cin, H, W), dtype), offset=_meta((N, 2 * dg * K, H, W), dtype),
             mask=_meta((N, dg * K, H, W), dtype), weight=_meta((Cout, Cin // group, k, k), dtype),
             bias=_meta((Cout,), dtype) if bias else None)
    return t, mdcn.Handle(stride=1, padding=k // 2, dilation=1, group=group, deformable_group=dg)


@pytest.mark.parametrize("N,Cin,Cout,H,group,bias,dtype", [
    (4, 128, 128, 80, 1, False, torch.float16),   # neck: one chunk
    (64, 128, 128, 80, 1, True, torch.float16),   # several chunks
    (2, 256, 256, 100, 4, True, torch.float32),   # grouped: one weight-gradient GEMM per image
    (3, 8, 6, 9, 2, False, torch.bfloat16),       # P = 81: rows break the 16-byte rule, cuBLAS
    (2, 64, 32, 16, 2, True, torch.bfloat16),     # grouped, tensor-core GEMMs
])
def test_backward_chunks_workspace_and_launches(lib, N, Cin, Cout, H, group, bias, dtype):
    """The backward's host plan: images go in chunks of at most 256 MB of
    per-chunk buffers (at least one image); the workspace holds the status
    word, the shared weight buffers, one chunk's buffers and, where the
    contractions run on cuBLAS (float32, or rows that break TMA's 16-byte
    rule), the call's cuBLAS workspace; the launch count follows the chunking
    (tensor-core path: one weight-gradient GEMM per chunk and the in-order sum
    of its split slices; cuBLAS, group 1: a grad_out re-layout and one GEMM per
    chunk; otherwise one GEMM per image; a memset of grad_x where the x
    transpose cannot clear it)."""
    t, h = _bwd_problem(N, Cin, Cout, H, H, group=group, bias=bias, dtype=dtype)
    es = torch.empty((), dtype=dtype).element_size()
    P = H * H
    K = 9
    KCg = K * (Cin // group)
    tc = dtype != torch.float32 and P % 8 == 0 and KCg % 8 == 0
    got = group == 1 and not tc
    cols, pix = P * K * Cin, H * H * Cin
    per_image = cols * (4 + es) + pix * (es + 4) + (Cout * P * es if got else 0)
    nb = max(1, min(N, (256 << 20) // per_image))
    chunks = -(-N // nb)
    ws = mdcn.mdcn_backward_workspace_size(h, t["x"], t["offset"], t["mask"], t["weight"], t["bias"])
    wel = Cout * KCg
    blas = 0 if tc else (32 << 20) + 256  # the call's own cuBLAS workspace (256-byte aligned inside the region)
    # tensor-core weight gradient: one fp32 slice per CTA sharing a 128 x 128 tile's contraction
    Og = Cout // group
    tiles = -(-KCg // 128) * -(-Og // (256 if Og > 128 else 128)) * group
    wsplits = max(1, min(160 // tiles, -(-P // 64) * nb)) if tc else 0
    slices = wsplits * wel * 4
    assert ws >= 256 + wel * es + wel * 4 + nb * per_image + blas + slices
    assert ws <= 256 + wel * es + wel * 4 + nb * per_image + blas + slices + 9 * 256
    launches = mdcn.mdcn_backward_launches(h, t["x"], t["offset"], t["mask"], t["weight"], t["bias"])
    wgrad = 2 * chunks if tc else (2 * chunks if got else N)
    # the x transpose clears grad_x where it takes 16-byte vectors (16-bit I/O, H*W and Cin multiples
    # of 8); else a memset
    memset = 0 if es == 2 and (H * H) % 8 == 0 and Cin % 8 == 0 else 1
    assert launches == 1 + chunks * (3 + memset + group) + wgrad + 1 + (1 if bias else 0)


@pytest.mark.parametrize("what,d,ok", [
    # output pixels N*Ho*Wo (Ho, Wo come from offset, independent of x): 2^31 refused, 2^31 - 1 accepted
    ("pixels", dict(N=2, Cin=8, H=8, W=8, Cout=8, Ho=1 << 15, Wo=1 << 15), False),
    ("pixels", dict(N=(1 << 31) - 1, Cin=8, H=1, W=1, Cout=8, Ho=1, Wo=1), True),
    # input pixels N*H*W of the fused path's channels-last copy (Cout = 16: (Cin/group) * (Cout/group)
    # above 64, so not a direct plan, which reads x in place with 64-bit indices)
    ("x pixels", dict(N=2, Cin=8, H=1 << 15, W=1 << 15, Cout=16, Ho=4, Wo=4), False),
    # k-tiles of all tiles: 256 groups x (2^19 tiles of 128 pixels) x 16 k-tiles (4x4 taps, 64 channels)
    ("k-tiles", dict(N=1, Cin=16384, H=8, W=8, Cout=4096, Ho=8192, Wo=8192, kh=4, kw=4, group=256), False),
    ("k-tiles", dict(N=1, Cin=16384, H=8, W=8, Cout=4096, Ho=8184, Wo=8192, kh=4, kw=4, group=256), True),
])
def test_32bit_limits_at_2_pow_31(lib, what, d, ok):
    """The kernels index pixels, tiles and k-tiles with 32-bit integers; the
    planner refuses (MDCN_ERR_UNSUPPORTED, before anything runs) every call
    whose count of output pixels, input pixels or k-tiles reaches 2^31, and
    accepts the same shapes just below it."""
    group = d.pop("group", 1)
    h = handle(lib, padding=(0, 0), group=group)
    dd = dims(bias=False, group=group, **d)
    s, n = ws_size(lib, h, dd, _abi.MDCN_F16)
    assert s == (_abi.MDCN_OK if ok else _abi.MDCN_ERR_UNSUPPORTED), (what, s)
    lib.mdcn_destroy(h)
