"""ctypes declarations of libmdcn's C ABI (include/mdcn.h). Marshalling only."""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmdcn.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "mdcn.h")

MDCN_OK = 0
MDCN_ERR_NULL = 1
MDCN_ERR_ATTR = 2
MDCN_ERR_SHAPE = 3
MDCN_ERR_DTYPE = 4
MDCN_ERR_ALIGN = 5
MDCN_ERR_WORKSPACE = 6
MDCN_ERR_ARCH = 7
MDCN_ERR_CUDA = 8
MDCN_ERR_TIMEOUT = 9
MDCN_ERR_UNSUPPORTED = 10

MDCN_F32 = 0
MDCN_F16 = 1
MDCN_BF16 = 2

i64 = ctypes.c_int64
vp = ctypes.c_void_p


class mdcn_attrs(ctypes.Structure):
    _fields_ = [("stride", i64 * 2), ("padding", i64 * 2), ("dilation", i64 * 2), ("group", i64),
                ("deformable_group", i64)]


class mdcn_tuning(ctypes.Structure):
    _fields_ = [("stages", ctypes.c_int32), ("tile_mode", ctypes.c_int32), ("max_ctas", ctypes.c_int32),
                ("kgroups", ctypes.c_int32), ("a_operand", ctypes.c_int32), ("ntile", ctypes.c_int32),
                ("path", ctypes.c_int32)]


class mdcn_plan_info(ctypes.Structure):
    _fields_ = [("tiles", i64), ("ktiles_per_tile", i64), ("ktiles_per_cta", i64), ("ctas", ctypes.c_int32),
                ("split", ctypes.c_int32), ("stages", ctypes.c_int32), ("kgroups", ctypes.c_int32),
                ("tile_mode", ctypes.c_int32), ("launches", ctypes.c_int32), ("a_operand", ctypes.c_int32),
                ("path", ctypes.c_int32)]


class mdcn_dims(ctypes.Structure):
    _fields_ = [("x", i64 * 4), ("offset", i64 * 4), ("mask", i64 * 4), ("weight", i64 * 4), ("bias", i64)]


_lock = threading.Lock()
_lib = None


def declared_functions(header: str = HEADER):
    """Names of the functions include/mdcn.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mdcn_\w+)\s*\(", text)))


def load(path: str = LIB_PATH):
    """Loads libmdcn.so (built by ``build.py``). Raises if it is missing:
    there is no fallback implementation."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libmdcn.so not built ({path}); run modulated_deformable_convolution_gb300.build")
        lib = ctypes.CDLL(path)
        st = ctypes.c_int
        lib.mdcn_create.argtypes = [ctypes.POINTER(mdcn_attrs), ctypes.POINTER(vp)]
        lib.mdcn_create.restype = st
        lib.mdcn_create_tuned.argtypes = [ctypes.POINTER(mdcn_attrs), ctypes.POINTER(mdcn_tuning), ctypes.POINTER(vp)]
        lib.mdcn_create_tuned.restype = st
        lib.mdcn_destroy.argtypes = [vp]
        lib.mdcn_destroy.restype = st
        lib.mdcn_output_dims.argtypes = [vp, ctypes.POINTER(mdcn_dims), ctypes.POINTER(i64)]
        lib.mdcn_output_dims.restype = st
        lib.mdcn_workspace_size.argtypes = [vp, ctypes.POINTER(mdcn_dims), ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)]
        lib.mdcn_workspace_size.restype = st
        fwd = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, ctypes.POINTER(mdcn_dims), ctypes.c_int, vp]
        lib.mdcn_forward.argtypes = fwd
        lib.mdcn_forward.restype = st
        lib.mdcn_prepare_input.argtypes = [vp, vp, vp, ctypes.c_size_t, ctypes.POINTER(mdcn_dims), ctypes.c_int, vp]
        lib.mdcn_prepare_input.restype = st
        lib.mdcn_pack_weight.argtypes = [vp, vp, vp, ctypes.c_size_t, ctypes.POINTER(mdcn_dims), ctypes.c_int, vp]
        lib.mdcn_pack_weight.restype = st
        lib.mdcn_forward_prepared.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_size_t, ctypes.POINTER(mdcn_dims),
                                              ctypes.c_int, vp]
        lib.mdcn_forward_prepared.restype = st
        lib.mdcn_im2col_gemm_workspace_size.argtypes = [vp, ctypes.POINTER(mdcn_dims), ctypes.c_int,
                                                        ctypes.POINTER(ctypes.c_size_t)]
        lib.mdcn_im2col_gemm_workspace_size.restype = st
        lib.mdcn_forward_im2col_gemm.argtypes = fwd
        lib.mdcn_forward_im2col_gemm.restype = st
        lib.mdcn_query_plan.argtypes = [vp, ctypes.POINTER(mdcn_dims), ctypes.c_int, ctypes.POINTER(mdcn_plan_info)]
        lib.mdcn_query_plan.restype = st
        lib.mdcn_pack_workspace_size.argtypes = [vp, ctypes.POINTER(mdcn_dims), ctypes.c_int,
                                                 ctypes.POINTER(ctypes.c_size_t)]
        lib.mdcn_pack_workspace_size.restype = st
        lib.mdcn_forward_pack.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                          ctypes.POINTER(mdcn_dims), ctypes.c_int, vp]
        lib.mdcn_forward_pack.restype = st
        lib.mdcn_host_buffer_size.argtypes = [vp, ctypes.POINTER(mdcn_dims), ctypes.c_int,
                                              ctypes.POINTER(ctypes.c_size_t)]
        lib.mdcn_host_buffer_size.restype = st
        lib.mdcn_forward_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, ctypes.POINTER(mdcn_dims),
                                          ctypes.c_int, vp]
        lib.mdcn_forward_host.restype = st
        lib.mdcn_backward_workspace_size.argtypes = [vp, ctypes.POINTER(mdcn_dims), ctypes.c_int,
                                                     ctypes.POINTER(ctypes.c_size_t)]
        lib.mdcn_backward_workspace_size.restype = st
        lib.mdcn_backward_launches.argtypes = [vp, ctypes.POINTER(mdcn_dims), ctypes.c_int,
                                               ctypes.POINTER(ctypes.c_int32)]
        lib.mdcn_backward_launches.restype = st
        lib.mdcn_backward.argtypes = [vp] * 12 + [ctypes.c_size_t, ctypes.POINTER(mdcn_dims), ctypes.c_int, vp]
        lib.mdcn_backward.restype = st
        lib.mdcn_query_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.mdcn_query_status.restype = st
        lib.mdcn_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint32, vp]
        lib.mdcn_selftest_wait_timeout.restype = st
        lib.mdcn_last_cuda_error.argtypes = []
        lib.mdcn_last_cuda_error.restype = ctypes.c_int
        lib.mdcn_status_string.argtypes = [ctypes.c_int]
        lib.mdcn_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib
