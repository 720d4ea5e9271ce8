"""ctypes view of ``libbeamboundary.so`` (the C ABI in ``include/beam_boundary.h``)."""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbeamboundary.so")

BEAM_OK = 0
BEAM_ERR_NULL = 1
BEAM_ERR_ALIGN = 2
BEAM_ERR_SHAPE = 3
BEAM_ERR_ARG = 4
BEAM_ERR_ALIAS = 5
BEAM_ERR_CUDA = 6
BEAM_ERR_TIMEOUT = 7
BEAM_ERR_DEVICE = 8
BEAM_MAX_D = 32768
BEAM_MOE_TOPK = 8
BEAM_ROUTE_EXPERTS = 256
BEAM_ROUTE_MAX_TOPK = 16
BEAM_QK_HEAD_DIM = 128
BEAM_QK_ROPE = 0
BEAM_QK_SSMAX = 1
BEAM_OPT_FORCE_EXACT_SUM = 0x1
BEAM_OPT_TEST_WAIT_TIMEOUT = 0x2
BEAM_OPT_PDL = 0x4


class LaunchOpts(ctypes.Structure):
    """``beam_launch_opts``: flags, vectors per thread, CTAs per SM, L2 prefetch distance,
    ring stages (0 = automatic for each)."""
    _fields_ = [("flags", ctypes.c_uint32), ("vec_per_thread", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("prefetch_rows", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("reserved", ctypes.c_int32 * 3)]


# name -> (restype, argtypes)
_vp, _i32, _i64, _f32, _u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_uint32
_OPTS = ctypes.POINTER(LaunchOpts)
SIGNATURES = {
    "beam_boundary_fused": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _f32, _i64, _i32, _vp]),
    "beam_moe_combine_boundary": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _f32, _i64, _i32, _vp]),
    "beam_boundary_fused_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _f32, _i64, _i32, _vp, _OPTS]),
    "beam_moe_combine_boundary_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _f32, _i64, _i32, _vp,
                                            _OPTS]),
    "beam_moe_combine_boundary_scaled": (_i32, [_vp, _vp, _vp, _vp, _f32, _vp, _vp, _i32, _f32, _i64,
                                                 _i32, _vp]),
    "beam_boundary_fused_nvfp4": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _f32, _i64, _i32, _f32, _vp,
                                          _vp, _vp]),
    "beam_moe_combine_boundary_nvfp4": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _f32, _i64, _i32,
                                                _f32, _vp, _vp, _vp]),
    "beam_boundary_fused_host": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _f32, _i64, _i32, _vp]),
    "beam_moe_combine_boundary_host": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _f32, _i64, _i32,
                                               _vp]),
    "beam_moe_route": (_i32, [_vp, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _f32, _vp, _vp]),
    "beam_moe_route_ex": (_i32, [_vp, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _f32, _vp, _vp, _u32]),
    "beam_router_sigmoid": (_i32, [_vp, _vp, _vp, _i64]),
    "beam_router_sigmoid_fast": (_i32, [_vp, _vp, _vp, _i64]),
    "beam_qk_norm": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _f32,
                             _i32]),
    "beam_qk_norm_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32,
                                _f32, _i32, _u32]),
    "beam_sync_status": (_i32, [_vp]),
    "beam_exact_sum_count": (_i32, [_vp, ctypes.POINTER(ctypes.c_uint64), _i32]),
    "beam_status_string": (ctypes.c_char_p, [_i32]),
    "beam_version": (_i32, []),
}

_lock = threading.Lock()
_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the library (built by ``sandwich_norm_residual_gb300.build``); no fallback."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(
                f"{p} is missing: build it with `python -m sandwich_norm_residual_gb300.build` "
                "(nvcc for sm_103a). There is no CPU or PyTorch fallback.")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib
