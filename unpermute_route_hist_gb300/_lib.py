"""ctypes loader for libgg.so and the signatures of its C ABI (include/gg.h).

Loading fails loudly when the library has not been built: there is no CPU
fallback for any entry point.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libgg.so")

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_sz = ctypes.c_size_t
_cstr = ctypes.c_char_p

# name -> (restype, argtypes); the order follows include/gg.h
SIGNATURES = {
    "gg_status_string": (_cstr, [_int]),
    "gg_device_status_string": (_cstr, [_int]),
    "gg_last_cuda_error": (_cstr, []),
    "gg_workspace_size": (_sz, [_int, _i64, _int, _int, _i64, _i64, _int]),
    "gg_read_status": (_int, [_vp, _vp, _vp]),
    "gg_set_gemm_schedule": (_int, [_int]),
    "gg_selftest_bounded_wait": (_int, [_vp, _vp, ctypes.c_uint64, _vp]),
    "gg_route_workspace_size": (_sz, [_i64, _int, _int]),
    "gg_route_hist_offsets": (_int, [_vp, _i64, _int, _int, _int, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                     _vp, _vp]),
    "gg_route_hist_offsets_noalloc": (_int, [_vp, _i64, _int, _int, _int, _vp, _vp, _vp, _vp, _vp,
                                             _vp, _vp]),
    "gg_permute": (_int, [_vp, _vp, _i64, _int, _i64, _vp, _vp, _vp]),
    "gg_unpermute_combine": (_int, [_vp, _vp, _vp, _i64, _int, _i64, _vp, _vp, _vp]),
    "gg_unpermute_combine_bwd": (_int, [_vp, _vp, _vp, _vp, _i64, _int, _i64, _vp, _vp, _vp, _vp]),
    "gg_forward": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _i64, _i64, _int, _int, _int,
                          _vp, _vp, _vp]),
    "gg_forward_combine": (_int, [_vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _i64, _i64, _int, _vp,
                                  _vp, _sz, _vp, _vp]),
    "gg_forward_swiglu": (_int, [_vp, _vp, _vp, _vp, _i64, _int, _int, _i64, _i64, _int, _vp, _vp,
                                 _vp, _vp]),
    "gg_swiglu_bwd": (_int, [_vp, _vp, _i64, _i64, _vp, _vp]),
    "gg_backward_dX": (_int, [_vp, _vp, _vp, _vp, _i64, _int, _int, _i64, _i64, _int, _int, _vp, _vp,
                              _vp, _vp]),
    "gg_backward_dX_swiglu": (_int, [_vp, _vp, _vp, _i64, _int, _int, _i64, _i64, _vp, _vp, _vp,
                                     _vp]),
    "gg_backward_dW": (_int, [_vp, _vp, _vp, _vp, _i64, _int, _int, _i64, _i64, _int, _int, _vp, _vp,
                              _sz, _vp, _vp]),
    "gg_dual_asym": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _int, _int,
                            _vp, _vp]),
    "gg_ep_plan": (_int, [_vp, _vp, _int, _int, _vp, _vp, _vp, _vp, _i64]),
    "gg_ep_recv_map": (_int, [_vp, _int, _int, _i64, _vp, _vp, _vp]),
}

GG_OK = 0
GG_ERR_INVALID_ARG = -1
GG_ERR_UNSUPPORTED = -2
GG_ERR_CUDA = -3
GG_ERR_DEVICE_CHECK = -4
GG_ERR_TIMEOUT = -5
GG_ERR_WORKSPACE = -6
GG_DEV_OK = 0
GG_DEV_BAD_EXPERT_ID = 1
GG_DEV_BAD_ROW_INDEX = 2
GG_DEV_SIZES_MISMATCH = 3
GG_DEV_TIMEOUT = 4
GG_MAX_EXPERTS = 2048
GG_MAX_TOPK = 64
GG_ROUTE_NOALLOC_SCRATCH_BYTES = 1 << 20
GG_COMBINE_BF16_MAX_TOPK = 16
GG_OP_ROUTE = 1
GG_OP_BACKWARD_DW = 2
GG_OP_FORWARD_COMBINE = 3
GG_PERMUTE_X = 1
GG_PERMUTE_Y = 2
GG_SCHEDULE_AUTO = 0
GG_SCHEDULE_STATIC = 1
GG_SCHEDULE_DYNAMIC = 2

_lock = threading.Lock()
_lib = None


class GGError(RuntimeError):
    def __init__(self, fn: str, code: int, detail: str = ""):
        self.code = code
        super().__init__("%s failed: %s (%d)%s" % (fn, status_string(code), code,
                                                   (": " + detail) if detail else ""))


def load() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libgg.so is not built (%s); run `python -c 'import __graft_entry__ as g; g.build()'`"
                % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().gg_status_string(int(code)).decode()


def device_status_string(code: int) -> str:
    return load().gg_device_status_string(int(code)).decode()


def last_cuda_error() -> str:
    return load().gg_last_cuda_error().decode()


def check(fn: str, rc: int) -> None:
    if rc != GG_OK:
        raise GGError(fn, rc, last_cuda_error() if rc == GG_ERR_CUDA else "")
