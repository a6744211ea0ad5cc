"""ctypes loader for the CUDA library ``lib/libmxfp4_expert_linear.so``.

There is no fallback: if the library has not been built, every call raises.
Build it with ``python -m mxfp4_routed_expert_route_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmxfp4_expert_linear.so")

# Values of the #defines in include/mxfp4_expert_linear.h.
OK = 0
ERR_INVALID_ARGUMENT = -1
ERR_UNSUPPORTED_DTYPE = -2
ERR_ALIAS = -3
ERR_WORKSPACE = -4
ERR_CUDA = -5
ERR_TOO_LARGE = -6
STAGE_ROUTE = 0
STAGE_LINEAR = 1
STAGE_COMBINE = 2
STAGE_GATHER = 3
NUM_STAGES = 4
PATH_GEMV = 0
PATH_GEMM = 1
DTYPE_F32 = 0
DTYPE_BF16 = 1
INDEX_I32 = 0
INDEX_I64 = 1

# Every symbol the header declares: (name, restype, argtypes).
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_SZ = ctypes.c_size_t
SIGNATURES = {
    "mxfp4_expert_linear": (_INT, [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64,
                                   _I64, _I64, _INT, _INT, _P]),
    "mxfp4_expert_linear_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I64, _INT]),
    "mxfp4_expert_linear_with_workspace": (_INT, [_P, _P, _P, _P, _P, _P, _P, _I64,
                                                  _I64, _I64, _I64, _I64, _INT, _INT,
                                                  _P, _SZ, _P]),
    "mxfp4_expert_linear_static_scratch": (_INT, [_P, _P, _P, _P, _P, _P, _P, _I64,
                                                  _I64, _I64, _I64, _I64, _INT, _INT,
                                                  _P]),
    "mxfp4_expert_linear_static_scratch_bytes": (_SZ, []),
    "mxfp4el_device_errors": (_INT, [_P, ctypes.POINTER(_I64)]),
    "mxfp4el_wait_timeouts": (_INT, [_P, ctypes.POINTER(_I64)]),
    "mxfp4el_set_stage_events": (_INT, [_INT, _P, _P]),
    "mxfp4el_kernel_launches": (_I64, []),
    "mxfp4el_linear_path": (_INT, [_I64, _I64, _I64, _I64, _I64, _INT]),
    "mxfp4el_status_string": (ctypes.c_char_p, [_INT]),
    "mxfp4el_version": (_INT, []),
    "mxfp4_router_topk": (_INT, [_P, _P, _I64, _I64, _I64, ctypes.c_float, _P, _P, _P]),
    "mxfp4_expert_linear_routed": (_INT, [_P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P,
                                          _P, _I64, _I64, _I64, _I64, _I64, _INT, _P]),
    "mxfp4_swiglu_expert": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64,
                                   _I64, _I64, _I64, _INT, _INT, _P]),
    "mxfp4_swiglu_expert_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I64, _I64, _INT]),
    "mxfp4_swiglu_expert_with_workspace": (_INT, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64,
                                                  _I64, _I64, _I64, _I64, _I64, _INT, _INT,
                                                  _P, _SZ, _P]),
    "mxfp4_expert_linear_prepared_bytes": (_SZ, [_I64, _I64, _I64]),
    "mxfp4_expert_linear_prepare": (_INT, [_P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "mxfp4_expert_linear_prepared": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                            _I64, _INT, _INT, _P]),
    "mxfp4_expert_linear_prepared_workspace_size": (_SZ, [_I64, _I64, _I64, _I64, _I64,
                                                          _INT]),
    "mxfp4_expert_linear_prepared_with_workspace": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64,
                                                           _I64, _I64, _I64, _INT, _INT, _P,
                                                           _SZ, _P]),
}

_lock = threading.Lock()
_lib = None


class LibraryNotBuilt(RuntimeError):
    pass


def load(path: str = LIB_PATH):
    """Load the CUDA library once; raise if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise LibraryNotBuilt(
                f"{path} is missing: build the CUDA library first "
                "(python -m mxfp4_routed_expert_route_gb300.build)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class MXFP4Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        text = load().mxfp4el_status_string(status).decode()
        super().__init__(f"{what}: {text} (status {status})" if what else text)


def check(status: int, what: str = "") -> None:
    if status != OK:
        raise MXFP4Error(status, what)
