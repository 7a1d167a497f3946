"""ctypes declarations of libssd.so (the C ABI in include/ssd.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation anywhere in this package.
"""

from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libssd.so")

SSD_OK = 0
STATUS_NAMES = {0: "SSD_OK", 1: "SSD_ERR_INVALID_ARG", 2: "SSD_ERR_UNSUPPORTED",
                3: "SSD_ERR_ALIGNMENT", 4: "SSD_ERR_WORKSPACE", 5: "SSD_ERR_CUDA",
                6: "SSD_ERR_TIMEOUT", 7: "SSD_ERR_DEVICE"}
DTYPE_F32 = 0
DTYPE_BF16 = 1


class Problem(ctypes.Structure):
    """Mirror of ssd_problem_t."""
    _fields_ = [
        ("batch", ctypes.c_int64),
        ("seqlen", ctypes.c_int64),
        ("nheads", ctypes.c_int32),
        ("headdim", ctypes.c_int32),
        ("dstate", ctypes.c_int32),
        ("ngroups", ctypes.c_int32),
        ("chunk_size", ctypes.c_int32),
        ("nseq", ctypes.c_int32),
        ("delta_init", ctypes.c_float),
        ("dtype", ctypes.c_int32),
    ]


class SSDError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s" % (where, STATUS_NAMES.get(status, str(status))))


_lib = None

_VP = ctypes.c_void_p
_PP = ctypes.POINTER(Problem)
_SZ = ctypes.c_size_t
_SIGS = {
    "ssd_workspace_size": (ctypes.c_int, [_PP, ctypes.c_int, ctypes.POINTER(_SZ)]),
    "ssd_forward": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "ssd_backward": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                    _VP, _SZ, _VP]),
    "ssd_backward_after_forward": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                                  _VP, _VP, _VP, _SZ, _VP]),
    "ssd_forward_state": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _SZ,
                                         _VP]),
    "ssd_backward_state": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                          _VP, _VP, _VP, ctypes.c_int, _VP, _SZ, _VP]),
    "ssd_decode_step": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "ssd_bidirectional_workspace_size": (ctypes.c_int, [_PP, ctypes.c_int, ctypes.POINTER(_SZ)]),
    "ssd_bidirectional_forward": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                                 _VP, _SZ, _VP]),
    "ssd_bidirectional_backward": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                                  _VP, _VP, _VP, _SZ, _VP]),
    "ssd_forward_noalloc": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "ssd_forward_noalloc_status": (ctypes.c_int, [_VP, ctypes.POINTER(ctypes.c_int32)]),
    "ssd_step_host_size": (ctypes.c_int, [_PP, ctypes.POINTER(_SZ)]),
    "ssd_step_host": (ctypes.c_int, [_PP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                     _VP, _VP, _VP, _SZ, _VP]),
    "ssd_device_status": (ctypes.c_int, [_VP, _VP, ctypes.POINTER(ctypes.c_int32)]),
    "ssd_dispatch_path": (ctypes.c_char_p, [_PP, ctypes.c_int]),
    "ssd_last_launch_count": (ctypes.c_int, []),
    "ssd_profiler_enable": (ctypes.c_int, [ctypes.c_int]),
    "ssd_profiler_only": (ctypes.c_int, [ctypes.c_char_p]),
    "ssd_profiler_reset": (None, []),
    "ssd_profiler_count": (ctypes.c_int, []),
    "ssd_profiler_entry": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_char_p),
                                          ctypes.POINTER(ctypes.c_int64),
                                          ctypes.POINTER(ctypes.c_double)]),
    "ssd_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "ssd_version": (ctypes.c_int, []),
}


def lib():
    """The loaded libssd.so with argument types declared."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libssd.so is not built (%s); run state_space_model_ssd_gb300/build.py or "
                "__graft_entry__.build()" % LIB_PATH)
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def check(status: int, where: str) -> None:
    if status != SSD_OK:
        raise SSDError(status, where)
