"""ctypes loader for the C ABI in include/ssd.h (libssd_gb300.so, built in-tree).

Argument marshalling only.  There is no fallback: if the library is missing
or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libssd_gb300.so")

SSD_OK = 0
SSD_ERR_INVALID_ARG = 1
SSD_ERR_UNSUPPORTED = 2
SSD_ERR_CUDA = 3
SSD_ERR_NO_MEMORY = 4
SSD_ERR_TIMEOUT = 5
SSD_ERR_SCRATCH_TOO_SMALL = 6
SSD_ERR_RANGE = 7
SSD_NOALLOC_SCRATCH_BYTES = 64 << 20

# name -> (restype, argtypes); the exported surface of include/ssd.h
_p, _i, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
SIGNATURES = {
    "ssd_status_string": (ctypes.c_char_p, [_i]),
    "ssd_chunk_cumsum": (_i, [_p, _p, _i, _i, _i, _i, _p, _p, _p]),
    "ssd_chunk_state": (_i, [_p, _p, _p, _p] + [_i] * 7 + [_p, _p]),
    "ssd_state_passing": (_i, [_p, _p, _p] + [_i] * 6 + [_p, _p, _p]),
    "ssd_chunk_scan": (_i, [_p] * 7 + [_i] * 7 + [_p, _p]),
    "ssd_forward": (_i, [_p] * 7 + [_i] * 7 + [_p, _p, _p]),
    "ssd_forward_noalloc": (_i, [_p] * 7 + [_i] * 7 + [_p, _p, _p]),
    "ssd_forward_heads": (_i, [_p] * 7 + [_i] * 9 + [_p, _p, _p]),
    "ssd_partition_heads": (_i, [_i] * 4 + [_p, _p]),
    "ssd_step": (_i, [_p] * 7 + [_i] * 5 + [_p, _p]),
    "ssd_step_multi": (_i, [_p] * 7 + [_i] * 6 + [_p, _p]),
    "ssd_forward_plan": (_i, [_i] * 7 + [_p, _p, _p]),
    "ssd_forward_ex": (_i, [_p] * 7 + [_i] * 7 + [_p, _p, _p, _p]),
    "ssd_step_ex": (_i, [_p] * 7 + [_i] * 5 + [_p, _p, _p]),
    "ssd_backward": (_i, [_p] * 9 + [_i] * 7 + [_p] * 8),
    "ssd_get_device_error": (_i, []),
    "ssd_debug_set_wait_limit_ns": (_i, [ctypes.c_ulonglong]),
    "ssd_debug_stall": (_i, [_i]),
    "ssd_profile_enable": (_i, [_i]),
    "ssd_profile_reset": (_i, []),
    "ssd_profile_read": (_i, [_p, _p, _i, _p]),
    "ssd_kernel_name": (ctypes.c_char_p, [_i]),
    "ssd_launch_count": (ctypes.c_longlong, []),
}



class InputOptions(ctypes.Structure):
    """struct ssd_input_options (field order and types as in include/ssd.h)."""
    _fields_ = [("dt_bias", ctypes.c_void_p), ("dt_softplus", ctypes.c_int), ("dt_limit", ctypes.c_int),
                ("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float), ("D_per_channel", ctypes.c_int),
                ("z", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


class SSDError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed with status {status}: {msg}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load libssd_gb300.so once; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"SSD CUDA library not found at {LIB_PATH}; build it with "
                    "`python -m state_space_sequence_ssd_gb300.build` (no CPU fallback exists)")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(l, name)
                fn.restype = res
                fn.argtypes = args
            _lib = l
    return _lib


def status_string(status: int) -> str:
    return lib().ssd_status_string(status).decode()


def check(fn: str, status: int) -> None:
    if status != SSD_OK:
        raise SSDError(fn, status, status_string(status))
