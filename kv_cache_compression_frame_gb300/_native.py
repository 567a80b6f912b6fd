"""ctypes view of libstatekv's C ABI (include/statekv.h).

Only argument marshalling lives here; every step of the prefill path runs in
the library's CUDA kernels.  Loading fails loudly if the library was not
built: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libstatekv.so")

OK = 0
E_INVALID_ARG = -1
E_UNSUPPORTED = -2
E_CAPACITY = -3
E_OOM = -4
E_CUDA = -5
E_TIMEOUT = -6
E_DEVICE = -7

BF16 = 0
F32 = 1

KERNEL_ROPE_TABLE = 0
KERNEL_ROPE = 1
KERNEL_ATTENTION = 2
KERNEL_SELECT = 3
KERNEL_NAMES = ("rope_table", "rope", "attention", "select")

EXPORTS = (
    "statekv_status_string", "statekv_create", "statekv_destroy",
    "statekv_prefill_frame", "statekv_prefill_frame_host", "statekv_prefill_frames_host",
    "statekv_get_compressed", "statekv_get_detailed", "statekv_frame_index",
    "statekv_reset", "statekv_check_device_status", "statekv_get_scores",
    "statekv_get_rotated_query", "statekv_set_frame_index",
    "statekv_set_compressed", "statekv_profile_enable", "statekv_profile_read",
    "statekv_profile_kernels",
    "statekv_attend_scores_static", "statekv_decode", "statekv_text_tokens",
)


class Config(C.Structure):
    _fields_ = [
        ("num_streams", C.c_int32), ("num_layers", C.c_int32),
        ("num_q_heads", C.c_int32), ("num_kv_heads", C.c_int32),
        ("head_dim", C.c_int32), ("frame_tokens", C.c_int32),
        ("budget", C.c_int32), ("max_frames", C.c_int32),
        ("dtype", C.c_int32), ("device", C.c_int32),
        ("rope_theta", C.c_double), ("rope_alpha", C.c_double),
        ("rope_orig_ctx", C.c_int64), ("position_offset", C.c_int64),
        ("select_policy", C.c_int32),
    ]


class StateKVError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None
_P = C.c_void_p
_PP = C.POINTER(C.c_void_p)


def load() -> C.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -m kv_cache_compression_frame_gb300.build_lib`")
    lib = C.CDLL(LIB_PATH)
    h = _P
    sig = {
        "statekv_status_string": (C.c_char_p, [C.c_int]),
        "statekv_create": (C.c_int, [C.POINTER(Config), C.POINTER(h)]),
        "statekv_destroy": (C.c_int, [h]),
        "statekv_prefill_frame": (C.c_int, [h, _P, _P, _P, _P, _P]),
        "statekv_prefill_frame_host": (C.c_int, [h, _P, _P, _P, _P, _P]),
        "statekv_prefill_frames_host": (C.c_int, [h, C.c_int32, _P, _P, _P, _P, _P]),
        "statekv_get_compressed": (C.c_int, [h, C.c_int32, C.c_int32, _PP, _PP, _PP,
                                             C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
        "statekv_get_detailed": (C.c_int, [h, C.c_int32, C.c_int32, _PP, _PP,
                                           C.POINTER(C.c_int64), C.POINTER(C.c_int64)]),
        "statekv_frame_index": (C.c_int64, [h]),
        "statekv_decode": (C.c_int, [h, C.c_int32, _P, _P, _P, _P, _P]),
        "statekv_text_tokens": (C.c_int64, [h]),
        "statekv_reset": (C.c_int, [h]),
        "statekv_check_device_status": (C.c_int, [h, _P]),
        "statekv_get_scores": (C.c_int, [h, C.c_int32, C.c_int32, _PP, _PP,
                                         C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
        "statekv_get_rotated_query": (C.c_int, [h, _PP]),
        "statekv_set_frame_index": (C.c_int, [h, C.c_int64]),
        "statekv_set_compressed": (C.c_int, [h, C.c_int32, C.c_int32, _P, _P, _P,
                                             C.c_int32, _P]),
        "statekv_profile_enable": (C.c_int, [h, C.c_int]),
        "statekv_profile_kernels": (C.c_int, [h, C.c_uint32]),
        "statekv_profile_read": (C.c_int, [h, C.c_int32, C.POINTER(C.c_double),
                                           C.POINTER(C.c_int64)]),
        "statekv_attend_scores_static": (C.c_int, [_P, _P, _P, C.c_int32, C.c_int32,
                                                   C.c_int32, C.c_int32, C.c_int32,
                                                   C.c_int32, C.c_double, C.c_int32,
                                                   _P, _P, _P, _P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().statekv_status_string(status).decode()
    except RuntimeError:
        return f"status {status}"


def check(status: int, what: str) -> None:
    if status != OK:
        raise StateKVError(status, what)
