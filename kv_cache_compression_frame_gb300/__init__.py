"""StateKV streaming video prefill for GB300 (sm_103a).

A C-ABI CUDA library (libstatekv.so, include/statekv.h) with a thin Python
binding.  Build it with ``python -m kv_cache_compression_frame_gb300.build_lib``.
"""

from .statekv import StateKV, StateKVConfig  # noqa: F401
from ._native import StateKVError, load as load_library  # noqa: F401

__all__ = ["StateKV", "StateKVConfig", "StateKVError", "load_library"]
