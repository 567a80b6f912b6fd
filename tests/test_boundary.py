"""The C-ABI boundary on the host: the library builds and loads, exports every
entry point include/statekv.h declares, and rejects bad arguments before any
device work (no GPU needed)."""

import ctypes as C
import os
import re

import pytest

from kv_cache_compression_frame_gb300 import _native as N
from kv_cache_compression_frame_gb300 import build_lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "statekv.h")


@pytest.fixture(scope="module")
def lib():
    build_lib.build()
    return N.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(statekv_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(N.EXPORTS)


def test_status_strings(lib):
    for s in (0, -1, -2, -3, -4, -5, -6, -7):
        assert lib.statekv_status_string(s)
    assert lib.statekv_status_string(-99) == b"unknown status"


def _cfg(**kw):
    base = dict(num_streams=1, num_layers=1, num_q_heads=4, num_kv_heads=2,
                head_dim=64, frame_tokens=16, budget=32, max_frames=4,
                dtype=N.BF16, device=0, rope_theta=1e4, rope_alpha=1.0,
                rope_orig_ctx=0, position_offset=0)
    base.update(kw)
    return N.Config(**base)


@pytest.mark.parametrize("bad,want", [
    (dict(num_streams=0), N.E_INVALID_ARG),
    (dict(num_q_heads=3), N.E_INVALID_ARG),            # not a multiple of Hkv
    (dict(frame_tokens=0), N.E_INVALID_ARG),
    (dict(budget=-1), N.E_INVALID_ARG),
    (dict(dtype=7), N.E_INVALID_ARG),
    (dict(rope_theta=1.0), N.E_INVALID_ARG),
    (dict(rope_alpha=0.5), N.E_INVALID_ARG),
    (dict(rope_alpha=4.0, rope_orig_ctx=0), N.E_INVALID_ARG),
    (dict(position_offset=-1), N.E_INVALID_ARG),
    (dict(head_dim=96), N.E_UNSUPPORTED),
    (dict(budget=30000, max_frames=4096), N.E_UNSUPPORTED),   # selects over > 24576 rows
    (dict(budget=1 << 25), N.E_UNSUPPORTED),                    # no eviction, pool too large
    (dict(select_policy=7), N.E_INVALID_ARG),
    (dict(max_frames=1 << 30, frame_tokens=256), N.E_UNSUPPORTED),
])
def test_create_rejects_bad_config_before_device_work(lib, bad, want):
    h = C.c_void_p(123)
    assert lib.statekv_create(C.byref(_cfg(**bad)), C.byref(h)) == want
    assert h.value is None


def test_null_handle_and_pointers(lib):
    assert lib.statekv_create(None, None) == N.E_INVALID_ARG
    assert lib.statekv_destroy(None) == N.OK
    assert lib.statekv_prefill_frame(None, None, None, None, None, None) == N.E_INVALID_ARG
    assert lib.statekv_prefill_frame_host(None, None, None, None, None, None) == N.E_INVALID_ARG
    assert lib.statekv_prefill_frames_host(None, 1, None, None, None, None, None) == N.E_INVALID_ARG
    assert lib.statekv_reset(None) == N.E_INVALID_ARG
    assert lib.statekv_frame_index(None) == -1
    assert lib.statekv_set_frame_index(None, 0) == N.E_INVALID_ARG
    assert lib.statekv_check_device_status(None, None) == N.E_INVALID_ARG
    assert lib.statekv_profile_enable(None, 1) == N.E_INVALID_ARG
    assert lib.statekv_profile_kernels(None, 1) == N.E_INVALID_ARG
    k = C.c_void_p()
    assert lib.statekv_get_rotated_query(None, C.byref(k)) == N.E_INVALID_ARG
    assert lib.statekv_get_compressed(None, 0, 0, None, None, None, None, None) == N.E_INVALID_ARG
    assert lib.statekv_get_detailed(None, 0, 0, None, None, None, None) == N.E_INVALID_ARG
    assert lib.statekv_get_scores(None, 0, 0, None, None, None, None) == N.E_INVALID_ARG
    assert lib.statekv_set_compressed(None, 0, 0, None, None, None, 0, None) == N.E_INVALID_ARG
    assert lib.statekv_profile_read(None, 0, None, None) == N.E_INVALID_ARG
    assert lib.statekv_decode(None, 1, None, None, None, None, None) == N.E_INVALID_ARG
    assert lib.statekv_text_tokens(None) == -1


def _static(**kw):
    # a valid-looking request with 16-byte aligned fake pointers: every check
    # below fires on the host, before any device work
    a = dict(q_rot=16, pool_k=32, pool_v=48, units=2, group=2, frame_tokens=64, head_dim=128,
             pool_rows=256, compressed=128, logit_scale=0.1, dtype=N.BF16, o=64, scores=80,
             status=96, stream=None)
    a.update(kw)
    st = a["status"]
    return (a["q_rot"], a["pool_k"], a["pool_v"], a["units"], a["group"], a["frame_tokens"],
            a["head_dim"], a["pool_rows"], a["compressed"], a["logit_scale"], a["dtype"], a["o"],
            C.cast(C.c_void_p(a["scores"]), C.POINTER(C.c_float)) if a["scores"] else None,
            st, a["stream"])


@pytest.mark.parametrize("bad,want", [
    (dict(q_rot=None), N.E_INVALID_ARG),
    (dict(pool_k=40), N.E_INVALID_ARG),            # not 16-byte aligned
    (dict(scores=None), N.E_INVALID_ARG),
    (dict(status=None), N.E_INVALID_ARG),          # status is required
    (dict(status=98), N.E_INVALID_ARG),            # status not 4-byte aligned
    (dict(units=0), N.E_INVALID_ARG),
    (dict(frame_tokens=0), N.E_INVALID_ARG),       # empty frame
    (dict(pool_rows=100), N.E_INVALID_ARG),        # pool shorter than compressed + frame
    (dict(logit_scale=0.0), N.E_INVALID_ARG),
    (dict(dtype=9), N.E_INVALID_ARG),
    (dict(head_dim=96), N.E_UNSUPPORTED),
    (dict(pool_rows=30000, compressed=29000), N.E_UNSUPPORTED),   # beyond the selection's rows
    (dict(group=1024, frame_tokens=128), N.E_UNSUPPORTED),        # G*T > 65536
])
def test_static_entry_rejects_bad_requests_on_the_host(lib, bad, want):
    assert lib.statekv_attend_scores_static(*_static(**bad)) == want


def test_python_config_mirror_matches_shapes():
    from synth import SHAPES
    from kv_cache_compression_frame_gb300 import StateKVConfig
    c = StateKVConfig.from_shape(SHAPES["internvl3_2b_stack"])
    cc = c._c(0)
    assert (cc.num_layers, cc.num_q_heads, cc.num_kv_heads, cc.head_dim) == (28, 12, 2, 128)
    assert (cc.frame_tokens, cc.budget, cc.max_frames) == (256, 4096, 512)
    assert cc.rope_alpha == 4.0 and cc.rope_orig_ctx == 32960 and cc.dtype == N.BF16
