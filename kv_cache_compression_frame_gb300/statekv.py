"""Python binding of libstatekv: StateKV streaming video prefill on GB300.

Thin marshalling over the C ABI declared in include/statekv.h.  PyTorch is
used only for device memory and CUDA streams; each step runs in the
library's sm_103a kernels.  See the header for the method ("Linear Scaling
Video VLMs for Long Video Understanding", 方法详解 / 关键设计 1-3) and for the
meaning, layout and ownership of every argument.
"""

from __future__ import annotations

import ctypes as C
from dataclasses import dataclass, asdict

import torch

from . import _native as N

_DTYPES = {"bf16": (N.BF16, torch.bfloat16), "f32": (N.F32, torch.float32)}
_POLICIES = {"topb": 0, "window": 1}


@dataclass
class StateKVConfig:
    """Mirror of ``statekv_config``."""
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    frame_tokens: int
    budget: int
    max_frames: int
    num_streams: int = 1
    num_layers: int = 1
    dtype: str = "bf16"
    rope_theta: float = 1e6
    rope_alpha: float = 1.0
    rope_orig_ctx: int = 0
    position_offset: int = 0
    select_policy: str = "topb"      # "topb" (StateKV) or "window" (sliding-window baseline)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @classmethod
    def from_shape(cls, sh, **over) -> "StateKVConfig":
        """From a workload shape (synth.WorkloadShape or anything with the
        same attribute names)."""
        kw = dict(num_streams=sh.streams, num_layers=sh.layers,
                  num_q_heads=sh.q_heads, num_kv_heads=sh.kv_heads,
                  head_dim=sh.head_dim, frame_tokens=sh.frame_tokens,
                  budget=sh.budget, max_frames=sh.frames, dtype=sh.dtype,
                  rope_theta=sh.rope_theta, rope_alpha=sh.rope_alpha,
                  rope_orig_ctx=sh.rope_orig_ctx)
        kw.update(over)
        return cls(**kw)

    def _c(self, device: int) -> N.Config:
        if self.dtype not in _DTYPES:
            raise ValueError(f"dtype must be one of {list(_DTYPES)}")
        if self.select_policy not in _POLICIES:
            raise ValueError(f"select_policy must be one of {list(_POLICIES)}")
        d = asdict(self)
        d["dtype"] = _DTYPES[self.dtype][0]
        d["select_policy"] = _POLICIES[self.select_policy]
        return N.Config(device=device, **d)


class _DevArray:
    """Borrowed device memory described by __cuda_array_interface__."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {
            "shape": tuple(int(s) for s in shape), "typestr": typestr,
            "data": (int(ptr), False), "version": 3, "strides": None}


def _stream_ptr(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


class StateKV:
    """One handle: the compressed and detailed states of every (stream,
    layer, KV head) of a configuration, on one CUDA device."""

    def __init__(self, cfg: StateKVConfig, device: int | torch.device | None = None):
        lib = N.load()
        if device is None:
            idx = torch.cuda.current_device()
        elif isinstance(device, int):
            idx = device
        else:
            idx = torch.device(device).index or 0
        self.device = torch.device("cuda", idx)
        self.cfg = cfg
        self._lib = lib
        self._h = C.c_void_p()
        N.check(lib.statekv_create(C.byref(cfg._c(self.device.index)), C.byref(self._h)),
                "statekv_create")
        self.torch_dtype = _DTYPES[cfg.dtype][1]
        c = cfg
        self.q_shape = (c.num_streams, c.num_layers, c.num_q_heads, c.frame_tokens, c.head_dim)
        self.kv_shape = (c.num_streams, c.num_layers, c.num_kv_heads, c.frame_tokens, c.head_dim)

    # ------------------------------------------------------------ lifetime
    def close(self) -> None:
        if self._h:
            self._lib.statekv_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # ---------------------------------------------------------------- step
    def _check_in(self, t: torch.Tensor, shape, name: str, device: bool = True):
        if tuple(t.shape) != shape or t.dtype != self.torch_dtype or not t.is_contiguous():
            raise ValueError(f"{name}: want contiguous {self.torch_dtype} {shape}, "
                             f"got {t.dtype} {tuple(t.shape)}")
        if device and t.device != self.device:
            raise ValueError(f"{name} must be on {self.device}")
        if not device and t.device.type != "cpu":
            raise ValueError(f"{name} must be a host tensor")

    def prefill_frame(self, q, k, v, o=None, stream=None) -> torch.Tensor:
        """One frame step (device tensors).  Returns o [S][L][Hq][T][d]."""
        self._check_in(q, self.q_shape, "q")
        self._check_in(k, self.kv_shape, "k")
        self._check_in(v, self.kv_shape, "v")
        if o is None:
            o = torch.empty(self.q_shape, dtype=self.torch_dtype, device=self.device)
        self._check_in(o, self.q_shape, "o")
        N.check(self._lib.statekv_prefill_frame(
            self._h, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            _stream_ptr(stream, self.device)), "statekv_prefill_frame")
        return o

    def prefill_frame_host(self, q, k, v, o, stream=None) -> torch.Tensor:
        """One frame step from host tensors (pinned for async copies)."""
        for t, s, nme in ((q, self.q_shape, "q"), (k, self.kv_shape, "k"),
                          (v, self.kv_shape, "v"), (o, self.q_shape, "o")):
            self._check_in(t, s, nme, device=False)
        N.check(self._lib.statekv_prefill_frame_host(
            self._h, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            _stream_ptr(stream, self.device)), "statekv_prefill_frame_host")
        return o

    def prefill_frames_host(self, q, k, v, o, stream=None) -> torch.Tensor:
        """F consecutive frame steps from frame-major host tensors
        q, o [F][S][L][Hq][T][d], k, v [F][S][L][Hkv][T][d] (pinned), with
        the copies overlapping the device work; ordered on `stream` as one call."""
        frames = q.shape[0] if q.dim() == len(self.q_shape) + 1 else -1
        if frames < 0:
            raise ValueError(f"q: want [F] + {self.q_shape}, got {tuple(q.shape)}")
        for t, s, nme in ((q, self.q_shape, "q"), (k, self.kv_shape, "k"),
                          (v, self.kv_shape, "v"), (o, self.q_shape, "o")):
            self._check_in(t, (frames,) + tuple(s), nme, device=False)
        N.check(self._lib.statekv_prefill_frames_host(
            self._h, frames, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            _stream_ptr(stream, self.device)), "statekv_prefill_frames_host")
        return o

    def decode(self, q, k, v, o=None, stream=None) -> torch.Tensor:
        """Text tokens over the detailed state: q [S][L][Hq][tok][d],
        k, v [S][L][Hkv][tok][d] (device, pre-RoPE).  Returns o like q."""
        tok = q.shape[3] if q.dim() == 5 else -1
        qs = self.q_shape[:3] + (tok, self.q_shape[4])
        ks = self.kv_shape[:3] + (tok, self.kv_shape[4])
        self._check_in(q, qs, "q")
        self._check_in(k, ks, "k")
        self._check_in(v, ks, "v")
        if o is None:
            o = torch.empty(qs, dtype=self.torch_dtype, device=self.device)
        self._check_in(o, qs, "o")
        N.check(self._lib.statekv_decode(
            self._h, tok, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            _stream_ptr(stream, self.device)), "statekv_decode")
        return o

    @property
    def text_tokens(self) -> int:
        return int(self._lib.statekv_text_tokens(self._h))

    # ------------------------------------------------------------- state
    @property
    def frame_index(self) -> int:
        return int(self._lib.statekv_frame_index(self._h))

    def reset(self) -> None:
        N.check(self._lib.statekv_reset(self._h), "statekv_reset")

    def set_frame_index(self, n: int) -> None:
        N.check(self._lib.statekv_set_frame_index(self._h, n), "statekv_set_frame_index")

    def _view(self, ptr: int, shape, dtype: torch.dtype) -> torch.Tensor:
        if dtype == torch.bfloat16:
            return torch.as_tensor(_DevArray(ptr, shape, "<i2"), device=self.device).view(torch.bfloat16)
        typestr = {torch.float32: "<f4", torch.int32: "<i4"}[dtype]
        return torch.as_tensor(_DevArray(ptr, shape, typestr), device=self.device)

    def compressed(self, s: int = 0, layer: int = 0):
        """Borrowed views of C: (k [Hkv][B+T][d], v, pos [Hkv][B+T], count).
        Slots [0, count) are live, in slot order."""
        k, v, p = C.c_void_p(), C.c_void_p(), C.c_void_p()
        cnt, pitch = C.c_int32(), C.c_int32()
        N.check(self._lib.statekv_get_compressed(self._h, s, layer, C.byref(k), C.byref(v),
                                                 C.byref(p), C.byref(cnt), C.byref(pitch)),
                "statekv_get_compressed")
        c = self.cfg
        shape = (c.num_kv_heads, pitch.value, c.head_dim)
        return (self._view(k.value, shape, self.torch_dtype),
                self._view(v.value, shape, self.torch_dtype),
                self._view(p.value, shape[:2], torch.int32), cnt.value)

    def detailed(self, s: int = 0, layer: int = 0):
        """Borrowed views of D: (k [Hkv][N_max*T][d], v, count)."""
        k, v = C.c_void_p(), C.c_void_p()
        cnt, pitch = C.c_int64(), C.c_int64()
        N.check(self._lib.statekv_get_detailed(self._h, s, layer, C.byref(k), C.byref(v),
                                               C.byref(cnt), C.byref(pitch)),
                "statekv_get_detailed")
        c = self.cfg
        shape = (c.num_kv_heads, pitch.value, c.head_dim)
        return (self._view(k.value, shape, self.torch_dtype),
                self._view(v.value, shape, self.torch_dtype), cnt.value)

    def scores(self, s: int = 0, layer: int = 0):
        """Borrowed views of the last step's scores: (s_j [Hkv][pitch] fp32,
        pool positions [Hkv][pitch] int32, m candidates)."""
        sp, pp = C.c_void_p(), C.c_void_p()
        m, pitch = C.c_int32(), C.c_int32()
        N.check(self._lib.statekv_get_scores(self._h, s, layer, C.byref(sp), C.byref(pp),
                                             C.byref(m), C.byref(pitch)), "statekv_get_scores")
        shape = (self.cfg.num_kv_heads, pitch.value)
        return (self._view(sp.value, shape, torch.float32),
                self._view(pp.value, shape, torch.int32), m.value)

    def rotated_query(self) -> torch.Tensor:
        """Borrowed view of the last step's Q' [S][L][Hq][T][d]."""
        p = C.c_void_p()
        N.check(self._lib.statekv_get_rotated_query(self._h, C.byref(p)),
                "statekv_get_rotated_query")
        return self._view(p.value, self.q_shape, self.torch_dtype)

    def set_compressed(self, s: int, layer: int, k, v, pos, stream=None) -> None:
        """Overwrite C of (s, layer): k, v [Hkv][count][d] and pos
        [Hkv][count] int32 device tensors, count = min(B, n*T)."""
        count = int(pos.shape[1])
        c = self.cfg
        if tuple(k.shape) != (c.num_kv_heads, count, c.head_dim) or k.shape != v.shape:
            raise ValueError("k/v must be [Hkv][count][d]")
        k, v = k.contiguous(), v.contiguous()
        pos = pos.to(torch.int32).contiguous()
        N.check(self._lib.statekv_set_compressed(
            self._h, s, layer, k.data_ptr() if count else None,
            v.data_ptr() if count else None, pos.data_ptr() if count else None,
            count, _stream_ptr(stream, self.device)), "statekv_set_compressed")

    def check_device_status(self, stream=None) -> None:
        """Synchronise and raise if a kernel recorded a device-side failure."""
        N.check(self._lib.statekv_check_device_status(self._h, _stream_ptr(stream, self.device)),
                "device status")

    # ---------------------------------------------------------- profiling
    def profile_enable(self, on: bool = True) -> None:
        N.check(self._lib.statekv_profile_enable(self._h, int(on)), "statekv_profile_enable")

    def profile_kernels(self, *names: str) -> None:
        """Bracket only these kernels ("rope", "attention", "select", ...) with
        events while profiling; no names = every kernel."""
        mask = 0
        for name in names:
            if name not in N.KERNEL_NAMES:
                raise ValueError(f"unknown kernel {name!r}: one of {N.KERNEL_NAMES}")
            mask |= 1 << N.KERNEL_NAMES.index(name)
        N.check(self._lib.statekv_profile_kernels(self._h, mask if names else 0xffffffff),
                "statekv_profile_kernels")

    def profile_mask(self, mask: int) -> None:
        """Bracket exactly the kernels whose bit (1 << STATEKV_KERNEL_*) is set
        in mask while profiling; 0 brackets none (launches keep their
        overlap) without resetting the accumulated times."""
        N.check(self._lib.statekv_profile_kernels(self._h, int(mask) & 0xffffffff),
                "statekv_profile_kernels")

    def profile_read(self) -> dict:
        """{kernel name: (total device ms, launches)} since profiling started."""
        out = {}
        for kid, name in enumerate(N.KERNEL_NAMES):
            ms, n = C.c_double(), C.c_int64()
            N.check(self._lib.statekv_profile_read(self._h, kid, C.byref(ms), C.byref(n)),
                    "statekv_profile_read")
            out[name] = (ms.value, n.value)
        return out
