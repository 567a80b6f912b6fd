"""Workload shapes for StateKV streaming prefill.

The method ("Linear Scaling Video VLMs for Long Video Understanding",
section "实验关键数据 / 主实验") is evaluated at 1 FPS with up to 512 frames and a
compressed budget B = 4096 on InternVL3 / Qwen3-VL models.  The shapes below
mirror the attention geometry of those models (query heads, KV heads, head
dim, visual tokens per frame) with synthetic data in place of the benchmark
videos, which are not available here.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace


@dataclass(frozen=True)
class WorkloadShape:
    name: str
    streams: int
    layers: int
    q_heads: int
    kv_heads: int
    head_dim: int
    frame_tokens: int          # T
    budget: int                # B
    frames: int                # N (also the detailed-cache capacity)
    rope_theta: float
    rope_alpha: float          # static global RoPE scale, fixed for the run
    rope_orig_ctx: int         # YaRN original context (ignored when alpha == 1)
    dtype: str                 # "bf16" | "f32"
    sinks_per_frame: int       # temporal-sink key rows planted per frame
    sink_gain: float           # magnitude added along the sink direction
    sink_drift: float          # 0 = fixed direction; else u_n = normalize(u_{n-1} + drift*N(0,I))
    key_scale_sigma: float     # 0 = none; else per-channel log-normal key scale
    seed: int = 20260

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def units(self) -> int:
        """Independent (stream, layer, KV head) selection units."""
        return self.streams * self.layers * self.kv_heads

    def with_(self, **kw) -> "WorkloadShape":
        return replace(self, **kw)

    def visible_pairs_steady(self) -> int:
        """Visible (query, key) pairs per query head once the state is full."""
        t = self.frame_tokens
        return t * self.budget + t * (t + 1) // 2

    def visible_pairs(self, n: int) -> int:
        """Visible (query, key) pairs per query head at frame n (0-based)."""
        t = self.frame_tokens
        c = min(self.budget, n * t)
        return t * c + t * (t + 1) // 2

    def attention_flops(self, n: int) -> float:
        """Algorithmic MMA flops of one frame step over all heads and layers:
        2*d per visible pair for QK^T and 2*d for PV."""
        return 4.0 * self.head_dim * self.visible_pairs(n) * self.q_heads \
            * self.layers * self.streams


def _yarn_orig_ctx(frames: int, frame_tokens: int, alpha: float,
                   prompt: int = 256, decode: int = 512) -> int:
    """L_orig for a static YaRN scale alpha chosen up front for the whole run
    (video tokens + prompt + decode budget), rounded up."""
    total = frames * frame_tokens + prompt + decode
    return int(math.ceil(total / alpha))


SHAPES: dict[str, WorkloadShape] = {
    # oracle-scale case: fp32 storage, fixed sink direction
    "tiny_f32": WorkloadShape(
        name="tiny_f32", streams=1, layers=1, q_heads=2, kv_heads=1,
        head_dim=64, frame_tokens=16, budget=32, frames=8,
        rope_theta=1e4, rope_alpha=1.0, rope_orig_ctx=0, dtype="f32",
        sinks_per_frame=2, sink_gain=3.0, sink_drift=0.0,
        key_scale_sigma=0.0),
    # InternVL3-1B attention geometry, one layer
    "internvl3_1b_layer": WorkloadShape(
        name="internvl3_1b_layer", streams=1, layers=1, q_heads=14,
        kv_heads=2, head_dim=64, frame_tokens=256, budget=4096, frames=64,
        rope_theta=1e6, rope_alpha=1.0, rope_orig_ctx=0, dtype="bf16",
        sinks_per_frame=4, sink_gain=3.0, sink_drift=0.05,
        key_scale_sigma=0.0),
    # InternVL3-2B attention geometry, full 28-layer stack, 512 frames
    "internvl3_2b_stack": WorkloadShape(
        name="internvl3_2b_stack", streams=1, layers=28, q_heads=12,
        kv_heads=2, head_dim=128, frame_tokens=256, budget=4096, frames=512,
        rope_theta=1e6, rope_alpha=4.0,
        rope_orig_ctx=_yarn_orig_ctx(512, 256, 4.0), dtype="bf16",
        sinks_per_frame=4, sink_gain=3.0, sink_drift=0.05,
        key_scale_sigma=0.0),
    # Qwen3-VL-2B attention geometry, heavy-tailed key channels
    "qwen3vl_2b_stack": WorkloadShape(
        name="qwen3vl_2b_stack", streams=1, layers=28, q_heads=16,
        kv_heads=8, head_dim=128, frame_tokens=256, budget=4096, frames=512,
        rope_theta=5e6, rope_alpha=4.0,
        rope_orig_ctx=_yarn_orig_ctx(512, 256, 4.0), dtype="bf16",
        sinks_per_frame=4, sink_gain=3.0, sink_drift=0.05,
        key_scale_sigma=0.5),
}


def serving_shape(frame_tokens: int, budget: int, frames: int = 2048,
                  streams: int = 16, layers: int = 4) -> WorkloadShape:
    """Batched serving sweep: independent video streams stepped together."""
    return WorkloadShape(
        name=f"serving_T{frame_tokens}_B{budget}", streams=streams,
        layers=layers, q_heads=16, kv_heads=8, head_dim=128,
        frame_tokens=frame_tokens, budget=budget, frames=frames,
        rope_theta=5e6, rope_alpha=4.0,
        rope_orig_ctx=_yarn_orig_ctx(frames, frame_tokens, 4.0),
        dtype="bf16", sinks_per_frame=4, sink_gain=3.0, sink_drift=0.05,
        key_scale_sigma=0.5)


for _t in (64, 256):
    for _b in (1024, 4096):
        _s = serving_shape(_t, _b)
        SHAPES[_s.name] = _s
