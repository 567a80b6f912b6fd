"""Seeded per-frame Q/K/V for StateKV workloads.

Every (stream, layer, frame) draws from its own counter-keyed
``numpy.random.SeedSequence`` so that any frame can be regenerated alone.

Recipe (the same on both sides of every parity test):
  * Q, K, V ~ N(0, 1) i.i.d.
  * optional per-channel key scale exp(sigma * z_c), z_c ~ N(0, 1), fixed per
    (stream, layer, KV head)  -- heavy-tailed key channels;
  * ``sinks_per_frame`` key rows per (KV head, frame), chosen without
    replacement, get ``sink_gain * u`` added, u a unit vector per
    (stream, layer, KV head).  With ``sink_drift > 0`` the direction drifts:
    u_n = normalize(u_{n-1} + drift * N(0, I));
  * finally every value is rounded to the storage dtype (bf16 round-to-nearest
    -even through torch's CPU cast, or kept as float32).

No step of the StateKV method is computed here.
"""

from __future__ import annotations

import numpy as np
import torch

from .shapes import WorkloadShape

_TAG_FRAME = 1
_TAG_U0 = 2
_TAG_DRIFT = 3
_TAG_KSCALE = 4


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _unit(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x)


class FrameSource:
    """Generates the inputs of frame n for every (stream, layer)."""

    def __init__(self, shape: WorkloadShape, seed: int | None = None):
        self.shape = shape
        self.seed = shape.seed if seed is None else seed
        self._u_cache: dict[tuple[int, int, int], list[np.ndarray]] = {}

    # ----------------------------------------------------------------- helpers
    def _sink_dir(self, s: int, l: int, h: int, n: int) -> np.ndarray:
        key = (s, l, h)
        chain = self._u_cache.get(key)
        d = self.shape.head_dim
        if chain is None:
            chain = [_unit(_rng(self.seed, _TAG_U0, s, l, h).standard_normal(d))]
            self._u_cache[key] = chain
        if self.shape.sink_drift == 0.0:
            return chain[0]
        while len(chain) <= n:
            m = len(chain)
            step = _rng(self.seed, _TAG_DRIFT, s, l, h, m).standard_normal(d)
            chain.append(_unit(chain[-1] + self.shape.sink_drift * step))
        return chain[n]

    def _key_scale(self, s: int, l: int) -> np.ndarray | None:
        sig = self.shape.key_scale_sigma
        if sig == 0.0:
            return None
        z = _rng(self.seed, _TAG_KSCALE, s, l).standard_normal(
            (self.shape.kv_heads, self.shape.head_dim))
        return np.exp(sig * z)

    def _to_storage(self, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        if self.shape.dtype == "bf16":
            t = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32)
            return t.numpy()
        return x

    # -------------------------------------------------------------------- API
    def layer_frame(self, s: int, l: int, n: int):
        """(q [Hq][T][d], k [Hkv][T][d], v [Hkv][T][d]) as float32 arrays whose
        values are exactly representable in the storage dtype."""
        sh = self.shape
        T, d = sh.frame_tokens, sh.head_dim
        rng = _rng(self.seed, _TAG_FRAME, s, l, n)
        q = rng.standard_normal((sh.q_heads, T, d), dtype=np.float32)
        k = rng.standard_normal((sh.kv_heads, T, d), dtype=np.float32)
        v = rng.standard_normal((sh.kv_heads, T, d), dtype=np.float32)
        scale = self._key_scale(s, l)
        if scale is not None:
            k = (k * scale[:, None, :]).astype(np.float32)
        if sh.sinks_per_frame > 0:
            for h in range(sh.kv_heads):
                rows = rng.choice(T, size=min(sh.sinks_per_frame, T), replace=False)
                u = self._sink_dir(s, l, h, n)
                k[h, rows, :] += (sh.sink_gain * u).astype(np.float32)
        return self._to_storage(q), self._to_storage(k), self._to_storage(v)

    def frame(self, n: int):
        """All streams and layers of frame n:
        q [S][L][Hq][T][d], k, v [S][L][Hkv][T][d] (float32 arrays)."""
        sh = self.shape
        T, d = sh.frame_tokens, sh.head_dim
        q = np.empty((sh.streams, sh.layers, sh.q_heads, T, d), np.float32)
        k = np.empty((sh.streams, sh.layers, sh.kv_heads, T, d), np.float32)
        v = np.empty_like(k)
        for s in range(sh.streams):
            for l in range(sh.layers):
                q[s, l], k[s, l], v[s, l] = self.layer_frame(s, l, n)
        return q, k, v

    def frame_tensors(self, n: int, device: str | torch.device = "cpu"):
        """Frame n as torch tensors in the storage dtype."""
        dt = torch.bfloat16 if self.shape.dtype == "bf16" else torch.float32
        return tuple(torch.from_numpy(a).to(dt).to(device) for a in self.frame(n))
