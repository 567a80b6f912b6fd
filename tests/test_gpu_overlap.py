"""End-to-end selection overlap on the full-size stacks.

The GPU path and the CPU oracle each run free on their own state for a whole
stretch of frames (no teacher forcing), and after every frame the kept index
sets of a unit -- one (layer, KV head) -- are compared:
overlap = |S_gpu ∩ S_oracle| / B (StateKV, 关键设计 2: the Top-B state update
C_n = TopK(s, B) over the pool of C_{n-1} and the frame).  Rounding
differences can swap near-tied candidates at the cut; a swap changes the
next pool, so the two runs may drift apart over frames; the overlap measures
how far.  The oracle's units run in parallel in spawned worker processes
(the oracle itself is unchanged); each worker regenerates its own inputs
from the seeded source.  With STATEKV_OVERLAP_OUT set, the per-layer and
per-frame table is written there as JSON; STATEKV_OVERLAP_FRAMES runs a
longer stretch than the default 40 frames.
"""

from __future__ import annotations

import json
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

from synth import SHAPES, FrameSource

pytestmark = pytest.mark.gpu

OVERLAP_REPORT: list = []


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kv_cache_compression_frame_gb300 import build_lib
    build_lib.build()


def _oracle_unit_stream(args):
    """Runs the oracle on one (layer, KV head) for frames 0..frames-1 and
    returns the kept positions after each frame (ascending)."""
    name, layer, hk, frames = args
    import oracle.statekv_oracle as orc
    sh = SHAPES[name]
    src = FrameSource(sh)
    omega, ms = orc.rope_frequencies(sh.head_dim, sh.rope_theta, sh.rope_alpha, sh.rope_orig_ctx)
    scale = orc.logit_scale(sh.head_dim, ms)
    st = orc.UnitState(sh.head_dim)
    G = sh.group
    kept = []
    for n in range(frames):
        q, k, v = src.layer_frame(0, layer, n)
        orc.prefill_unit_frame(st, q[hk * G:(hk + 1) * G], k[hk], v[hk], n, budget=sh.budget,
                               omega=omega, scale=scale, dtype=sh.dtype)
        kept.append(st.comp_pos.astype(np.int64).copy())
    return kept


@pytest.mark.parametrize("name,layers,frames", [
    ("internvl3_2b_stack", (0, 9, 18, 27), 40),
    ("qwen3vl_2b_stack", (0, 27), 40),
])
def test_free_running_selection_overlap_per_layer(name, layers, frames):
    from kv_cache_compression_frame_gb300 import StateKV, StateKVConfig
    sh = SHAPES[name]
    # a longer stretch for a study (the default keeps the test to a minute or two)
    frames = min(sh.frames, int(os.environ.get("STATEKV_OVERLAP_FRAMES", frames)))
    units = [(l, hk) for l in layers for hk in range(sh.kv_heads)]
    # the pool starts before the first CUDA call of this process's workers
    ctx = mp.get_context("spawn")
    pool = ctx.Pool(processes=min(len(units), max(1, (os.cpu_count() or 2) - 1)))
    try:
        pending = pool.map_async(_oracle_unit_stream, [(name, l, hk, frames) for l, hk in units])
        src = FrameSource(sh)
        h = StateKV(StateKVConfig.from_shape(sh))
        dev = h.device
        gpu = {u: [] for u in units}
        for n in range(frames):
            q, k, v = (torch.from_numpy(a).to(torch.bfloat16).to(dev) for a in src.frame(n))
            h.prefill_frame(q, k, v)
            h.check_device_status()
            for l in layers:
                _, _, p, c = h.compressed(0, l)
                pc = p[:, :c].cpu().numpy().astype(np.int64)
                for hk in range(sh.kv_heads):
                    gpu[(l, hk)].append(np.sort(pc[hk]))
        h.close()
        ref = dict(zip(units, pending.get(timeout=3600)))
    finally:
        pool.close()
        pool.join()
    first_evict = next(n for n in range(frames) if (n + 1) * sh.frame_tokens > sh.budget)
    per_unit = {}
    for u in units:
        ov = []
        for n in range(frames):
            a, b = gpu[u][n], ref[u][n]
            assert len(a) == len(b) == min(sh.budget, (n + 1) * sh.frame_tokens)
            if n < first_evict:
                np.testing.assert_array_equal(a, b)      # nothing selected yet
                continue
            ov.append(len(np.intersect1d(a, b, assume_unique=True)) / sh.budget)
        per_unit[u] = ov
    per_layer = {l: np.array([per_unit[(l, hk)] for hk in range(sh.kv_heads)]) for l in layers}
    per_frame = np.array([per_unit[u] for u in units]).mean(axis=0)
    row = {"workload": name, "frames": frames, "budget": sh.budget,
           "first_eviction_frame": first_evict,
           "per_layer": {str(l): {"min": float(x.min()), "mean": float(x.mean()),
                                  "last_frame_mean": float(x[:, -1].mean())}
                         for l, x in per_layer.items()},
           "per_frame_mean": [float(x) for x in per_frame],
           "per_unit_last": {f"{l}/{hk}": float(per_unit[(l, hk)][-1]) for l, hk in units}}
    OVERLAP_REPORT.append(row)
    out = os.environ.get("STATEKV_OVERLAP_OUT")
    if out:
        with open(out, "w") as f:
            json.dump(OVERLAP_REPORT, f, indent=1)
    for l, x in per_layer.items():
        assert x.mean() > 0.9, f"layer {l}: mean overlap {x.mean():.4f}"
