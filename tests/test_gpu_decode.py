"""GPU parity of text decode over the detailed state D against the CPU
oracle, through the C ABI (Python binding).

Each checked call compares the RoPE of the new text keys appended to D (ulp
bound) and their values (bit-exact), and O (row-relative error) against the
oracle's attention over the GPU's own D rows and rotated text queries
(teacher forcing, so the tolerance is not spent on earlier roundings).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.statekv_oracle as orc
from synth import SHAPES, FrameSource, WorkloadShape
from parity import O_TOL, check_rope, f64, raw_equal, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kv_cache_compression_frame_gb300 import build_lib
    build_lib.build()


def _shape(name, **kw) -> WorkloadShape:
    base = dict(name=name, streams=1, layers=2, q_heads=4, kv_heads=2,
                head_dim=128, frame_tokens=64, budget=96, frames=4,
                rope_theta=1e4, rope_alpha=1.0, rope_orig_ctx=0, dtype="bf16",
                sinks_per_frame=2, sink_gain=3.0, sink_drift=0.05,
                key_scale_sigma=0.0)
    base.update(kw)
    return WorkloadShape(**base)


class Decoder:
    """A handle that has prefilled frames, decoding text and checking calls."""

    def __init__(self, sh: WorkloadShape, frames: int, ring: int = 0, offset: int = 0,
                 max_frames: int = 0):
        from kv_cache_compression_frame_gb300 import StateKV, StateKVConfig
        self.sh = sh
        self.src = FrameSource(sh)
        self.offset = offset
        self.h = StateKV(StateKVConfig.from_shape(sh, position_offset=offset,
                                                  max_frames=max_frames or sh.frames))
        self.dev, self.tdt = self.h.device, self.h.torch_dtype
        n_src = ring or frames
        dev_frames = [tuple(torch.from_numpy(a).to(self.tdt).to(self.dev) for a in self.src.frame(i))
                      for i in range(n_src)]
        for n in range(frames):
            self.h.prefill_frame(*dev_frames[n % n_src])
        torch.cuda.synchronize()
        self.omega, ms = orc.rope_frequencies(sh.head_dim, sh.rope_theta, sh.rope_alpha,
                                              sh.rope_orig_ctx)
        self.scale = orc.logit_scale(sh.head_dim, ms)
        self.rng = np.random.default_rng(1234)

    def text(self, tok):
        sh = self.sh
        q = self.rng.standard_normal((sh.streams, sh.layers, sh.q_heads, tok, sh.head_dim))
        k = self.rng.standard_normal((sh.streams, sh.layers, sh.kv_heads, tok, sh.head_dim))
        v = self.rng.standard_normal((sh.streams, sh.layers, sh.kv_heads, tok, sh.head_dim))
        return [torch.from_numpy(a).to(self.tdt).to(self.dev) for a in (q, k, v)]

    def step(self, tok, units=None):
        sh, h = self.sh, self.h
        G = sh.q_heads // sh.kv_heads
        first = h.frame_index * sh.frame_tokens + h.text_tokens
        q, k, v = self.text(tok)
        o = h.decode(q, k, v)
        h.check_device_status()
        assert h.text_tokens == first - h.frame_index * sh.frame_tokens + tok
        pos = self.offset + first + np.arange(tok, dtype=np.int64)
        R = G * tok
        U = sh.streams * sh.layers * sh.kv_heads
        qrot = h.rotated_query().reshape(-1)[:U * R * sh.head_dim].view(
            sh.streams, sh.layers, sh.q_heads, tok, sh.head_dim).clone().cpu()
        q_ref = orc.round_to_storage(orc.rope_rotate(q.double().cpu().numpy(), pos, self.omega),
                                     sh.dtype)
        check_rope(qrot, q_ref, q.double().cpu().numpy(), sh.dtype, f"text Q' at {first}")
        o_cpu = o.cpu()
        worst = 0.0
        if units is None:
            units = [(s, l, hk) for s in range(sh.streams) for l in range(sh.layers)
                     for hk in range(sh.kv_heads)]
        for (s, l, hk) in units:
            what = f"decode at row {first} unit ({s},{l},{hk})"
            dk, dv, cnt = h.detailed(s, l)
            assert cnt == first + tok
            krot = dk[hk, first:first + tok].clone().cpu()
            kn = k[s, l, hk].double().cpu().numpy()
            check_rope(krot, orc.round_to_storage(orc.rope_rotate(kn, pos, self.omega), sh.dtype),
                       kn, sh.dtype, f"text K' {what}")
            assert raw_equal(dv[hk, first:first + tok].cpu(), v[s, l, hk].cpu()), f"D V {what}"
            pool_k = f64(dk[hk, :first + tok].cpu())
            pool_v = f64(dv[hk, :first + tok].cpu())
            O_ref, _ = orc.attend_frame(f64(qrot[s, l, hk * G:(hk + 1) * G]), pool_k, pool_v,
                                        first, self.scale)
            e = row_rel_err(f64(o_cpu[s, l, hk * G:(hk + 1) * G]), O_ref)
            assert e <= O_TOL[sh.dtype], f"O {what}: row-relative error {e:.3g}"
            worst = max(worst, e)
        return worst


@pytest.mark.parametrize("q_heads,toks", [(4, (1, 3, 2, 8)),      # G = 2: N = 16
                                          (16, (1, 3, 8))])        # G = 8: N = 16, 32, 64
def test_decode_after_frames(q_heads, toks):
    d = Decoder(_shape("dec", q_heads=q_heads), frames=3)
    for tok in toks:
        d.step(tok)


def test_decode_before_any_frame_and_yarn_offset():
    """Text only (empty D before the first call), YaRN scaling, an offset."""
    sh = _shape("dec0", rope_alpha=4.0, rope_orig_ctx=64, rope_theta=1e6, frames=2)
    d = Decoder(sh, frames=0, offset=1000)
    d.step(5)
    d.step(1)


def test_decode_spans_several_key_chunks():
    """D longer than one 2048-key work item, ragged last chunk and tile."""
    sh = _shape("declong", layers=1, frame_tokens=256, budget=256, frames=12)
    d = Decoder(sh, frames=11, ring=4)
    d.step(3)
    d.step(16)


def test_decode_rules():
    from kv_cache_compression_frame_gb300 import StateKVError
    sh = _shape("decrules", frames=2)
    d = Decoder(sh, frames=2)                       # D full of frames: room for 0 rows
    q, k, v = d.text(1)
    with pytest.raises(StateKVError) as ei:
        d.h.decode(q, k, v)
    assert ei.value.status == -3 and d.h.text_tokens == 0
    d2 = Decoder(sh, frames=1)
    d2.step(2)
    fq, fk, fv = (torch.from_numpy(a).to(d2.tdt).to(d2.dev) for a in d2.src.frame(1))
    with pytest.raises(StateKVError) as ei:         # no frames once text was decoded
        d2.h.prefill_frame(fq, fk, fv)
    assert ei.value.status == -1
    q, k, v = d2.text(17)                           # more than 16 tokens per call
    with pytest.raises(StateKVError):
        d2.h.decode(q, k, v)
    d2.h.reset()
    assert d2.h.text_tokens == 0
    d2.h.prefill_frame(fq, fk, fv)


def test_decode_full_size_internvl3_2b_sampled():
    """The 2B stack after 512 frames (D = 131,072 rows per KV head, 64 key
    chunks per unit, 56 units): one text token, sampled units.  D holds one
    frame's worth of rows more than the video, for the text."""
    sh = SHAPES["internvl3_2b_stack"]
    d = Decoder(sh, frames=sh.frames, ring=4, max_frames=sh.frames + 1)
    d.step(1, units=[(0, 0, 0), (0, 13, 1), (0, 27, 1)])
    d.step(2, units=[(0, 5, 0), (0, 27, 0)])
