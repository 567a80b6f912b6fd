"""GPU parity of the CUDA path against the CPU oracle, one frame step at a
time, through the C ABI (Python binding).

Every checked step compares: RoPE of Q and K (ulp), the D append (bit-exact
K' copy and V copy), O (row-relative error), the scores s_j, the Top-B
selection (up to near-ties) and the slot-reuse gather into C (bit-exact).
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle.statekv_oracle as orc
from synth import SHAPES, FrameSource, WorkloadShape
from parity import (O_TOL, check_rope, check_scores, check_selection, f64,
                    raw_equal, record_step, row_rel_err)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kv_cache_compression_frame_gb300 import build_lib
    build_lib.build()


def _small(name, **kw) -> WorkloadShape:
    base = dict(name=name, streams=1, layers=1, q_heads=2, kv_heads=1,
                head_dim=64, frame_tokens=16, budget=32, frames=8,
                rope_theta=1e4, rope_alpha=1.0, rope_orig_ctx=0, dtype="bf16",
                sinks_per_frame=2, sink_gain=3.0, sink_drift=0.05,
                key_scale_sigma=0.0)
    base.update(kw)
    return WorkloadShape(**base)


class Stepper:
    """Runs the CUDA path frame by frame and checks steps against the oracle."""

    def __init__(self, shape: WorkloadShape, position_offset: int = 0, policy: str = "topb"):
        from kv_cache_compression_frame_gb300 import StateKV, StateKVConfig
        self.sh = shape
        self.src = FrameSource(shape)
        self.offset = position_offset
        self.policy = policy
        self.h = StateKV(StateKVConfig.from_shape(shape, position_offset=position_offset,
                                                  select_policy=policy))
        self.dev = self.h.device
        self.tdt = self.h.torch_dtype
        self.omega, ms = orc.rope_frequencies(shape.head_dim, shape.rope_theta,
                                              shape.rope_alpha, shape.rope_orig_ctx)
        self.scale = orc.logit_scale(shape.head_dim, ms)
        self.stats = []

    def tensors(self, n):
        q, k, v = self.src.frame(n)
        t = [torch.from_numpy(a).to(self.tdt).to(self.dev) for a in (q, k, v)]
        return (q, k, v), t

    def run(self, n):
        _, (q, k, v) = self.tensors(n)
        o = self.h.prefill_frame(q, k, v)
        self.h.check_device_status()
        return o

    def advance(self, n_to, ring=4):
        """Run frames up to (not including) n_to quickly: frame n takes the
        inputs of frame n % ring (generated once).  The frames checked later
        with step() come from the source itself; the checks are
        teacher-forced on the GPU's state, so only the shape of the history
        matters here, not its values."""
        if not hasattr(self, "_ring"):
            self._ring = [self.tensors(i)[1] for i in range(max(1, min(ring, n_to)))]
        n = self.h.frame_index
        while n < n_to:
            q, k, v = self._ring[n % len(self._ring)]
            self.h.prefill_frame(q, k, v)
            n += 1
        self.h.check_device_status()

    def step(self, n, units=None):
        sh, h = self.sh, self.h
        assert h.frame_index == n
        T, G, B = sh.frame_tokens, sh.group, sh.budget
        (qn, kn, vn), (q, k, v) = self.tensors(n)
        if units is None:
            units = [(s, l, hk) for s in range(sh.streams) for l in range(sh.layers)
                     for hk in range(sh.kv_heads)]
        pre = {}
        for (s, l) in {(s, l) for s, l, _ in units}:
            ck, cv, cp, cnt = h.compressed(s, l)
            pre[(s, l)] = (ck[:, :cnt].clone().cpu(), cv[:, :cnt].clone().cpu(),
                           cp[:, :cnt].clone().cpu().numpy(), cnt)
        o = h.prefill_frame(q, k, v)
        h.check_device_status()
        pos = self.offset + n * T + np.arange(T, dtype=np.int64)
        # RoPE of every query row
        q_ref = orc.round_to_storage(orc.rope_rotate(qn, pos, self.omega), sh.dtype)
        qrot = h.rotated_query().clone().cpu()
        rq = check_rope(qrot, q_ref, qn, sh.dtype, f"Q' frame {n}")
        o_cpu = o.cpu()
        worst = dict(o=0.0, s=0.0, swaps=0, rope_q=rq)
        for (s, l, hk) in units:
            what = f"frame {n} unit ({s},{l},{hk})"
            dk, dv, dcnt = h.detailed(s, l)
            assert dcnt == (n + 1) * T
            krot = dk[hk, n * T:(n + 1) * T].clone().cpu()
            check_rope(krot, orc.round_to_storage(orc.rope_rotate(kn[s, l, hk], pos, self.omega),
                                                  sh.dtype), kn[s, l, hk], sh.dtype, f"K' {what}")
            assert raw_equal(dv[hk, n * T:(n + 1) * T].cpu(), v[s, l, hk].cpu()), f"D V {what}"
            ck, cv, cp, cnt = pre[(s, l)]
            pool_k_raw = torch.cat([ck[hk], krot])
            pool_v_raw = torch.cat([cv[hk], v[s, l, hk].cpu()])
            pool_pos = np.concatenate([cp[hk].astype(np.int64), pos])
            qr = f64(qrot[s, l, hk * G:(hk + 1) * G])
            O_ref, P = orc.attend_frame(qr, f64(pool_k_raw), f64(pool_v_raw), cnt, self.scale)
            s_ref = orc.importance_scores(P)
            e = row_rel_err(f64(o_cpu[s, l, hk * G:(hk + 1) * G]), O_ref)
            assert e <= O_TOL[sh.dtype], f"O {what}: row-relative error {e:.3g}"
            worst["o"] = max(worst["o"], e)
            sc, sp, m = h.scores(s, l)
            assert m == cnt + T
            np.testing.assert_array_equal(sp[hk, :m].cpu().numpy(), pool_pos)
            worst["s"] = max(worst["s"], check_scores(f64(sc[hk, :m]), s_ref, f"s {what}"))
            nk, nv, npos, ncnt = h.compressed(s, l)
            assert ncnt == min(B, cnt + T)
            kept = npos[hk, :ncnt].cpu().numpy().astype(np.int64)
            if self.policy == "window":          # the B most recent, exactly
                np.testing.assert_array_equal(np.sort(kept), np.sort(pool_pos)[-ncnt:])
            else:
                worst["swaps"] += check_selection(kept, s_ref, pool_pos, B, f"select {what}")
            # slot-reuse gather: every live slot is a bit copy of its pool row
            where = {int(p): i for i, p in enumerate(pool_pos)}
            idx = torch.tensor([where[int(p)] for p in kept], dtype=torch.long)
            assert raw_equal(nk[hk, :ncnt].cpu(), pool_k_raw[idx]), f"C K gather {what}"
            assert raw_equal(nv[hk, :ncnt].cpu(), pool_v_raw[idx]), f"C V gather {what}"
        self.stats.append((n, worst))
        record_step(self.sh.name, n, len(units), worst)
        return worst


# ------------------------------------------------------------------- tests
def test_tiny_f32_every_frame():
    st = Stepper(SHAPES["tiny_f32"])
    for n in range(SHAPES["tiny_f32"].frames):
        st.step(n)


def test_ragged_bf16_partial_fill():
    # G*T = 144 rows: two query tiles, the second ragged and spanning heads;
    # B = 100 is not a multiple of T, so frame 2 evicts while C is filling
    sh = _small("ragged", layers=2, q_heads=6, kv_heads=2, head_dim=64,
                frame_tokens=48, budget=100, frames=6)
    st = Stepper(sh)
    for n in range(sh.frames):
        st.step(n)


def test_d128_streams_layers_offset_yarn():
    sh = _small("multi", streams=2, layers=2, q_heads=4, kv_heads=2, head_dim=128,
                frame_tokens=64, budget=192, frames=6, rope_theta=1e6,
                rope_alpha=4.0, rope_orig_ctx=200, key_scale_sigma=0.5)
    st = Stepper(sh, position_offset=1000)
    for n in range(sh.frames):
        st.step(n)


def test_zero_budget_is_per_frame_attention():
    sh = _small("b0", q_heads=4, kv_heads=2, head_dim=64, frame_tokens=80, budget=0, frames=3)
    st = Stepper(sh)
    for n in range(3):
        st.step(n)
        _, _, _, cnt = st.h.compressed(0, 0)
        assert cnt == 0


def test_internvl3_1b_layer_through_fill_to_steady_state():
    sh = SHAPES["internvl3_1b_layer"]
    st = Stepper(sh)
    for n in range(18):
        if n in (0, 1, 15, 16, 17):
            st.step(n)
        else:
            st.run(n)


@pytest.mark.parametrize("name,layers", [("internvl3_2b_stack", (0, 13, 25, 27)),
                                         ("qwen3vl_2b_stack", (0, 27))])
def test_full_size_steady_state_sampled(name, layers):
    """The workload bench.py times, at full size: all layers run; the step at
    frame 16 (state full, c = B) is checked on sampled layers.  On a 152-SM
    GPU the 2B stack's last 64 query tiles (layers 25-27) are key-split CTA
    pairs: layer 27 entirely, layer 25 mixes whole and split tiles."""
    sh = SHAPES[name]
    st = Stepper(sh)
    for n in range(16):
        st.run(n)
    units = [(0, l, hk) for l in layers for hk in range(sh.kv_heads)]
    st.step(16, units=units)


@pytest.mark.parametrize("name,layers", [("internvl3_2b_stack", (0, 27)),
                                         ("qwen3vl_2b_stack", (0, 27))])
def test_full_size_last_frame_sampled(name, layers):
    """The last frame of a 512-frame video (n = 511): positions reach
    130,816..131,071 (the fp64 angle reduction and the alpha = 4 YaRN
    frequencies carry all of RoPE's accuracy there) and the step appends
    the last rows the detailed state can hold (n = max_frames - 1)."""
    sh = SHAPES[name]
    st = Stepper(sh)
    st.advance(sh.frames - 1)
    units = [(0, l, hk) for l in layers for hk in range(sh.kv_heads)]
    st.step(sh.frames - 1, units=units)
    _, _, dcnt = st.h.detailed(0, layers[-1])
    assert dcnt == sh.frames * sh.frame_tokens


def test_internvl3_2b_budget_16384_steady_state():
    """The largest budget of the page's budget ablation (B = 16384): a pool of
    16,640 candidates per unit (a wider radix cut and key buffer in the
    selection, 130 key tiles per query tile), checked on the first two
    frames with a full state."""
    sh = SHAPES["internvl3_2b_stack"].with_(name="internvl3_2b_B16384", budget=16384, frames=80)
    st = Stepper(sh)
    n_full = sh.budget // sh.frame_tokens
    st.advance(n_full)
    units = [(0, l, hk) for l in (0, 27) for hk in range(sh.kv_heads)]
    for n in (n_full, n_full + 1):
        st.step(n, units=units)


@pytest.mark.parametrize("cluster", ["", "1"])
def test_largest_selectable_pool(cluster, monkeypatch):
    """The largest pool the selection takes: B + T = 24,576 candidates per
    unit (its key buffer fills the shared memory a CTA may hold), on the 2B
    layer geometry (two layers), checked on the first two frames with a full
    state; once with the selection spread over a cluster (the default for
    so few units) and once with one CTA per unit."""
    if cluster:
        monkeypatch.setenv("STATEKV_SELECT_CLUSTER", cluster)
    sh = SHAPES["internvl3_2b_stack"].with_(name="internvl3_2b_maxpool", layers=2,
                                            budget=24576 - 256, frames=97)
    st = Stepper(sh)
    n_full = sh.budget // sh.frame_tokens
    st.advance(n_full)
    for n in (n_full, n_full + 1):
        st.step(n)


@pytest.mark.parametrize("name,n", [("serving_T64_B1024", 17), ("serving_T64_B4096", 65),
                                    ("serving_T256_B1024", 5), ("serving_T256_B4096", 17)])
def test_serving_shape_steady_state_sampled(name, n):
    """The batched-serving configuration: 16 independent streams x 4 layers x
    8 KV heads stepped together (512 units; at T = 64 one 128-row query tile
    per unit), checked after the state filled, on sampled streams."""
    sh = SHAPES[name]
    st = Stepper(sh)
    st.advance(n)
    units = [(s, l, hk) for s in (0, 7, 15) for l in (0, 3) for hk in range(sh.kv_heads)]
    st.step(n, units=units)


def test_teacher_forced_from_oracle_state():
    """C_{n-1} taken from the oracle's own free-running state."""
    sh = SHAPES["internvl3_1b_layer"].with_(frames=20)
    src = FrameSource(sh)
    ref = orc.StateKVOracle(sh)
    for n in range(17):
        ref.prefill_frame(*src.frame(n))
    st = Stepper(sh)
    st.h.set_frame_index(17)
    u = [ref.units[(0, 0, hk)] for hk in range(sh.kv_heads)]
    dt = st.tdt
    k = torch.from_numpy(np.stack([x.comp_k for x in u])).to(dt).cuda()
    v = torch.from_numpy(np.stack([x.comp_v for x in u])).to(dt).cuda()
    p = torch.from_numpy(np.stack([x.comp_pos for x in u]).astype(np.int32)).cuda()
    st.h.set_compressed(0, 0, k, v, p)
    torch.cuda.synchronize()
    st.step(17)


def test_free_running_selection_overlap():
    """End to end: the GPU and the oracle each run on their own state; the
    per-frame overlap of the kept position sets is reported."""
    sh = SHAPES["internvl3_1b_layer"].with_(frames=40)
    src = FrameSource(sh)
    ref = orc.StateKVOracle(sh)
    st = Stepper(sh)
    overlaps = []
    for n in range(sh.frames):
        q, k, v = src.frame(n)
        ref.prefill_frame(q, k, v)
        st.run(n)
        if (n + 1) * sh.frame_tokens > sh.budget:
            for hk in range(sh.kv_heads):
                _, _, p, c = st.h.compressed(0, 0)
                got = set(p[hk, :c].cpu().numpy().tolist())
                want = set(ref.units[(0, 0, hk)].comp_pos.tolist())
                overlaps.append(len(got & want) / sh.budget)
    print("selection overlap: min %.4f mean %.4f" % (min(overlaps), float(np.mean(overlaps))))
    assert float(np.mean(overlaps)) > 0.9


def test_capacity_is_rejected_and_state_kept():
    from kv_cache_compression_frame_gb300 import StateKVError
    sh = _small("cap", frames=2)
    st = Stepper(sh)
    st.run(0)
    st.run(1)
    _, (q, k, v) = st.tensors(2)
    with pytest.raises(StateKVError) as ei:
        st.h.prefill_frame(q, k, v)
    assert ei.value.status == -3
    assert st.h.frame_index == 2


def test_host_entry_point_matches_device_entry_point():
    sh = _small("host", q_heads=4, kv_heads=2, head_dim=128, frame_tokens=64,
                budget=128, frames=4)
    a, b = Stepper(sh), Stepper(sh)
    for n in range(4):
        _, (q, k, v) = a.tensors(n)
        oa = a.h.prefill_frame(q, k, v)
        ob = torch.empty(oa.shape, dtype=oa.dtype).pin_memory()
        b.h.prefill_frame_host(q.cpu().pin_memory(), k.cpu().pin_memory(),
                               v.cpu().pin_memory(), ob)
        torch.cuda.synchronize()
        assert raw_equal(oa.cpu(), ob)
        ka, _, pa, ca = a.h.compressed(0, 0)
        kb, _, pb, cb = b.h.compressed(0, 0)
        assert ca == cb and torch.equal(pa[:, :ca], pb[:, :cb])
        assert raw_equal(ka[:, :ca], kb[:, :cb])


@pytest.mark.parametrize("chunks", [(5,), (1, 2, 3)])
def test_batched_host_entry_point_matches_device_entry_point(chunks):
    """Frames streamed from host memory with overlapped copies give the same
    bits as one device call per frame, whatever the batch boundaries."""
    sh = _small("hostbatch", q_heads=4, kv_heads=2, head_dim=128, frame_tokens=64,
                budget=128, frames=6)
    a, b = Stepper(sh), Stepper(sh)
    F = sum(chunks)
    tens = [a.tensors(n)[1] for n in range(F)]
    o_dev = [a.h.prefill_frame(q, k, v).cpu() for q, k, v in tens]
    hq = torch.stack([t[0].cpu() for t in tens]).pin_memory()
    hk = torch.stack([t[1].cpu() for t in tens]).pin_memory()
    hv = torch.stack([t[2].cpu() for t in tens]).pin_memory()
    ho = torch.empty(hq.shape, dtype=hq.dtype).pin_memory()
    f0 = 0
    for c in chunks:
        b.h.prefill_frames_host(hq[f0:f0 + c], hk[f0:f0 + c], hv[f0:f0 + c], ho[f0:f0 + c])
        f0 += c
    torch.cuda.synchronize()
    b.h.check_device_status()
    assert b.h.frame_index == F
    for n in range(F):
        assert raw_equal(o_dev[n], ho[n]), f"O frame {n}"
    ka, va, pa, ca = a.h.compressed(0, 0)
    kb, vb, pb, cb = b.h.compressed(0, 0)
    assert ca == cb and torch.equal(pa[:, :ca], pb[:, :cb])
    assert raw_equal(ka[:, :ca], kb[:, :cb]) and raw_equal(va[:, :ca], vb[:, :cb])
    # a batch past max_frames is rejected before any work
    from kv_cache_compression_frame_gb300 import StateKVError
    with pytest.raises(StateKVError) as ei:
        b.h.prefill_frames_host(hq[:2], hk[:2], hv[:2], ho[:2])
    assert ei.value.status == -3 and b.h.frame_index == F


def test_reset_replays_bit_identically():
    sh = _small("replay", q_heads=4, kv_heads=2, head_dim=64, frame_tokens=64,
                budget=96, frames=4)
    st = Stepper(sh)
    first = [st.run(n).cpu() for n in range(4)]
    st.h.reset()
    again = [st.run(n).cpu() for n in range(4)]
    for x, y in zip(first, again):
        assert raw_equal(x, y)


def test_profile_counts_every_launch():
    sh = _small("prof", frames=3)
    st = Stepper(sh)
    st.h.profile_enable(True)
    for n in range(3):
        st.run(n)
    prof = st.h.profile_read()
    # the RoPE table is computed once at create; every other kernel once per frame
    assert prof.pop("rope_table") == (0.0, 0), prof
    assert all(cnt == 3 for _, cnt in prof.values()), prof
    assert all(ms > 0 for ms, _ in prof.values()), prof


def test_profile_kernels_brackets_only_the_chosen_kernel():
    sh = _small("prof1", frames=3)
    st = Stepper(sh)
    st.h.profile_kernels("attention")
    st.h.profile_enable(True)
    for n in range(3):
        st.run(n)
    prof = st.h.profile_read()
    assert prof["attention"][1] == 3 and prof["attention"][0] > 0, prof
    assert all(cnt == 0 for k, (_, cnt) in prof.items() if k != "attention"), prof
    with pytest.raises(ValueError):
        st.h.profile_kernels("nope")


class _ZeroKeys:
    """Frames of a source with every key set to zero (every logit 0)."""

    def __init__(self, src):
        self.src = src

    def frame(self, n):
        q, k, v = self.src.frame(n)
        return q, np.zeros_like(k), v


@pytest.mark.parametrize("cluster", ["1", "8"])
def test_exact_score_ties_keep_the_lower_positions(cluster, monkeypatch):
    """With K = 0 (so K' = 0 after RoPE) every logit is 0 and P is uniform
    over each query row's visible keys: every compressed key and the frame's
    key 0 (visible to every row) get bit-identical scores, the frame's later
    keys strictly lower ones.  Once the state is full the cut (E = T
    evictions) falls inside that tied group -- keys 1..T-1 plus one of the
    tied keys -- and the tie rule (the lower position wins) keeps the
    compressed keys: C holds positions 0..B-1 for ever.  Checked exactly, with
    no near-tie allowance.  Run with each unit's selection on one CTA and on
    a cluster of eight."""
    monkeypatch.setenv("STATEKV_SELECT_CLUSTER", cluster)
    sh = _small("ties", q_heads=4, kv_heads=2, layers=2, frames=7)
    st = Stepper(sh)
    st.src = _ZeroKeys(st.src)
    T, B = sh.frame_tokens, sh.budget
    for n in range(sh.frames):
        c = min(n * T, B)
        st.step(n)
        for l in range(sh.layers):
            sc, _, m = st.h.scores(0, l)
            _, _, npos, ncnt = st.h.compressed(0, l)
            for hk in range(sh.kv_heads):
                s = sc[hk, :m].cpu().numpy()
                assert (s[:c + 1] == s[0]).all(), f"frame {n} layer {l} head {hk}: tied scores differ"
                assert (s[c + 1:] < s[0]).all(), f"frame {n} layer {l} head {hk}: frame key above the tie"
                kept = np.sort(npos[hk, :ncnt].cpu().numpy().astype(np.int64))
                np.testing.assert_array_equal(kept, np.arange(min(B, (n + 1) * T)))


@pytest.mark.parametrize("cluster", ["1", "4"])
def test_window_policy_keeps_the_most_recent_tokens(cluster, monkeypatch):
    """The sliding-window baseline on the same kernels: every step checked,
    through the fill and well past it."""
    monkeypatch.setenv("STATEKV_SELECT_CLUSTER", cluster)
    sh = _small("window", q_heads=4, kv_heads=2, head_dim=128, frame_tokens=64,
                budget=160, frames=6)
    st = Stepper(sh, policy="window")
    for n in range(sh.frames):
        st.step(n)


def test_full_attention_beyond_the_selection_limit():
    """B >= max_frames*T never evicts: full causal self-attention over the
    whole stream, with a pool (26,112 rows) larger than selection supports."""
    sh = _small("fullsa", q_heads=2, kv_heads=1, head_dim=64, frame_tokens=256,
                budget=102 * 256, frames=102)
    st = Stepper(sh)
    for n in range(sh.frames - 2):
        st.run(n)
    for n in (sh.frames - 2, sh.frames - 1):
        st.step(n)
    _, _, _, cnt = st.h.compressed(0, 0)
    assert cnt == sh.frames * sh.frame_tokens


@pytest.mark.parametrize("head_dim,q_heads,kv_heads,T,B", [
    (128, 6, 2, 1, 5),        # one token per frame, G = 3, budget below a tile
    (64, 6, 2, 3, 7),         # odd T, odd B
    (128, 3, 1, 129, 130),    # G*T = 387: a ragged fourth query tile, pool 259 rows
    (64, 2, 2, 33, 0),        # G = 1, per-frame attention only
    (64, 4, 2, 16, 8),        # budget below a frame: holes and movers at most B each
])
def test_odd_shapes_every_step(head_dim, q_heads, kv_heads, T, B):
    sh = _small("odd", q_heads=q_heads, kv_heads=kv_heads, head_dim=head_dim,
                frame_tokens=T, budget=B, frames=6)
    st = Stepper(sh)
    for n in range(sh.frames):
        st.step(n)


def test_overlapped_launches_match_serialised():
    """Frames launched back to back (the next frame's RoPE starting while the
    selection still runs, the attention set-up overlapping RoPE's end) give
    the same bits as the same frames with events between every launch,
    which serialise them.  Several units and query tiles, eviction every frame."""
    from kv_cache_compression_frame_gb300 import StateKV, StateKVConfig
    sh = _small("overlap", layers=4, q_heads=8, kv_heads=2, head_dim=128, frame_tokens=128,
                budget=256, frames=10)
    src = FrameSource(sh)
    dev = torch.device("cuda:0")
    frames = [tuple(torch.from_numpy(a).to(torch.bfloat16).to(dev) for a in src.frame(n))
              for n in range(sh.frames)]
    outs = {}
    for mode in ("overlapped", "serialised"):
        h = StateKV(StateKVConfig.from_shape(sh))
        if mode == "serialised":
            h.profile_enable(True)
        os_ = [torch.empty_like(frames[0][0]) for _ in range(sh.frames)]
        torch.cuda.synchronize()
        for n, (q, k, v) in enumerate(frames):
            h.prefill_frame(q, k, v, os_[n])
        torch.cuda.synchronize()
        h.check_device_status()
        comp = [h.compressed(0, l) for l in range(sh.layers)]
        outs[mode] = ([o.cpu() for o in os_],
                      [(ck[:, :cnt].cpu(), cv[:, :cnt].cpu(), cp[:, :cnt].cpu()) for ck, cv, cp, cnt in comp])
        h.close()
    (oa, ca), (ob, cb) = outs["overlapped"], outs["serialised"]
    for n in range(sh.frames):
        assert torch.equal(oa[n].view(torch.int16), ob[n].view(torch.int16)), f"O of frame {n}"
    for l in range(sh.layers):
        for x, y in zip(ca[l], cb[l]):
            assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                               y.view(torch.int16) if y.dtype == torch.bfloat16 else y), f"C of layer {l}"


@pytest.mark.parametrize("split,ways,head_dim,q_heads,kv_heads,T,B", [
    ("all", 2, 128, 8, 2, 128, 256),  # every query tile as a key-split CTA pair
    ("all", 2, 64, 6, 2, 3, 7),       # one-tile keys: one half holds none
    ("3", 2, 128, 6, 2, 64, 200),     # the last three tiles split, the rest whole
    ("all", 3, 128, 8, 2, 128, 300),  # odd ways: owner blocks of 48 columns, the last 32
    ("all", 4, 64, 6, 2, 64, 700),    # 16-column owner blocks
    ("all", 5, 64, 14, 2, 64, 1000),  # 16-column blocks, the fifth CTA owns none
    ("all", 6, 128, 12, 2, 96, 900),  # 24-column blocks spanning 32-column chunks
    ("all", 8, 128, 4, 2, 128, 1200), # eight CTAs, 16-column blocks
    ("all", 8, 64, 6, 2, 3, 7),       # more CTAs than key tiles: most hold none
    ("2", 4, 128, 12, 2, 64, 200),    # 6 tiles: 4 whole (one cluster of 4), 2 split 4 ways
])
def test_key_split_query_tiles(split, ways, head_dim, q_heads, kv_heads, T, B, monkeypatch):
    """Query tiles computed by the `ways` CTAs of a cluster, one key range
    each (lse partials and O columns exchanged through distributed shared
    memory): every frame against the oracle."""
    monkeypatch.setenv("STATEKV_ATTN_SPLIT", split)
    monkeypatch.setenv("STATEKV_ATTN_SPLIT_WAYS", str(ways))
    sh = _small("split", q_heads=q_heads, kv_heads=kv_heads, head_dim=head_dim,
                frame_tokens=T, budget=B, frames=6)
    st = Stepper(sh)
    for n in range(sh.frames):
        st.step(n)


@pytest.mark.parametrize("name", ["internvl3_2b_stack", "qwen3vl_2b_stack"])
def test_one_layer_per_launch_steady_state(name):
    """One layer per launch (a model whose layers feed each other): fewer
    query tiles than SMs, so every tile's keys are spread over a cluster of
    CTAs chosen from the device's cluster occupancy; checked on every unit
    through the fill and at a full state."""
    sh = SHAPES[name].with_(name=f"{name}_1layer", layers=1, frames=24)
    st = Stepper(sh)
    for n in range(sh.frames):
        if n in (0, 1, 16, 17):
            st.step(n)
        else:
            st.run(n)


def test_split_launches_are_deterministic():
    """A split launch gives the same bits on a replay (every CTA of a split
    tile combines the partials in rank order)."""
    sh = SHAPES["internvl3_1b_layer"].with_(frames=20)
    st = Stepper(sh)
    first = [st.run(n).cpu() for n in range(18)]
    st.h.reset()
    again = [st.run(n).cpu() for n in range(18)]
    for x, y in zip(first, again):
        assert raw_equal(x, y)


@pytest.mark.parametrize("cluster", ["1", "2", "4", "8"])
def test_select_cluster_sizes_agree(cluster, monkeypatch):
    """A unit's selection spread over 1, 2, 4 or 8 CTAs of a cluster (each
    finishes the scores of a slice of the candidates, the keys are shared
    through distributed shared memory, every CTA runs the cut and moves a
    share of the rows): every frame against the oracle, and the same scores,
    kept positions and C contents, bit for bit, as on one CTA."""
    sh = _small("selcl", layers=3, q_heads=4, kv_heads=2, head_dim=128, frame_tokens=64,
                budget=160, frames=6)
    monkeypatch.setenv("STATEKV_SELECT_CLUSTER", "1")
    ref = Stepper(sh)
    monkeypatch.setenv("STATEKV_SELECT_CLUSTER", cluster)
    st = Stepper(sh)
    for n in range(sh.frames):
        monkeypatch.setenv("STATEKV_SELECT_CLUSTER", "1")
        ref.run(n)
        monkeypatch.setenv("STATEKV_SELECT_CLUSTER", cluster)
        st.step(n)
        for l in range(sh.layers):
            a, b = ref.h.compressed(0, l), st.h.compressed(0, l)
            assert a[3] == b[3]
            for x, y in zip(a[:3], b[:3]):
                assert raw_equal(x.cpu(), y.cpu()), f"C of layer {l}, frame {n}"
            sa, sb = ref.h.scores(0, l), st.h.scores(0, l)
            assert raw_equal(sa[0].cpu(), sb[0].cpu()), f"scores of layer {l}, frame {n}"
