"""Pins of the CPU oracle to things other than itself.

Each check below is fixed by the method's text or by mathematics, not by the
oracle: a hand-derived worked example, closed forms, special cases that reduce
to a textbook or library routine, brute force on tiny inputs, and invariants.
The mutation tests at the end plant plausible mistakes into the oracle (on the
CPU) and confirm that at least one pin catches each.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.statekv_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


class _Cfg:
    def __init__(self, **kw):
        self.streams, self.layers = 1, 1
        self.rope_alpha, self.rope_orig_ctx = 1.0, 0
        self.rope_theta = 1e4
        self.dtype = "f32"
        self.__dict__.update(kw)


# ----------------------------------------------------------------- pin checks
def check_golden_zero_keys(o=orc):
    """Worked example with all-zero keys: uniform attention over the visible
    keys, so P, O, s and the selection are rationals derived by hand."""
    g = _load("zero_keys_T2_B1.json")
    st = g["setup"]
    omega, ms = o.rope_frequencies(2, 1e4)
    scale = o.logit_scale(2, ms)
    # frame 0 always runs at B = 1; frame 1 at B = 1 and, separately, B = 2
    for budget1, key in ((1, "kept_positions"), (2, "kept_positions_if_B2")):
        state = o.UnitState(2)
        for n, budget in ((0, 1), (1, budget1)):
            q = np.array(st["q"][n], np.float64)
            k = np.zeros((2, 2))
            v = np.array(st["v"][n], np.float64)
            O, info = o.prefill_unit_frame(state, q, k, v, n, budget=budget,
                                           omega=omega, scale=scale, dtype="f32")
            exp = g[f"frame{n}"]
            np.testing.assert_array_equal(info["pool_pos"], exp["pool_positions"])
            np.testing.assert_allclose(info["P"][0], exp["P"], atol=1e-15)
            np.testing.assert_allclose(O[0], exp["O"], atol=1e-15)
            np.testing.assert_allclose(info["scores"], exp["scores"], atol=1e-15)
            want = exp[key] if n == 1 else exp["kept_positions"]
            np.testing.assert_array_equal(state.comp_pos, want)
        assert state.detailed_k.shape[0] == g["detailed_rows_after"]
        np.testing.assert_array_equal(state.detailed_v, np.concatenate(st["v"]))


def _complex_rope(x, positions, theta):
    """Textbook RoPE written with complex numbers: the pair (x_k, x_{k+d/2}) is
    the complex number x_k + i x_{k+d/2}, multiplied by exp(i p theta^(-2k/d))."""
    x = np.asarray(x, np.float64)
    assert x.ndim == 2
    d = x.shape[-1]
    half = d // 2
    out = np.empty_like(x)
    for t, p in enumerate(positions):
        for k in range(half):
            w = theta ** (-2.0 * k / d)
            z = complex(x[t, k], x[t, k + half])
            r = z * complex(math.cos(p * w), math.sin(p * w))
            out[t, k], out[t, k + half] = r.real, r.imag
    return out


def check_rope_complex(o=orc):
    rng = np.random.default_rng(1)
    for d, theta in ((8, 1e4), (16, 1e6)):
        x = rng.standard_normal((5, d))
        pos = np.array([0, 1, 7, 1000, 131071])
        omega, ms = o.rope_frequencies(d, theta)
        assert ms == 1.0
        got = o.rope_rotate(x, pos, omega)
        want = _complex_rope(x, pos, theta)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-9)


def _brute_full_causal(qs, ks, vs, theta, scale, G):
    """Ordinary causal self-attention over the whole token sequence, one query
    at a time, with float32-stored rotated q/k (loops; tiny inputs only).
    qs: [NT, Hq=G, d], ks/vs: [NT, d] (one KV head)."""
    NT, _, d = qs.shape
    pos = np.arange(NT)
    qr = np.stack([_complex_rope(qs[:, g, :], pos, theta) for g in range(G)], 1)
    kr = _complex_rope(ks, pos, theta)
    qr = qr.astype(np.float32).astype(np.float64)
    kr = kr.astype(np.float32).astype(np.float64)
    out = np.zeros_like(qs)
    for t in range(NT):
        for g in range(G):
            logits = [float(np.dot(qr[t, g], kr[j])) * scale for j in range(t + 1)]
            mx = max(logits)
            w = [math.exp(a - mx) for a in logits]
            tot = sum(w)
            out[t, g] = sum(w[j] / tot * vs[j] for j in range(t + 1))
    return out


def check_full_sa_when_budget_covers_all(o=orc):
    """With B >= N*T nothing is ever evicted, so every frame's output must be
    exactly full causal self-attention over the whole stream (Full SA)."""
    G, T, d, N = 2, 4, 8, 3
    theta = 1e4
    rng = np.random.default_rng(7)
    q = rng.standard_normal((N, G, T, d))
    k = rng.standard_normal((N, T, d))
    v = rng.standard_normal((N, T, d))
    omega, ms = o.rope_frequencies(d, theta)
    scale = o.logit_scale(d, ms)
    state = o.UnitState(d)
    outs = []
    for n in range(N):
        O, _ = o.prefill_unit_frame(state, q[n], k[n], v[n], n, budget=N * T,
                                    omega=omega, scale=scale, dtype="f32")
        outs.append(O.transpose(1, 0, 2))          # [T, G, d]
    got = np.concatenate(outs)
    # textbook softmax scale 1/sqrt(d) (alpha = 1)
    want = _brute_full_causal(q.transpose(0, 2, 1, 3).reshape(N * T, G, d),
                              k.reshape(N * T, d), v.reshape(N * T, d),
                              theta, 1.0 / math.sqrt(d), G)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def check_decode_is_full_causal_over_the_stream(o=orc):
    """Text decoded after N frames (in two calls) must equal the last rows of
    ordinary causal self-attention over the whole token sequence (video then
    text, positions 0..), whatever the budget B: decode reads the detailed
    state D, which holds every row.  B = 1 evicts almost everything from C."""
    G, T, d, N = 2, 4, 8, 3
    theta = 1e4
    rng = np.random.default_rng(11)
    q = rng.standard_normal((N, G, T, d))
    k = rng.standard_normal((N, T, d))
    v = rng.standard_normal((N, T, d))
    tq = rng.standard_normal((G, 3, d))
    tk = rng.standard_normal((3, d))
    tv = rng.standard_normal((3, d))
    omega, ms = o.rope_frequencies(d, theta)
    scale = o.logit_scale(d, ms)
    qs = np.concatenate([q.transpose(0, 2, 1, 3).reshape(N * T, G, d), tq.transpose(1, 0, 2)])
    want = _brute_full_causal(qs, np.concatenate([k.reshape(N * T, d), tk]),
                              np.concatenate([v.reshape(N * T, d), tv]), theta,
                              1.0 / math.sqrt(d), G)[N * T:]       # [3, G, d]
    for budget in (N * T, 1):
        state = o.UnitState(d)
        for n in range(N):
            o.prefill_unit_frame(state, q[n], k[n], v[n], n, budget=budget,
                                 omega=omega, scale=scale, dtype="f32")
        o1, _, _ = o.decode_unit_tokens(state, tq[:, :1], tk[:1], tv[:1], N * T,
                                        omega=omega, scale=scale, dtype="f32")
        o2, _, _ = o.decode_unit_tokens(state, tq[:, 1:], tk[1:], tv[1:], N * T + 1,
                                        omega=omega, scale=scale, dtype="f32")
        got = np.concatenate([o1, o2], axis=1).transpose(1, 0, 2)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
        assert state.detailed_k.shape[0] == N * T + 3


def check_window_policy_is_a_sliding_window(o=orc):
    """The sliding-window baseline (ReKV, compute-matched B): after every
    frame C holds exactly the B most recent positions, and each frame query at
    position p attends to the keys at positions [frame start - min(B, nT), p]
    -- a contiguous range, checked by brute force."""
    G, T, d, N, B = 2, 4, 8, 4, 6
    theta = 1e4
    rng = np.random.default_rng(5)
    q = rng.standard_normal((N, G, T, d))
    k = rng.standard_normal((N, T, d))
    v = rng.standard_normal((N, T, d))
    omega, ms = o.rope_frequencies(d, theta)
    scale = o.logit_scale(d, ms)
    pos_all = np.arange(N * T)
    qr = [np.stack([_complex_rope(q[n, g], n * T + np.arange(T), theta) for g in range(G)])
          .astype(np.float32).astype(np.float64) for n in range(N)]
    kr = _complex_rope(k.reshape(N * T, d), pos_all, theta).astype(np.float32).astype(np.float64)
    vv = v.reshape(N * T, d)
    state = o.UnitState(d)
    for n in range(N):
        O, _ = o.prefill_unit_frame(state, q[n], k[n], v[n], n, budget=B, omega=omega,
                                    scale=scale, dtype="f32", policy="window")
        kept = min(B, (n + 1) * T)
        np.testing.assert_array_equal(np.sort(state.comp_pos),
                                      np.arange((n + 1) * T - kept, (n + 1) * T))
        lo = n * T - min(B, n * T)
        for i in range(T):
            for g in range(G):
                js = range(lo, n * T + i + 1)
                logits = [float(np.dot(qr[n][g, i], kr[j])) / math.sqrt(d) for j in js]
                mx = max(logits)
                w = [math.exp(a - mx) for a in logits]
                want = sum(wj / sum(w) * vv[j] for wj, j in zip(w, js))
                np.testing.assert_allclose(O[g, i], want, rtol=0, atol=1e-12)


def check_zero_budget_is_per_frame_causal(o=orc):
    """B = 0: no cross-frame state, so each frame is plain causal attention
    over its own tokens -- torch's scaled_dot_product_attention in fp64."""
    G, T, d = 3, 6, 16
    theta = 1e6
    rng = np.random.default_rng(3)
    omega, ms = o.rope_frequencies(d, theta)
    scale = o.logit_scale(d, ms)
    state = o.UnitState(d)
    for n in range(3):
        q = rng.standard_normal((G, T, d))
        k = rng.standard_normal((T, d))
        v = rng.standard_normal((T, d))
        O, _ = o.prefill_unit_frame(state, q, k, v, n, budget=0, omega=omega,
                                    scale=scale, dtype="f32")
        pos = n * T + np.arange(T)
        qr = np.stack([_complex_rope(q[g], pos, theta) for g in range(G)])
        kr = _complex_rope(k, pos, theta)
        qr = torch.from_numpy(qr.astype(np.float32).astype(np.float64))
        kr = torch.from_numpy(kr.astype(np.float32).astype(np.float64))
        vt = torch.from_numpy(v)
        want = torch.nn.functional.scaled_dot_product_attention(
            qr[None], kr[None, None].expand(1, G, T, d),
            vt[None, None].expand(1, G, T, d), is_causal=True,
            scale=1.0 / math.sqrt(d))[0]
        np.testing.assert_allclose(O, want.numpy(), rtol=0, atol=1e-12)
        assert state.comp_k.shape[0] == 0


def check_topb_rank_definition(o=orc):
    """Top-B against the rank definition: j is kept iff fewer than B
    candidates beat it (higher score, or equal score at a lower position)."""
    rng = np.random.default_rng(11)
    for trial in range(30):
        m = int(rng.integers(1, 40))
        B = int(rng.integers(0, 45))
        s = rng.integers(0, 6, size=m).astype(np.float64) / 5.0   # many ties
        pos = rng.permutation(1000)[:m]
        keep = o.select_top_b(s, pos, B)
        want = [j for j in range(m)
                if sum((s[i] > s[j]) or (s[i] == s[j] and pos[i] < pos[j])
                       for i in range(m)) < B]
        assert sorted(keep.tolist()) == sorted(want)
        assert list(pos[keep]) == sorted(pos[keep])


def check_golden_alpha4_logit_temperature(o=orc):
    """Hand-evaluated alpha = 4 step (tests/golden/yarn_alpha4_logit_d4.json):
    the logit against a key at the query's own position is q.k * mscale^2 /
    sqrt(d) (a common rotation preserves the inner product), and a zero key
    gives logit 0, so P, O, the scores and the kept position are closed
    forms in mscale = 0.1 ln 4 + 1.  Runs through StateKVOracle, so the
    temperature is taken where the oracle itself takes it."""
    g = _load("yarn_alpha4_logit_d4.json")
    st = g["setup"]
    cfg = _Cfg(q_heads=st["G"], kv_heads=1, head_dim=st["head_dim"], frame_tokens=st["T"],
               budget=st["B"], rope_theta=st["theta"], rope_alpha=st["alpha"],
               rope_orig_ctx=st["orig_ctx"], dtype=st["dtype"])
    ref = o.StateKVOracle(cfg)
    assert abs(ref.mscale ** 2 - g["mscale_squared"]) < 1e-9
    q = np.array(st["q"], np.float64)[None, None, None]      # [S][L][Hq][T][d]
    k = np.array(st["k"], np.float64)[None, None, None]
    v = np.array(st["v"], np.float64)[None, None, None]
    O, infos = ref.prefill_frame(q, k, v, keep_info=True)
    tol = g["abs_tol"]
    np.testing.assert_allclose(O[0, 0, 0], g["O"], rtol=0, atol=tol)
    info = infos[(0, 0, 0)]
    np.testing.assert_allclose(info["scores"], g["scores"], rtol=0, atol=tol)
    np.testing.assert_array_equal(ref.units[(0, 0, 0)].comp_pos, g["kept_positions"])
    # the probabilities themselves, through the unit-level attention
    unit = o.UnitState(st["head_dim"])
    omega, ms = o.rope_frequencies(st["head_dim"], st["theta"], st["alpha"], st["orig_ctx"])
    _, info = o.prefill_unit_frame(unit, q[0, 0, 0:1], k[0, 0, 0], v[0, 0, 0], 0,
                                   budget=st["B"], omega=omega,
                                   scale=o.logit_scale(st["head_dim"], ms), dtype=st["dtype"])
    np.testing.assert_allclose(info["P"][0], g["P"], rtol=0, atol=tol)


def _per_head_causal(q_h, k_h, v_h, pos, theta, scale):
    """Causal attention of one query head over one KV head's keys, one query
    at a time (loops), with fp32-stored rotated q/k.  q_h, k_h, v_h: [T, d]
    for a single frame at positions pos.  Returns (O [T, d], P [T, T])."""
    T, d = q_h.shape
    qr = _complex_rope(q_h, pos, theta).astype(np.float32).astype(np.float64)
    kr = _complex_rope(k_h, pos, theta).astype(np.float32).astype(np.float64)
    out = np.zeros((T, d))
    P = np.zeros((T, T))
    for i in range(T):
        logits = [float(np.dot(qr[i], kr[j])) * scale for j in range(i + 1)]
        mx = max(logits)
        w = [math.exp(a - mx) for a in logits]
        tot = sum(w)
        for j in range(i + 1):
            P[i, j] = w[j] / tot
            out[i] += P[i, j] * v_h[j]
    return out, P


def check_gqa_head_grouping(o=orc):
    """Query head j attends with KV head j // G (G = Hq / Hkv consecutive
    query heads share a KV head), and the scores of KV head h average the P
    of exactly those G heads.  StateKVOracle on Hq = 4, Hkv = 2 against
    per-query-head brute force: full causal attention over the whole stream
    (B covers every frame), and the first frame's scores."""
    Hq, Hkv, T, d, N = 4, 2, 3, 8, 3
    G = Hq // Hkv
    theta = 1e4
    rng = np.random.default_rng(21)
    q = rng.standard_normal((N, 1, 1, Hq, T, d))
    k = rng.standard_normal((N, 1, 1, Hkv, T, d))
    v = rng.standard_normal((N, 1, 1, Hkv, T, d))
    cfg = _Cfg(q_heads=Hq, kv_heads=Hkv, head_dim=d, frame_tokens=T, budget=N * T,
               rope_theta=theta, dtype="f32")
    ref = o.StateKVOracle(cfg)
    outs = [ref.prefill_frame(q[n], k[n], v[n]) for n in range(N)]
    for j in range(Hq):
        h = j // G
        want = _brute_full_causal(q[:, 0, 0, j][:, None].transpose(0, 2, 1, 3).reshape(N * T, 1, d),
                                  k[:, 0, 0, h].reshape(N * T, d), v[:, 0, 0, h].reshape(N * T, d),
                                  theta, 1.0 / math.sqrt(d), 1)[:, 0]
        got = np.concatenate([outs[n][0, 0, j] for n in range(N)])
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
    # scores of the first frame (no compressed keys): per KV head, the mean
    # over its G query heads and T rows of each head's P
    cfg2 = _Cfg(q_heads=Hq, kv_heads=Hkv, head_dim=d, frame_tokens=T, budget=1,
                rope_theta=theta, dtype="f32")
    ref2 = o.StateKVOracle(cfg2)
    _, infos = ref2.prefill_frame(q[0], k[0], v[0], keep_info=True)
    pos = np.arange(T)
    for h in range(Hkv):
        acc = np.zeros(T)
        for j in range(h * G, (h + 1) * G):
            _, P = _per_head_causal(q[0, 0, 0, j], k[0, 0, 0, h], v[0, 0, 0, h], pos, theta,
                                    1.0 / math.sqrt(d))
            acc += P.sum(0)
        np.testing.assert_allclose(infos[(0, 0, h)]["scores"], acc / (G * T), rtol=0, atol=1e-12)


# ----------------------------------------------------------------- the tests
def test_golden_zero_keys():
    check_golden_zero_keys()


def test_rope_is_complex_rotation():
    check_rope_complex()


def test_full_sa_special_case():
    check_full_sa_when_budget_covers_all()


def test_decode_matches_full_causal_over_the_stream():
    check_decode_is_full_causal_over_the_stream()


def test_window_policy_is_a_sliding_window():
    check_window_policy_is_a_sliding_window()


def test_zero_budget_matches_sdpa():
    check_zero_budget_is_per_frame_causal()


def test_topb_rank_definition():
    check_topb_rank_definition()


def test_golden_alpha4_logit_temperature():
    check_golden_alpha4_logit_temperature()


def test_gqa_head_grouping():
    check_gqa_head_grouping()


def test_yarn_golden_and_limits():
    g = _load("yarn_d4.json")
    om, ms = orc.rope_frequencies(g["head_dim"], g["theta"], g["alpha"], g["orig_ctx"])
    np.testing.assert_allclose(om, g["omega"], atol=g["abs_tol"])
    assert abs(ms - g["mscale"]) < g["abs_tol"]
    # alpha == 1 is plain RoPE whatever L_orig says
    plain, m1 = orc.rope_frequencies(128, 1e6)
    same, m2 = orc.rope_frequencies(128, 1e6, 1.0, 32960)
    np.testing.assert_array_equal(plain, same)
    assert m1 == m2 == 1.0
    # very high frequencies (many turns inside L_orig) are left alone; the
    # lowest frequencies are interpolated by exactly 1/alpha
    om4, _ = orc.rope_frequencies(128, 1e6, 4.0, 32960)
    wl = 2 * math.pi / plain
    hi = 32960 / wl > 32
    lo = 32960 / wl < 1
    assert hi.any() and lo.any()
    np.testing.assert_array_equal(om4[hi], plain[hi])
    np.testing.assert_allclose(om4[lo], plain[lo] / 4.0, rtol=1e-15)
    assert np.all(np.diff(om4) < 0)            # still strictly decreasing
    assert np.all(om4 <= plain) and np.all(om4 >= plain / 4.0)


def test_rope_norm_and_relative_position():
    rng = np.random.default_rng(5)
    d = 64
    omega, _ = orc.rope_frequencies(d, 1e6, 4.0, 32960)
    x = rng.standard_normal((7, d))
    y = rng.standard_normal((7, d))
    p = np.arange(7) * 911 + 3
    xr = orc.rope_rotate(x, p, omega)
    # per-pair norms are preserved by a rotation
    h = d // 2
    np.testing.assert_allclose(xr[:, :h] ** 2 + xr[:, h:] ** 2,
                               x[:, :h] ** 2 + x[:, h:] ** 2, rtol=1e-12)
    # q'(p)·k'(p') depends only on p - p' (the property virtual positions keep)
    for delta in (1, 4096, 131072):
        a = orc.rope_rotate(x, p, omega) @ orc.rope_rotate(y, p[::-1], omega).T
        b = orc.rope_rotate(x, p + delta, omega) @ orc.rope_rotate(y, p[::-1] + delta, omega).T
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-9 * np.abs(a).max())


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    x32 = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                          (rng.standard_normal(2000) * 1e-30).astype(np.float32),
                          np.array([0.0, -0.0, 1.0, 3.0], np.float32)])
    # include exact midpoints between neighbouring bf16 values (ties to even)
    mids = (torch.arange(1, 200, dtype=torch.int32) << 16) | (1 << 15)
    x32 = np.concatenate([x32, mids.view(torch.float32).numpy()])
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(orc.bf16_round(x32.astype(np.float64)), want)


def test_scores_are_a_distribution():
    rng = np.random.default_rng(9)
    G, T, d, c = 3, 10, 16, 17
    q = rng.standard_normal((G, T, d))
    K = rng.standard_normal((c + T, d))
    V = rng.standard_normal((c + T, d))
    O, P = orc.attend_frame(q, K, V, c, 0.3)
    np.testing.assert_allclose(P.sum(-1), 1.0, atol=1e-14)
    s = orc.importance_scores(P)
    assert np.all(s >= 0)
    assert abs(s.sum() - 1.0) < 1e-14
    # masked entries are exactly zero; O is a convex combination of V rows
    for i in range(T):
        assert np.all(P[:, i, c + i + 1:] == 0)
    assert np.all(O <= V.max(0) + 1e-12) and np.all(O >= V.min(0) - 1e-12)


def test_gqa_duplicate_heads_and_single_head():
    rng = np.random.default_rng(4)
    T, d, c = 8, 16, 5
    q1 = rng.standard_normal((1, T, d))
    K = rng.standard_normal((c + T, d))
    V = rng.standard_normal((c + T, d))
    O1, P1 = orc.attend_frame(q1, K, V, c, 0.25)
    O2, P2 = orc.attend_frame(np.concatenate([q1, q1]), K, V, c, 0.25)
    np.testing.assert_array_equal(O2[0], O1[0])
    np.testing.assert_array_equal(O2[1], O1[0])
    np.testing.assert_allclose(orc.importance_scores(P2), orc.importance_scores(P1),
                               rtol=1e-15)
    # with one head, s_j is the plain mean over the T queries
    np.testing.assert_allclose(orc.importance_scores(P1), P1[0].mean(0), rtol=1e-15)


def test_state_invariants_over_a_stream():
    cfg = _Cfg(q_heads=4, kv_heads=2, head_dim=16, frame_tokens=5, budget=12,
               rope_theta=1e6, rope_alpha=4.0, rope_orig_ctx=40, dtype="bf16")
    o = orc.StateKVOracle(cfg)
    rng = np.random.default_rng(6)
    for n in range(7):
        q = rng.standard_normal((1, 1, 4, 5, 16))
        k = rng.standard_normal((1, 1, 2, 5, 16))
        v = orc.bf16_round(rng.standard_normal((1, 1, 2, 5, 16)))
        o.prefill_frame(q, k, v)
        for st in o.units.values():
            c = st.comp_k.shape[0]
            assert c == min(cfg.budget, (n + 1) * 5)
            assert st.detailed_k.shape[0] == (n + 1) * 5
            assert len(set(st.comp_pos.tolist())) == c
            assert st.comp_pos.min() >= 0 and st.comp_pos.max() < (n + 1) * 5
            # compressed rows are copies of detailed rows at the same position
            np.testing.assert_array_equal(st.comp_k, st.detailed_k[st.comp_pos])
            np.testing.assert_array_equal(st.comp_v, st.detailed_v[st.comp_pos])
            # stored keys are storage-rounded
            np.testing.assert_array_equal(st.detailed_k, orc.bf16_round(st.detailed_k))


# -------------------------------------------------------- planted mistakes
def _mut_mask_offbyone(monkeypatch):
    real = orc.attend_frame

    def bad(q_rot, pool_k, pool_v, n_compressed, scale):
        # frame key i' visible iff i' < i  (drops the diagonal) -- emulate by
        # shifting the compressed count so the diagonal is masked
        q = np.asarray(q_rot, np.float64)
        K = np.asarray(pool_k, np.float64)
        V = np.asarray(pool_v, np.float64)
        G, T, _ = q.shape
        m = K.shape[0]
        c = n_compressed
        z = np.einsum("gtd,jd->gtj", q, K) * scale
        i = np.arange(T)[:, None]
        j = np.arange(m)[None, :]
        vis = (j < c) | ((j - c) < i) | ((i == 0) & (j == c))
        z = np.where(vis[None], z, -np.inf)
        z = z - z.max(-1, keepdims=True)
        e = np.where(vis[None], np.exp(z), 0.0)
        P = e / e.sum(-1, keepdims=True)
        return np.einsum("gtj,jd->gtd", P, V), P
    monkeypatch.setattr(orc, "attend_frame", bad)
    return real


def _mut_score_visible_mean(monkeypatch):
    def bad(P):
        G, T, m = P.shape
        flat = P.reshape(G * T, m)
        cnt = np.maximum((flat > 0).sum(0), 1)
        return flat.sum(0) / cnt
    monkeypatch.setattr(orc, "importance_scores", bad)


def _mut_tiebreak_high(monkeypatch):
    def bad(scores, positions, budget):
        s = np.asarray(scores, np.float64)
        p = np.asarray(positions, np.int64)
        if s.shape[0] <= budget:
            keep = np.arange(s.shape[0])
        else:
            keep = np.lexsort((-p, -s))[:budget]
        return keep[np.argsort(p[keep], kind="stable")]
    monkeypatch.setattr(orc, "select_top_b", bad)


def _mut_rope_sign(monkeypatch):
    def bad(x, positions, omega):
        x = np.asarray(x, np.float64)
        h = x.shape[-1] // 2
        ang = np.asarray(positions, np.float64)[:, None] * omega[None, :]
        a, b = x[..., :h], x[..., h:]
        return np.concatenate([a * np.cos(ang) + b * np.sin(ang),
                               b * np.cos(ang) - a * np.sin(ang)], -1)
    monkeypatch.setattr(orc, "rope_rotate", bad)


def _mut_rope_freq_index(monkeypatch):
    real = orc.rope_frequencies

    def bad(head_dim, theta, alpha=1.0, orig_ctx=0):
        om, ms = real(head_dim, theta, alpha, orig_ctx)
        k = np.arange(head_dim // 2)
        return np.power(float(theta), -1.0 * k / head_dim), ms   # 2k/d -> k/d
    monkeypatch.setattr(orc, "rope_frequencies", bad)


def _mut_no_scale(monkeypatch):
    monkeypatch.setattr(orc, "logit_scale", lambda d, ms: 1.0)


def _mut_pv_transposed_heads(monkeypatch):
    real = orc.attend_frame

    def bad(q_rot, pool_k, pool_v, n_compressed, scale):
        O, P = real(q_rot, pool_k, pool_v, n_compressed, scale)
        return O[::-1].copy(), P
    monkeypatch.setattr(orc, "attend_frame", bad)


_CHECKS = [check_golden_zero_keys, check_rope_complex,
           check_full_sa_when_budget_covers_all, check_decode_is_full_causal_over_the_stream,
           check_window_policy_is_a_sliding_window,
           check_zero_budget_is_per_frame_causal, check_topb_rank_definition,
           check_golden_alpha4_logit_temperature, check_gqa_head_grouping]


def _mut_decode_reads_compressed(monkeypatch):
    def bad(state, q, k, v, first_row, *, omega, scale, dtype, position_offset=0):
        tok = k.shape[0]
        pos = position_offset + first_row + np.arange(tok, dtype=np.int64)
        q_rot = orc.round_to_storage(orc.rope_rotate(q, pos, omega), dtype)
        k_rot = orc.round_to_storage(orc.rope_rotate(k, pos, omega), dtype)
        c = state.comp_k.shape[0]
        O, _ = orc.attend_frame(q_rot, np.concatenate([state.comp_k, k_rot]),
                                np.concatenate([state.comp_v, v]), c, scale)
        state.det_k.append(k_rot)
        state.det_v.append(np.asarray(v, np.float64))
        return O, q_rot, k_rot
    monkeypatch.setattr(orc, "decode_unit_tokens", bad)


def _mut_decode_position_restart(monkeypatch):
    good = orc.decode_unit_tokens
    def bad(state, q, k, v, first_row, **kw):
        return good(state, q, k, v, first_row, **kw) if first_row == 0 else \
            _shifted(good, state, q, k, v, first_row, kw)
    def _shifted(fn, state, q, k, v, first_row, kw):
        kw = dict(kw)
        kw["position_offset"] = kw.get("position_offset", 0) - first_row   # text from p = 0
        return fn(state, q, k, v, first_row, **kw)
    monkeypatch.setattr(orc, "decode_unit_tokens", bad)


def _mut_window_keeps_oldest(monkeypatch):
    def bad(positions, budget):
        m = positions.shape[0]
        return np.arange(m) if m <= budget else np.sort(np.argsort(positions)[:budget])
    monkeypatch.setattr(orc, "select_window", bad)


def _mut_mscale_not_squared(monkeypatch):
    # the YaRN temperature applied once instead of squared
    monkeypatch.setattr(orc, "logit_scale", lambda d, ms: ms / math.sqrt(d))


def _mut_no_temperature(monkeypatch):
    # alpha != 1 without the YaRN temperature: the plain 1/sqrt(d)
    monkeypatch.setattr(orc, "logit_scale", lambda d, ms: 1.0 / math.sqrt(d))


def _mut_heads_interleaved(monkeypatch):
    # query head j paired with KV head j % Hkv instead of j // G
    class Bad(orc.StateKVOracle):
        def prefill_frame(self, q, k, v, keep_info=False):
            cfg = self.cfg
            O = np.zeros(np.shape(q), np.float64)
            infos = {}
            for (s, l, h), st in self.units.items():
                heads = list(range(h, cfg.q_heads, cfg.kv_heads))
                o_, info = orc.prefill_unit_frame(
                    st, np.asarray(q[s][l])[heads], k[s][l][h], v[s][l][h], self.n,
                    budget=cfg.budget, omega=self.omega, scale=self.scale,
                    dtype=cfg.dtype, position_offset=self.offset)
                O[s, l, heads] = o_
                if keep_info:
                    info.pop("P")
                    infos[(s, l, h)] = info
            self.n += 1
            return (O, infos) if keep_info else O
    monkeypatch.setattr(orc, "StateKVOracle", Bad)


@pytest.mark.parametrize("mutation", [
    _mut_mask_offbyone, _mut_window_keeps_oldest, _mut_score_visible_mean, _mut_tiebreak_high,
    _mut_rope_sign, _mut_rope_freq_index, _mut_no_scale,
    _mut_pv_transposed_heads, _mut_decode_reads_compressed,
    _mut_decode_position_restart, _mut_mscale_not_squared, _mut_no_temperature,
    _mut_heads_interleaved])
def test_planted_mistake_is_caught(monkeypatch, mutation):
    mutation(monkeypatch)
    caught = 0
    for chk in _CHECKS:
        try:
            chk(orc)
        except AssertionError:
            caught += 1
    assert caught >= 1, f"no pin caught {mutation.__name__}"
