"""Plain fp64 CPU definition of StateKV streaming video prefill.

TEST INFRASTRUCTURE ONLY: this module is the oracle the CUDA path is checked
against.  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg
and reference arm may import it; the product path never does.

Source: "Linear Scaling Video VLMs for Long Video Understanding" (StateKV,
ECCV 2026), papernotes.org summary, section 方法详解:
  * 整体框架            -- two decoupled phases; per frame and layer the frame's
                          T tokens attend only to the compressed state C_{n-1}
                          and to the frame itself; per-frame cost O(T^2 + BT);
  * 关键设计 1 双状态解耦  -- detailed state D_n (every frame's K/V, kept for
                          decoding) and compressed state C_n with |K̄_n| = B;
                          Q_n attends over [K̄_{n-1}; K_n];
  * 关键设计 2 时间汇元更新 -- candidate pool U_n = S̄_{n-1} ∪ {1..T}; score s_j =
                          mean attention paid to key j by the frame's queries;
                          S̄_n = TopK({s_j}, B) builds C_n;
  * 关键设计 3 虚拟序列长度 -- virtual length L_n = nT, every RoPE angle uses the
                          logical stream position; one global RoPE scale alpha
                          ("e.g. YaRN") fixed before prefill for the whole run.

The page's two equations (the attention after "执行注意力计算" and the score
after "平均值确定") did not survive text extraction.  Readings taken where the
page is silent (all listed with reasons in the design notes):
  R1 mask: compressed keys fully visible; frame key i' visible to query i iff
     i' <= i (causal inside the frame, as in the frozen causal LLM);
  R2 score normaliser: divide by the number of query rows (G*T); a query that
     cannot see key j contributes 0;
  R3 GQA: average over the G query heads sharing a KV head; one index set per
     (stream, layer, KV head);
  R4 ties in Top-B go to the lower virtual position;
  R5 positions p_i = offset + n*T + i with n 0-based;
  R6 static scale alpha = YaRN "NTK-by-parts" (beta_fast 32, beta_slow 1) with
     attention temperature mscale = 0.1 ln(alpha) + 1 applied to the logits as
     mscale^2;
  R7 C and D hold post-RoPE keys, rounded to the storage dtype (the positions
     never change because alpha is fixed);
  R8 |C_n| = min(B, (n+1) T) before the state fills;
  R9 the order of rows inside C is not part of the state (a set with
     positions); this oracle keeps ascending position.

Everything is float64; the only roundings are the storage-dtype roundings of
the rotated Q/K (R7), which define what the CUDA path stores.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


# ---------------------------------------------------------------- RoPE (关键设计 3)
def rope_frequencies(head_dim: int, theta: float, alpha: float = 1.0,
                     orig_ctx: int = 0) -> tuple[np.ndarray, float]:
    """Angular frequency omega_k for each rotated pair k = 0..d/2-1 and the
    logit temperature factor mscale.

    Plain RoPE: omega_k = theta^(-2k/d).  With a static scale alpha != 1 (the
    page's "全局 RoPE 缩放因子 alpha (如 YaRN)"), the YaRN NTK-by-parts rule:
    wavelength lambda_k = 2 pi / omega_k, ratio r_k = L_orig / lambda_k,
    ramp gamma_k = clamp((r_k - 1) / (32 - 1), 0, 1), and
    omega'_k = (1 - gamma_k) * omega_k / alpha + gamma_k * omega_k;
    mscale = 0.1 ln(alpha) + 1 (1 when alpha == 1).
    """
    if head_dim % 2:
        raise ValueError("head_dim must be even")
    k = np.arange(head_dim // 2, dtype=np.float64)
    omega = np.power(float(theta), -2.0 * k / head_dim)
    if alpha == 1.0:
        return omega, 1.0
    if orig_ctx <= 0:
        raise ValueError("alpha != 1 needs the original context length")
    wavelength = 2.0 * math.pi / omega
    r = float(orig_ctx) / wavelength
    gamma = np.clip((r - 1.0) / (32.0 - 1.0), 0.0, 1.0)
    omega = (1.0 - gamma) * omega / alpha + gamma * omega
    return omega, 0.1 * math.log(alpha) + 1.0


def rope_rotate(x: np.ndarray, positions: np.ndarray,
                omega: np.ndarray) -> np.ndarray:
    """Rotate-half RoPE: pair (k, k + d/2) is turned by angle p * omega_k.

    x: [..., T, d]; positions: [T] (virtual stream positions, 关键设计 3)."""
    x = np.asarray(x, np.float64)
    half = x.shape[-1] // 2
    ang = np.asarray(positions, np.float64)[:, None] * omega[None, :]
    cos, sin = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), returned
    as float64.  bfloat16 keeps 8 significant bits and float32's exponent."""
    x = np.asarray(x, np.float64)
    out = np.array(x, copy=True)
    nz = np.isfinite(x) & (x != 0.0)
    _, e = np.frexp(x[nz])                    # |x| in [2^(e-1), 2^e)
    quantum = np.maximum(e - 1, -126) - 7     # exponent of one bf16 ulp
    out[nz] = np.ldexp(np.rint(np.ldexp(x[nz], -quantum)), quantum)
    return out


def round_to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """The storage boundary: bf16 (RNE) or float32 (RNE)."""
    if dtype == "bf16":
        return bf16_round(x)
    if dtype == "f32":
        return np.asarray(x, np.float64).astype(np.float32).astype(np.float64)
    raise ValueError(dtype)


def logit_scale(head_dim: int, mscale: float) -> float:
    """Softmax logit scale: mscale^2 / sqrt(d)."""
    return mscale * mscale / math.sqrt(head_dim)


# ------------------------------------------------- frame attention (关键设计 1)
def attend_frame(q_rot: np.ndarray, pool_k: np.ndarray, pool_v: np.ndarray,
                 n_compressed: int, scale: float):
    """Attention of the frame's queries over [K̄_{n-1}; K_n].

    q_rot: [G, T, d] rotated queries of the G query heads sharing one KV head.
    pool_k, pool_v: [c + T, d]; rows 0..c-1 are the compressed state, rows
    c..c+T-1 the frame's own (rotated) keys/values in token order.
    Visibility (R1): every compressed key; frame key i' iff i' <= i.
    Returns O [G, T, d] and the probabilities P [G, T, c + T] (0 where masked).
    """
    q = np.asarray(q_rot, np.float64)
    K = np.asarray(pool_k, np.float64)
    V = np.asarray(pool_v, np.float64)
    G, T, _ = q.shape
    m = K.shape[0]
    c = n_compressed
    if m != c + T:
        raise ValueError("pool must hold c + T rows")
    z = np.einsum("gtd,jd->gtj", q, K) * scale
    i = np.arange(T)[:, None]
    j = np.arange(m)[None, :]
    visible = (j < c) | ((j - c) <= i)                      # [T, m]
    z = np.where(visible[None], z, -np.inf)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.where(visible[None], np.exp(z), 0.0)
    P = e / e.sum(axis=-1, keepdims=True)
    O = np.einsum("gtj,jd->gtd", P, V)
    return O, P


# ------------------------------------------ importance and Top-B (关键设计 2)
def importance_scores(P: np.ndarray) -> np.ndarray:
    """s_j = average over the frame's query rows (all G heads x T tokens) of
    the probability paid to key j (R2, R3).  P: [G, T, m] -> s: [m]."""
    P = np.asarray(P, np.float64)
    G, T, m = P.shape
    return P.reshape(G * T, m).sum(axis=0) / (G * T)


def select_top_b(scores: np.ndarray, positions: np.ndarray,
                 budget: int) -> np.ndarray:
    """S̄_n = TopK({s_j}, B): indices of the B candidates ranked first by
    descending score, ties to the lower virtual position (R4).  When the pool
    holds at most B candidates all are kept.  Returned in ascending position."""
    s = np.asarray(scores, np.float64)
    p = np.asarray(positions, np.int64)
    m = s.shape[0]
    if m <= budget:
        keep = np.arange(m)
    else:
        order = np.lexsort((p, -s))        # primary -s, secondary position
        keep = order[:budget]
    return keep[np.argsort(p[keep], kind="stable")]


def select_window(positions: np.ndarray, budget: int) -> np.ndarray:
    """The sliding-window baseline the page compares against (ReKV with a
    window of R frames, compute-matched to B = R*T): keep the B most recent
    candidates instead of the B highest-scoring ones.  Returns the kept
    indices in ascending position."""
    m = positions.shape[0]
    if m <= budget:
        return np.arange(m)
    order = np.argsort(positions, kind="stable")
    return np.sort(order[m - budget:])


# ----------------------------------------------------- dual state (整体框架)
@dataclass
class UnitState:
    """State of one (stream, layer, KV head): compressed C and detailed D."""
    head_dim: int
    comp_k: np.ndarray = None      # [c, d] rotated, storage-rounded
    comp_v: np.ndarray = None      # [c, d]
    comp_pos: np.ndarray = None    # [c] virtual positions
    det_k: list = field(default_factory=list)   # per frame [T, d]
    det_v: list = field(default_factory=list)

    def __post_init__(self):
        d = self.head_dim
        if self.comp_k is None:
            self.comp_k = np.zeros((0, d))
            self.comp_v = np.zeros((0, d))
            self.comp_pos = np.zeros((0,), np.int64)

    @property
    def detailed_k(self) -> np.ndarray:
        return np.concatenate(self.det_k) if self.det_k else np.zeros((0, self.head_dim))

    @property
    def detailed_v(self) -> np.ndarray:
        return np.concatenate(self.det_v) if self.det_v else np.zeros((0, self.head_dim))


def prefill_unit_frame(state: UnitState, q: np.ndarray, k: np.ndarray,
                       v: np.ndarray, n: int, *, budget: int,
                       omega: np.ndarray, scale: float, dtype: str,
                       position_offset: int = 0, policy: str = "topb"):
    """One frame step of one (stream, layer, KV head).

    q: [G, T, d] pre-RoPE queries; k, v: [T, d] pre-RoPE keys and values.
    Steps, in the page's order of dependence:
      1. rotate Q and K at p = offset + nT + i (关键设计 3), round to storage;
      2. attend over [C_{n-1}; frame] (关键设计 1);
      3. score every candidate of U_n and keep Top-B (关键设计 2) -- or, for
         the sliding-window baseline (policy "window"), the B most recent;
      4. C_n = kept rows; D_n = D_{n-1} ++ (K'_n, V_n) (关键设计 1).
    Mutates ``state``; returns (O [G,T,d], info dict).
    """
    T = k.shape[0]
    pos_frame = position_offset + n * T + np.arange(T, dtype=np.int64)
    q_rot = round_to_storage(rope_rotate(q, pos_frame, omega), dtype)
    k_rot = round_to_storage(rope_rotate(k, pos_frame, omega), dtype)
    v = np.asarray(v, np.float64)
    c = state.comp_k.shape[0]
    pool_k = np.concatenate([state.comp_k, k_rot])
    pool_v = np.concatenate([state.comp_v, v])
    pool_pos = np.concatenate([state.comp_pos, pos_frame])
    O, P = attend_frame(q_rot, pool_k, pool_v, c, scale)
    s = importance_scores(P)
    keep = select_window(pool_pos, budget) if policy == "window" else \
        select_top_b(s, pool_pos, budget)
    state.comp_k, state.comp_v, state.comp_pos = pool_k[keep], pool_v[keep], pool_pos[keep]
    state.det_k.append(k_rot)
    state.det_v.append(v)
    info = dict(q_rot=q_rot, k_rot=k_rot, scores=s, pool_pos=pool_pos,
                keep=keep, n_compressed=c, P=P)
    return O, info


# ------------------------------------------ text decode over D (关键设计 1, 3)
def decode_unit_tokens(state: UnitState, q: np.ndarray, k: np.ndarray,
                       v: np.ndarray, first_row: int, *, omega: np.ndarray,
                       scale: float, dtype: str, position_offset: int = 0):
    """Text tokens of one (stream, layer, KV head) after the video.

    The detailed state keeps every frame's K/V for text decoding (关键设计 1);
    text continues the virtual positions with the same static scale
    (关键设计 3).  q: [G, tok, d], k, v: [tok, d] pre-RoPE; the tokens take
    D rows first_row.. and positions offset + first_row + j.  Every earlier D
    row is visible, the new tokens causally (the frame rule of attend_frame
    with the whole of D in the place of the compressed keys).  Appends K', V
    to D; returns (O [G, tok, d], q_rot, k_rot).
    """
    tok = k.shape[0]
    pos = position_offset + first_row + np.arange(tok, dtype=np.int64)
    q_rot = round_to_storage(rope_rotate(q, pos, omega), dtype)
    k_rot = round_to_storage(rope_rotate(k, pos, omega), dtype)
    v = np.asarray(v, np.float64)
    dk, dv = state.detailed_k, state.detailed_v
    assert dk.shape[0] == first_row
    O, _ = attend_frame(q_rot, np.concatenate([dk, k_rot]), np.concatenate([dv, v]),
                        first_row, scale)
    state.det_k.append(k_rot)
    state.det_v.append(v)
    return O, q_rot, k_rot


class StateKVOracle:
    """All (stream, layer, KV head) units of one configuration.

    ``cfg`` needs: streams, layers, q_heads, kv_heads, head_dim, frame_tokens,
    budget, rope_theta, rope_alpha, rope_orig_ctx, dtype; optional
    position_offset."""

    def __init__(self, cfg):
        self.cfg = cfg
        self.omega, self.mscale = rope_frequencies(
            cfg.head_dim, cfg.rope_theta, cfg.rope_alpha, cfg.rope_orig_ctx)
        self.scale = logit_scale(cfg.head_dim, self.mscale)
        self.offset = int(getattr(cfg, "position_offset", 0))
        self.group = cfg.q_heads // cfg.kv_heads
        self.n = 0
        self.text = 0                      # text tokens decoded after the video
        self.units = {(s, l, h): UnitState(cfg.head_dim)
                      for s in range(cfg.streams) for l in range(cfg.layers)
                      for h in range(cfg.kv_heads)}

    def prefill_frame(self, q, k, v, keep_info: bool = False):
        """q: [S][L][Hq][T][d]; k, v: [S][L][Hkv][T][d].  Returns O with q's
        shape (float64) and, if asked, per-unit step info."""
        cfg, G = self.cfg, self.group
        O = np.zeros(np.shape(q), np.float64)
        infos = {}
        for (s, l, h), st in self.units.items():
            o, info = prefill_unit_frame(
                st, q[s][l][h * G:(h + 1) * G], k[s][l][h], v[s][l][h], self.n,
                budget=cfg.budget, omega=self.omega, scale=self.scale,
                dtype=cfg.dtype, position_offset=self.offset,
                policy=getattr(cfg, "select_policy", "topb"))
            O[s, l, h * G:(h + 1) * G] = o
            if keep_info:
                info.pop("P")
                infos[(s, l, h)] = info
        self.n += 1
        return (O, infos) if keep_info else O

    def decode(self, q, k, v):
        """Text tokens after the frames: q [S][L][Hq][tok][d], k, v
        [S][L][Hkv][tok][d].  Returns O with q's shape (float64)."""
        cfg, G = self.cfg, self.group
        O = np.zeros(np.shape(q), np.float64)
        first = self.n * cfg.frame_tokens + self.text
        for (s, l, h), st in self.units.items():
            o, _, _ = decode_unit_tokens(
                st, q[s][l][h * G:(h + 1) * G], k[s][l][h], v[s][l][h], first,
                omega=self.omega, scale=self.scale, dtype=cfg.dtype,
                position_offset=self.offset)
            O[s, l, h * G:(h + 1) * G] = o
        self.text += np.shape(k)[3]
        return O
