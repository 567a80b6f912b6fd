"""Benchmark: StateKV streaming prefill throughput on GB300.

Metric: video frames/s through streaming prefill, all layers, B=4096, T=256,
on the InternVL3-2B attention geometry (28 layers, 12 query / 2 KV heads,
head_dim 128, 512 frames per video, static YaRN alpha=4), with the fraction
of the bf16 tensor-core peak reached by the attention kernel.

One step = one whole video: the handle is reset and all 512 frames stream
through every layer (the fill phase included, exactly as a user runs it).
Inputs: a ring of 16 distinct seeded synthetic frames resident in HBM, frame
n uses ring slot n % 16; the per-frame working set (compressed state of all
layers ~117 MB, Q/O ~44 MB, detailed-state append, scratch) exceeds L2.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
N > 1 runs under torchrun, one rank per GPU, each rank streaming its own
video (independent streams; no collective on the data path).
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "video frames/sec through streaming prefill (all layers, B=4096,T=256); % bf16 TC peak"
UNIT = "frames/s"
WORKLOAD = "internvl3_2b_stack"
RING = 16
E_RING = 32        # host frames per batched host call in the e2e leg


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm=j["hbm_gbs"], tc=j["bf16_tflops"], tc_sus=j["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, tc=1900.0, tc_sus=1700.0, src="fallback")


def _dist():
    """Replicas: one process per GPU (torchrun env).  Each rank streams its own
    independent videos; the only collectives are the barriers around the
    timed region and the max of the ranks' times.  NCCL on GPUs, gloo on a
    host without them (the multi-process tests)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return dist, int(os.environ["RANK"]), ws, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def max_over_ranks(x: float, dist, device="cpu") -> float:
    """The slowest rank's value (the job's time); x itself on one process."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(sh, rank: int) -> int:
    """Each replica's synthetic videos: a seed of their own."""
    return sh.seed + rank


class ClockSampler:
    """nvidia-smi clocks/throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def _traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f).get(kernel)
    if not j:
        return None
    src = os.path.join(ROOT, "kv_cache_compression_frame_gb300", "csrc", j["source"])
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    return j["bytes_per_launch"] if h == j["source_sha"] else None


# --------------------------------------------------------------- CPU oracle
class _OracleSample:
    """The oracle on `layers` layers (all their KV heads) of a stream in steady
    state: the compressed state starts full (B synthetic rows at positions
    0..B-1, rotated and storage-rounded like real keys; built untimed), and
    each frame() call runs the next frame n = B/T, B/T + 1, ... through the
    oracle's own step, so the state evolves by its own selection."""

    def __init__(self, sh, layers: int, seed: int = 1):
        import numpy as np
        import oracle.statekv_oracle as orc
        from synth import FrameSource
        self.orc, self.sh, self.layers = orc, sh, layers
        self.src = FrameSource(sh)
        self.omega, ms = orc.rope_frequencies(sh.head_dim, sh.rope_theta, sh.rope_alpha,
                                              sh.rope_orig_ctx)
        self.scale = orc.logit_scale(sh.head_dim, ms)
        self.n = sh.budget // sh.frame_tokens       # first frame with a full state
        rng = np.random.default_rng(seed)
        B, d = sh.budget, sh.head_dim
        self.states = []
        for _ in range(layers * sh.kv_heads):
            st = orc.UnitState(d)
            pos = np.arange(B, dtype=np.int64)
            st.comp_k = orc.round_to_storage(orc.rope_rotate(rng.standard_normal((B, d)), pos,
                                                             self.omega), sh.dtype)
            st.comp_v = orc.round_to_storage(rng.standard_normal((B, d)), sh.dtype)
            st.comp_pos = pos
            self.states.append(st)

    def frame(self) -> float:
        """Seconds of oracle work for the next frame of the sampled layers
        (input generation untimed)."""
        sh, G = self.sh, self.sh.group
        inputs = [self.src.layer_frame(0, l, self.n) for l in range(self.layers)]
        t0 = time.perf_counter()
        i = 0
        for l in range(self.layers):
            q, k, v = inputs[l]
            for hk in range(sh.kv_heads):
                self.orc.prefill_unit_frame(self.states[i], q[hk * G:(hk + 1) * G], k[hk], v[hk],
                                            self.n, budget=sh.budget, omega=self.omega,
                                            scale=self.scale, dtype=sh.dtype)
                i += 1
        self.n += 1
        return time.perf_counter() - t0


def cpu_baseline(sh, frames: int = 8, layers: int = 1) -> dict:
    """The oracle as it stands on 8 consecutive steady-state frames of one
    layer (all its KV heads), scaled to every layer of the workload."""
    smp = _OracleSample(sh, layers)
    n0 = smp.n
    secs = [smp.frame() for _ in range(frames)]
    per_frame = sum(secs) / frames * sh.layers / layers
    return {"value": 1.0 / per_frame, "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "s_per_frame": per_frame,
            "sample": f"fp64 NumPy oracle, {frames} consecutive steady-state frames "
                      f"(n = {n0}..{n0 + frames - 1}, c = B = {sh.budget}) of {layers} of "
                      f"{sh.layers} layers ({layers * sh.kv_heads} of {sh.units} units), "
                      f"{sum(secs):.1f} s, scaled x{sh.layers}/{layers}"}


def run_reference(args, sh):
    # the oracle on the host cores: rank 0 alone under torchrun
    if int(os.environ.get("RANK", "0")) != 0:
        return
    layers = 1
    smp = _OracleSample(sh, layers)
    for _ in range(args.warmup):
        smp.frame()
    n0 = smp.n
    times = [smp.frame() for _ in range(args.steps)]
    timed = sum(times)
    per_frame = timed / args.steps * sh.layers / layers     # all layers of one frame
    value = 1.0 / per_frame
    cores = len(os.sched_getaffinity(0))
    sample = (f"each step: the next steady-state frame (n = {n0}..{n0 + args.steps - 1}, c = B) "
              f"of {layers} of {sh.layers} layers ({layers * sh.kv_heads} of {sh.units} units), "
              f"the state continuing across steps; frames/s scaled x{sh.layers}/{layers}")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        # the measured time of what each step ran (one layer of one frame)
        "ms_per_step": 1000.0 * timed / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": sh.name, "layers": sh.layers, "q_heads": sh.q_heads,
                   "kv_heads": sh.kv_heads, "head_dim": sh.head_dim, "T": sh.frame_tokens,
                   "B": sh.budget, "step": f"one steady-state frame of {layers} layer(s)"},
        "extrapolation": {"layers_timed_per_step": layers, "layers_per_frame": sh.layers,
                          "value_scale": layers / sh.layers,
                          "ms_per_frame_all_layers": 1000.0 * per_frame},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------- GPU
def decode_text_frames(args, sh) -> int:
    """Whole frames of detailed-state rows the decode leg's text needs (its 3
    warm-up steps and the timed ones)."""
    return max(1, -(-(3 + args.decode_steps) * args.decode_tokens // sh.frame_tokens))


def run_gpu(args, sh):
    import torch
    from kv_cache_compression_frame_gb300 import StateKV, StateKVConfig
    from synth import FrameSource

    dist, rank, ws, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = _peaks()
    frames = args.frames or sh.frames
    src = FrameSource(sh, seed=replica_seed(sh, rank))
    ring = [src.frame(i) for i in range(RING)]
    dq = [torch.from_numpy(r[0]).to(torch.bfloat16).to(dev) for r in ring]
    dk = [torch.from_numpy(r[1]).to(torch.bfloat16).to(dev) for r in ring]
    dv = [torch.from_numpy(r[2]).to(torch.bfloat16).to(dev) for r in ring]
    o = torch.empty_like(dq[0])
    # extra detailed-state rows for the text of the decode leg (3 warm-up
    # steps and the timed ones), in whole frames
    text_frames = decode_text_frames(args, sh)
    h = StateKV(StateKVConfig.from_shape(sh, max_frames=frames + text_frames,
                                         select_policy=args.policy), device=local)
    stream = torch.cuda.current_stream(dev)

    def one_video():
        h.reset()
        for n in range(frames):
            r = n % RING
            h.prefill_frame(dq[r], dk[r], dv[r], o, stream)

    # the timed videos: the attention kernel of one frame in SAMPLE is
    # bracketed by CUDA events (the roofline's duration, measured live); an
    # event between two launches ends their overlap (programmatic dependent
    # launch), so the other frames run unbracketed
    attn_bit = 1 << N_KERNEL_ATTENTION
    sampled = [n for n in range(frames) if n % SAMPLE == SAMPLE - 1]

    def one_video_timed():
        h.reset()
        for n in range(frames):
            r = n % RING
            h.profile_mask(attn_bit if n % SAMPLE == SAMPLE - 1 else 0)
            h.prefill_frame(dq[r], dk[r], dv[r], o, stream)

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        one_video()
    h.check_device_status()

    # timed region: K whole videos, the attention kernel of 1 frame in SAMPLE
    # bracketed by events (one_video_timed)
    clocks = ClockSampler(local)
    h.profile_mask(0)
    h.profile_enable(True)
    torch.cuda.synchronize()
    barrier()
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        one_video_timed()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1)
    prof_attn = h.profile_read()["attention"]
    h.profile_enable(False)
    h.check_device_status()
    ms = max_over_ranks(ms, dist, dev)
    total_frames = args.steps * frames * ws
    value = total_frames / (ms / 1000.0)

    # per-frame latency vs n and every kernel's time (one extra, untimed
    # video; the events between launches serialise them)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(frames + 1)]
    h.reset()
    h.profile_kernels()
    h.profile_enable(True)
    evs[0].record(stream)
    for n in range(frames):
        r = n % RING
        h.prefill_frame(dq[r], dk[r], dv[r], o, stream)
        evs[n + 1].record(stream)
    torch.cuda.synchronize()
    prof = h.profile_read()
    h.profile_enable(False)
    per_frame = [evs[i].elapsed_time(evs[i + 1]) * 1000.0 for i in range(frames)]
    n_full = sh.budget // sh.frame_tokens
    steady = per_frame[n_full:]
    q1 = len(steady) // 4
    flat = (statistics.median(steady[-q1:]) / statistics.median(steady[:q1])) if q1 else None

    # each kernel's time per frame over a video (every launch bracketed, the
    # times read after every frame), medians per window of frames: where the
    # per-frame time moves, which kernel moves (untimed)
    windows = None
    if args.kernel_windows > 0:
        names = ("rope", "attention", "select")
        h.reset()
        h.profile_kernels()
        h.profile_enable(True)
        prev = {k: 0.0 for k in names}
        rows = []
        for n in range(frames):
            r = n % RING
            h.prefill_frame(dq[r], dk[r], dv[r], o, stream)
            p = h.profile_read()
            rows.append({k: (p[k][0] - prev[k]) * 1000.0 for k in names})
            prev = {k: p[k][0] for k in names}
        h.profile_enable(False)
        w = args.kernel_windows
        windows = [{"n0": n0, **{k: round(statistics.median([x[k] for x in rows[n0:n0 + w]]), 2)
                                 for k in names}}
                   for n0 in range(0, frames, w)]

    # e2e: host buffers through the C ABI, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        # a pinned host ring of E_RING frames (the device ring's frames
        # repeated), streamed E_RING frames per call: inside a call the
        # copies of frames i+1 (in) and i-1 (out) overlap the step of frame i
        def pinned(idx):
            t = torch.empty((E_RING,) + tuple(ring[0][idx].shape), dtype=torch.bfloat16).pin_memory()
            for i in range(E_RING):
                t[i].copy_(torch.from_numpy(ring[i % RING][idx]))
            return t
        hq, hk, hv = pinned(0), pinned(1), pinned(2)
        ho = torch.empty(hq.shape, dtype=torch.bfloat16).pin_memory()

        def one_video_host():
            h.reset()
            for n0 in range(0, frames, E_RING):
                c = min(E_RING, frames - n0)
                h.prefill_frames_host(hq[:c], hk[:c], hv[:c], ho[:c], stream)

        one_video_host()
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            one_video_host()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems = e0.elapsed_time(e1)
        ems = max_over_ranks(ems, dist, dev)
        in_b = (hq[0].numel() + hk[0].numel() + hv[0].numel()) * 2 * frames
        out_b = ho[0].numel() * 2 * frames
        e2e = {"value": args.e2e_steps * frames * ws / (ems / 1000.0), "unit": UNIT,
               "h2d_bytes_per_step": in_b, "d2h_bytes_per_step": out_b,
               "steps": args.e2e_steps}

    # decode leg: after a whole video, single text tokens over the detailed
    # state D (every frame's K/V); HBM-bound, algorithmic bytes = K and V of
    # every D row read once per step
    dec = None
    if not args.no_decode and sh.head_dim == 128:
        h.reset()
        for n in range(frames):
            r = n % RING
            h.prefill_frame(dq[r], dk[r], dv[r], o, stream)
        g = torch.Generator(device="cpu").manual_seed(5)
        tok = args.decode_tokens
        tq = torch.randn((sh.streams, sh.layers, sh.q_heads, tok, sh.head_dim), generator=g).to(torch.bfloat16).to(dev)
        tk = torch.randn((sh.streams, sh.layers, sh.kv_heads, tok, sh.head_dim), generator=g).to(torch.bfloat16).to(dev)
        tv = torch.randn((sh.streams, sh.layers, sh.kv_heads, tok, sh.head_dim), generator=g).to(torch.bfloat16).to(dev)
        to = torch.empty_like(tq)
        for _ in range(3):
            h.decode(tq, tk, tv, to, stream)
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        k0 = frames * sh.frame_tokens + h.text_tokens
        n_dec = args.decode_steps
        torch.cuda.synchronize()
        d0.record(stream)
        for _ in range(n_dec):
            h.decode(tq, tk, tv, to, stream)
        d1.record(stream)
        torch.cuda.synchronize()
        h.check_device_status()
        dms = d0.elapsed_time(d1) / n_dec
        units = sh.streams * sh.layers * sh.kv_heads
        rows = k0 + tok * (n_dec + 1) / 2.0                 # mean D rows read per step
        dbytes = units * rows * sh.head_dim * 2 * 2
        dec = {"tokens_per_s": tok * 1000.0 / dms, "us_per_step": dms * 1000.0,
               "tokens_per_step": tok,
               "d_rows_per_kv_head": int(k0), "steps": n_dec,
               "roofline": {"bound": "hbm", "achieved": dbytes / (dms / 1000.0) / 1e9,
                            "peak": peaks["hbm"], "unit": "GB/s",
                            "frac": dbytes / (dms / 1000.0) / 1e9 / peaks["hbm"],
                            "bytes_per_step": dbytes,
                            "kernel": "decode_kernel + decode_combine_kernel"}}

    # roofline of the dominant kernel (attention) over the timed region: the
    # sampled launches' flops over their bracketed durations
    flops_timed = args.steps * sum(sh.attention_flops(n) for n in sampled)
    attn_ms, attn_n = prof_attn
    achieved = flops_timed / (attn_ms / 1000.0) / 1e12
    step_flops = sum(sh.attention_flops(n) for n in range(frames))
    q_bytes = sh.streams * sh.layers * sh.q_heads * sh.frame_tokens * sh.head_dim * 2
    kv_bytes = sh.streams * sh.layers * sh.kv_heads * sh.frame_tokens * sh.head_dim * 2
    rope_bytes = 2 * q_bytes + 6 * kv_bytes
    # select: the column partials read, scores and positions written, the
    # live positions read, and the K/V rows moved by slot reuse (counted on
    # the untimed video's last frame: its surviving frame rows)
    T, B = sh.frame_tokens, sh.budget
    m = min(B, (frames - 1) * T) + T
    n_rt = -(-sh.group * T // 128)
    moved = 0
    for l in range(sh.layers):
        for s_ in range(sh.streams):
            _, _, p, c = h.compressed(s_, l)
            moved += int((p[:, :c] >= (frames - 1) * T).sum().item())
    sel_bytes = sh.units * (n_rt * m * 4 + 2 * m * 4 + min(B, (frames - 1) * T) * 4) \
        + moved * 2 * 2 * sh.head_dim * 2
    kernels = {}
    for name, (kms, cnt) in prof.items():
        ent = {"launches_untimed_video": cnt, "ms_per_launch": kms / max(cnt, 1),
               "share": kms / max(sum(x[0] for x in prof.values()), 1e-9)}
        if name == "rope":
            ent["gbs"] = rope_bytes / (kms / max(cnt, 1) / 1000.0) / 1e9
            ent["algorithmic_bytes_per_launch"] = rope_bytes
        if name == "select" and cnt:
            ent["gbs"] = sel_bytes / (kms / cnt / 1000.0) / 1e9
            ent["algorithmic_bytes_per_launch"] = sel_bytes
            ent["rows_moved_last_frame"] = moved
        if "gbs" in ent:
            ent["frac_of_hbm"] = ent["gbs"] / peaks["hbm"]
        kernels[name] = ent

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": sh.name, "layers": sh.layers, "q_heads": sh.q_heads,
                       "kv_heads": sh.kv_heads, "head_dim": sh.head_dim,
                       "T": sh.frame_tokens, "B": sh.budget, "frames_per_step": frames,
                       "policy": args.policy,
                       "rope_alpha": sh.rope_alpha, "parallelism": f"replicas x{ws}",
                       "l2": "inputs larger than L2 (16-frame ring, 117 MB compressed state)"},
            "tflops_algorithmic": step_flops * args.steps / (ms / 1000.0) / 1e12,
            # attention pairs of one video relative to full self-attention
            "attention_pairs_vs_full_sa": step_flops / sum(
                dataclasses.replace(sh, budget=1 << 40).attention_flops(n) for n in range(frames)),
            "tflops_executed": 1.5 * step_flops * args.steps / (ms / 1000.0) / 1e12,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["tc_sus"],
                         "unit": "TFLOP/s", "frac": achieved / peaks["tc_sus"],
                         "traffic": _traffic("attention"),
                         "kernel": "attn_tc_kernel<128>",
                         "peak_kind": f"bf16 sustained ({peaks['src']})",
                         "flops_per_launch_steady": sh.attention_flops(n_full),
                         "ms_per_launch": attn_ms / max(attn_n, 1),
                         "launches_timed": attn_n,
                         "sampling": f"attention bracketed by CUDA events on 1 frame in {SAMPLE} "
                                     f"(frames n % {SAMPLE} == {SAMPLE - 1}) of every timed video; "
                                     "events between launches end their overlap"},
            "kernels": kernels,
            "per_frame_us": {"fill_mean": statistics.mean(per_frame[:n_full]) if n_full else None,
                             "steady_median": statistics.median(steady) if steady else None,
                             "steady_p99": sorted(steady)[int(0.99 * (len(steady) - 1))] if steady else None,
                             "last_quarter_over_first_quarter": flat},
            "e2e": e2e,
            "decode": dec,
            **({"kernel_us_per_window": {"frames_per_window": args.kernel_windows,
                                         "windows": windows}} if windows else {}),
            # RoPE, attention and selection per frame (the RoPE table is made
            # once, at create)
            "gpu_launches": LAUNCHES_PER_FRAME * frames * args.steps,
            "clocks": clk,
        }
        if not args.no_cpu_baseline and ws == 1:
            line["cpu_baseline"] = cpu_baseline(sh)
        print(json.dumps(line), flush=True)
    h.close()
    if dist is not None:
        dist.destroy_process_group()


LAUNCHES_PER_FRAME = 3
SAMPLE = 8                 # 1 frame in SAMPLE has its attention kernel bracketed by events
N_KERNEL_ATTENTION = 2     # STATEKV_KERNEL_ATTENTION


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--frames", type=int, default=0, help="frames per video (default: N of the workload)")
    ap.add_argument("--e2e-steps", type=int, default=2)
    ap.add_argument("--decode-steps", type=int, default=20)
    ap.add_argument("--decode-tokens", type=int, default=1)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel-windows", type=int, default=0,
                    help="also run one video with every frame synchronised and report each "
                         "kernel's median device time per window of this many frames")
    ap.add_argument("--policy", default="topb", choices=["topb", "window"],
                    help="selection: Top-B by score (the method) or the B most recent tokens "
                         "(the sliding-window baseline)")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the workload's layer count (1 = one layer per launch, "
                         "the shape of a model whose layers feed each other)")
    ap.add_argument("--budget", default="",
                    help="override B; 'full' = full self-attention (B covers every frame)")
    args = ap.parse_args()
    from synth import SHAPES
    sh = SHAPES[args.workload]
    if args.layers:
        sh = dataclasses.replace(sh, layers=args.layers,
                                 name=f"{sh.name}_{args.layers}layer" if args.layers != sh.layers
                                 else sh.name)
    if args.budget:
        frames = args.frames or sh.frames
        b = ((frames + decode_text_frames(args, sh)) * sh.frame_tokens if args.budget == "full"
             else int(args.budget))
        sh = dataclasses.replace(sh, budget=b)
    if args.impl == "reference":
        run_reference(args, sh)
    else:
        import __graft_entry__
        __graft_entry__.build()
        run_gpu(args, sh)


if __name__ == "__main__":
    main()
