"""bench.py's reference arm and CPU baseline, run on the host with a tiny shape.

The reference arm times the CPU oracle (there is no other reference
implementation): its JSON line must carry the contract's keys, report the
measured time of what each step ran as ms_per_step, and state the scaling to
a whole frame separately."""

import argparse
import io
import json
import contextlib

import bench
from synth import SHAPES


def _tiny():
    # tiny_f32 scaled to a few layers so the extrapolation is visible
    return SHAPES["tiny_f32"].with_(layers=3)


def test_reference_arm_line():
    sh = _tiny()
    args = argparse.Namespace(steps=3, warmup=1, gpus=1)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, sh)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "dtype", "config", "cpu_baseline", "e2e", "extrapolation"):
        assert key in line, key
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == bench.UNIT and line["steps"] == 3
    ex = line["extrapolation"]
    assert ex["layers_timed_per_step"] == 1 and ex["layers_per_frame"] == 3
    # value (frames/s of every layer) follows from the measured step time
    per_frame_ms = line["ms_per_step"] * ex["layers_per_frame"] / ex["layers_timed_per_step"]
    assert abs(line["value"] - 1000.0 / per_frame_ms) <= 1e-9 * line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1


def test_cpu_baseline_samples_consecutive_steady_frames():
    sh = _tiny()
    smp = bench._OracleSample(sh, layers=1)
    n0 = smp.n
    assert n0 == sh.budget // sh.frame_tokens            # the first full-state frame
    t = [smp.frame() for _ in range(3)]
    assert smp.n == n0 + 3 and all(x > 0 for x in t)
    # the state evolved by the oracle's own selection: still B rows, unique positions
    for st in smp.states:
        assert st.comp_pos.shape[0] == sh.budget
        assert len(set(st.comp_pos.tolist())) == sh.budget
    cb = bench.cpu_baseline(sh, frames=2, layers=1)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and "consecutive steady-state" in cb["sample"]


def test_decode_text_rows_cover_the_decode_leg():
    """The handle's extra detailed-state frames hold every text token the
    decode leg writes (3 warm-up steps and the timed ones), and --budget
    full never evicts with that many frames."""
    sh = _tiny()
    for steps, tokens in ((20, 1), (30, 8), (5, 16), (0, 1)):
        args = argparse.Namespace(decode_steps=steps, decode_tokens=tokens)
        extra = bench.decode_text_frames(args, sh)
        assert extra >= 1
        assert extra * sh.frame_tokens >= (3 + steps) * tokens
        assert (extra - 1) * sh.frame_tokens < max(1, (3 + steps) * tokens)
