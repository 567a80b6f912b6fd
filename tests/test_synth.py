"""The seeded input generator: reproducible frame by frame, storage-exact."""

import numpy as np
import torch

from synth import SHAPES, FrameSource


def test_frames_regenerate_alone_and_are_storage_exact():
    sh = SHAPES["internvl3_1b_layer"].with_(frames=4)
    a = FrameSource(sh)
    q0, k0, v0 = a.frame(0)
    q3, k3, v3 = a.frame(3)
    b = FrameSource(sh)
    q3b, k3b, v3b = b.frame(3)          # without generating 0..2 first
    np.testing.assert_array_equal(q3, q3b)
    np.testing.assert_array_equal(k3, k3b)
    np.testing.assert_array_equal(v3, v3b)
    assert not np.array_equal(k0, k3)
    for x in (q3, k3, v3):
        rt = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
        np.testing.assert_array_equal(x, rt)
    assert q3.shape == (1, 1, 14, 256, 64) and k3.shape == (1, 1, 2, 256, 64)


def test_sinks_are_planted_along_a_drifting_direction():
    sh = SHAPES["internvl3_1b_layer"]
    src = FrameSource(sh)
    u4 = src._sink_dir(0, 0, 0, 4)
    u5 = src._sink_dir(0, 0, 0, 5)
    assert abs(np.linalg.norm(u5) - 1) < 1e-12
    # one step of 0.05*N(0,I) in 64 dims turns u by about 0.4 rad
    assert 0.85 < float(u4 @ u5) < 1.0
    _, k, _ = src.frame(5)
    proj = k[0, 0, 0] @ u5
    # 4 planted rows stand out by about +3 along u
    assert (proj > 2.0).sum() >= 3


def test_f32_shape_and_key_scale():
    src = FrameSource(SHAPES["tiny_f32"])
    q, k, v = src.frame(0)
    assert q.dtype == np.float32 and q.shape == (1, 1, 2, 16, 64)
    qs = FrameSource(SHAPES["qwen3vl_2b_stack"].with_(layers=1))
    _, k, _ = qs.frame(0)
    std = k[0, 0].reshape(8, -1, 128).std(axis=1)
    assert std.max() / std.min() > 3            # heavy-tailed channel scales
