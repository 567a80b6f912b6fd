"""The allocation-free entry point, statekv_attend_scores_static.

It serves callers that cannot allocate device memory: their memory belongs to
another allocator (an inference server's pool, a framework hosting the library
as a plugin), or they cannot afford the device-wide synchronisation that
cudaMalloc/cudaFree may cause.  Its only scratch is a fixed __device__ array
inside the library.  Each case calls it through the C ABI on two frames in a
row and checks its O and scores against the handle-based path
(statekv_prefill_frame) on the same inputs and against the CPU oracle
(teacher-forced on the same rotated queries and pool), with the parity
tolerances used everywhere else (O row-relative 2e-2 for bf16, 1e-5 for fp32;
scores 1e-3 relative + 1e-6/m).  The cases cover the tcgen05 path with one
and with three 128-row query tiles per unit (the score finish sums the tiles'
column partials) and the fp32 path (16-row tiles).  It lives in its own file,
collected last.
"""

import math

import numpy as np
import pytest
import torch

import oracle.statekv_oracle as orc
from parity import O_TOL, check_scores, f64, row_rel_err
from synth import FrameSource, WorkloadShape

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from kv_cache_compression_frame_gb300 import build_lib
    build_lib.build()


def _shape(dtype, q_heads, kv_heads, head_dim, T, B):
    return WorkloadShape(name="noalloc", streams=1, layers=2, q_heads=q_heads,
                         kv_heads=kv_heads, head_dim=head_dim, frame_tokens=T, budget=B,
                         frames=6, rope_theta=1e6, rope_alpha=1.0, rope_orig_ctx=0,
                         dtype=dtype, sinks_per_frame=2, sink_gain=3.0, sink_drift=0.05,
                         key_scale_sigma=0.0)


@pytest.mark.parametrize("dtype,q_heads,kv_heads,head_dim,T,B", [
    ("bf16", 4, 2, 128, 64, 192),     # G*T = 128: one query tile per unit
    ("bf16", 12, 2, 64, 64, 160),     # G*T = 384: three tiles summed by the score finish
    ("f32", 4, 2, 64, 16, 40),        # fp32 path: G*T = 32, two 16-row tiles
])
def test_static_scratch_entry_matches_handle_path_and_oracle(dtype, q_heads, kv_heads,
                                                             head_dim, T, B):
    from kv_cache_compression_frame_gb300 import StateKV, StateKVConfig
    from kv_cache_compression_frame_gb300 import _native as N
    lib = N.load()
    sh = _shape(dtype, q_heads, kv_heads, head_dim, T, B)
    src = FrameSource(sh)
    h = StateKV(StateKVConfig.from_shape(sh))
    dev = h.device
    tdt = h.torch_dtype
    G, d, U = sh.group, sh.head_dim, sh.units
    scale = 1.0 / math.sqrt(d)                  # alpha = 1: plain 1/sqrt(d)
    stream = torch.cuda.current_stream(dev)
    # a stale nonzero status word: the call must clear it itself
    status = torch.tensor([5, 1, 2, 3], dtype=torch.int32, device=dev)
    for n in range(3):                          # fill the compressed state
        h.prefill_frame(*(torch.from_numpy(a).to(tdt).to(dev) for a in src.frame(n)))
    for call, n in enumerate((3, 4)):           # two calls in a row
        c = h.compressed(0, 0)[3]
        pre = [h.compressed(0, l) for l in range(sh.layers)]
        pre_k = [p[0][:, :c].clone() for p in pre]
        pre_v = [p[1][:, :c].clone() for p in pre]
        q, k, v = (torch.from_numpy(a).to(tdt).to(dev) for a in src.frame(n))
        o_ref = h.prefill_frame(q, k, v)
        h.check_device_status()
        q_rot = h.rotated_query().clone()       # [1][L][Hq][T][d] = [U][G*T][d]
        pk, pv = [], []
        for l in range(sh.layers):
            dk, dv, _ = h.detailed(0, l)
            pk.append(torch.cat([pre_k[l], dk[:, n * T:(n + 1) * T]], dim=1))
            pv.append(torch.cat([pre_v[l], dv[:, n * T:(n + 1) * T]], dim=1))
        pool_k = torch.stack(pk).reshape(U, c + T, d).contiguous()
        pool_v = torch.stack(pv).reshape(U, c + T, d).contiguous()
        o = torch.empty_like(q_rot)
        scores = torch.empty((U, c + T), dtype=torch.float32, device=dev)
        st = lib.statekv_attend_scores_static(
            q_rot.data_ptr(), pool_k.data_ptr(), pool_v.data_ptr(), U, G, T, d, c + T, c,
            scale, N.BF16 if dtype == "bf16" else N.F32, o.data_ptr(), scores.data_ptr(),
            status.data_ptr(), stream.cuda_stream)
        assert st == N.OK, N.status_string(st)
        torch.cuda.synchronize()
        assert status.cpu().tolist() == [0, 0, 0, 0], f"call {call}: device status {status.cpu().tolist()}"
        tol = O_TOL[dtype]
        err = row_rel_err(f64(o), f64(o_ref))
        assert err <= tol, f"call {call}: O vs handle path, row-relative error {err:.3g}"
        q_units = f64(q_rot.reshape(U, G, T, d))
        o_units = f64(o.reshape(U, G, T, d))
        for l in range(sh.layers):
            s_ref, _, m = h.scores(0, l)
            for hk in range(sh.kv_heads):
                u = l * sh.kv_heads + hk
                what = f"call {call} layer {l} head {hk}"
                check_scores(f64(scores[u]), f64(s_ref[hk, :m]), f"{what} vs handle path")
                O_or, P = orc.attend_frame(q_units[u], f64(pool_k[u]), f64(pool_v[u]), c, scale)
                e = row_rel_err(o_units[u], O_or)
                assert e <= tol, f"{what}: O vs oracle, row-relative error {e:.3g}"
                check_scores(f64(scores[u]), orc.importance_scores(P), f"{what} vs oracle")
        status.fill_(7)                         # stale again for the second call
        torch.cuda.synchronize()
    h.close()


def test_static_scratch_entry_rejects_bad_requests():
    from kv_cache_compression_frame_gb300 import _native as N
    lib = N.load()
    buf = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    p = buf.data_ptr()
    sc = torch.zeros(16, dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    # 4096 units x 12 query tiles x 4352 padded rows x 4 B >> 16 MiB
    st = lib.statekv_attend_scores_static(p, p, p, 4096, 6, 256, 128, 4352, 4096, 0.1,
                                          N.BF16, p, sc.data_ptr(), status.data_ptr(), None)
    assert st == N.E_CAPACITY
    st = lib.statekv_attend_scores_static(p, p, p, 1, 1, 64, 96, 64, 0, 0.1, N.BF16, p,
                                          sc.data_ptr(), status.data_ptr(), None)
    assert st == N.E_UNSUPPORTED
    # the status word is required: without it a timed-out call could not be seen
    st = lib.statekv_attend_scores_static(p, p, p, 1, 1, 64, 128, 64, 0, 0.1, N.BF16, p,
                                          sc.data_ptr(), None, None)
    assert st == N.E_INVALID_ARG
    assert np.all(status.cpu().numpy() == 0)
