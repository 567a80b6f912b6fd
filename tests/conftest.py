import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped, not failed, on a machine without a GPU; the
    # "-m gpu" run on a GPU machine executes them.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    _parity_summary(terminalreporter)
    _overlap_summary(terminalreporter)


def _parity_summary(tr):
    # worst parity errors of every checked GPU step (none on a CPU-only run)
    try:
        from parity import STEP_REPORT
    except Exception:  # pragma: no cover
        return
    if not STEP_REPORT:
        return
    tr.write_sep("-", "GPU parity: worst errors per checked step")
    tr.write_line("test | workload | frame | units | O row-rel | score err / tol | "
                  "near-tie swaps | Q' max ulp beyond the fp32 bound | Q' fraction differing")
    for r in STEP_REPORT:
        tr.write_line(f"{r['test']} | {r['workload']} | {r['frame']} | {r['units']} | "
                      f"{r['o_row_rel']:.3g} | {r['score_err_x_tol']:.3g} | "
                      f"{r['near_tie_swaps']} | {r['rope_q_max_ulp']} | "
                      f"{(r['rope_q_mismatch'] or 0):.2g}")


def _overlap_summary(tr):
    try:
        from test_gpu_overlap import OVERLAP_REPORT
    except Exception:  # pragma: no cover
        return
    if not OVERLAP_REPORT:
        return
    tr.write_sep("-", "free-running selection overlap |S_gpu ∩ S_oracle| / B")
    for r in OVERLAP_REPORT:
        for l, x in r["per_layer"].items():
            tr.write_line(f"{r['workload']} layer {l}: min {x['min']:.4f} mean {x['mean']:.4f} "
                          f"last frame {x['last_frame_mean']:.4f} (frames {r['first_eviction_frame']}"
                          f"..{r['frames'] - 1})")
