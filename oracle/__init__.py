"""CPU oracle for StateKV streaming prefill -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and ``--impl reference`` arm) may import this package.
The CUDA library never imports it and it imports nothing from the library.
"""

from .statekv_oracle import (  # noqa: F401
    rope_frequencies, rope_rotate, bf16_round, round_to_storage,
    logit_scale, attend_frame, importance_scores, select_top_b,
    UnitState, prefill_unit_frame, StateKVOracle,
)
