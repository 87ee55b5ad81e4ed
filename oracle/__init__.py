"""CPU oracle for per-window int8 recurrent-state decode.

TEST INFRASTRUCTURE, NOT THE PRODUCT. A plain, slow C implementation of the
method's steps (append A0-A7, fold F0-F6, init-fold) in one fixed fp32
evaluation order, used to check the CUDA path. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import it.
It shares no code with the CUDA path.

Every function is pinned by the CPU tests in ``tests/test_oracle_pins.py``.
"""
from .oracle import FoldDiag, OracleState, dot, fit, fp32_run, lib, sum_abs  # noqa: F401
