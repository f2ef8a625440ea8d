"""CPU oracle for the packed verify + OPD-loss pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path (the
CUDA library and its Python binding) never calls it and shares no code with it.

Two implementations of the same definitions, both float64: ``oracle.opd`` (numpy,
one row at a time; the parity tests' reference) and ``oracle.cpp``, the plain C++
loops of ``opd_ref.cpp`` (pinned on its own and checked element by element against
``oracle.opd``; the CPU baseline the benchmark times).
"""

from .opd import (  # noqa: F401
    acceptance_rate,
    first_argmax,
    greedy_accept,
    hard_label_ce,
    log_sum_exp,
    opd_loss_bwd,
    opd_loss_fwd,
    row_forward,
    row_grad,
    verify_packed,
)
