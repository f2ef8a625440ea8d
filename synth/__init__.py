"""Seeded synthetic inputs for the packed verify + OPD-loss pass.

This package builds the logits, draft tokens and per-request offsets that both
the CUDA path and the CPU oracle consume.  It holds none of the method's
arithmetic (no softmax, no divergence, no acceptance rule): only random draws,
rounding to the storage dtype, and the planted structure each workload asks for.
"""

from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_workload,
    materialize,
)
