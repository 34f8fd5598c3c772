"""Seeded synthetic workloads for the CONF-KV decode-step cache manager.

This package only draws random inputs (prefill K/V, per-step queries, new K/V
and logits) and describes the workload shapes.  It holds none of the method's
arithmetic, so both the CUDA path and the CPU oracle may use it.
"""
from .gen import (  # noqa: F401
    Workload,
    WORKLOADS,
    get_workload,
    heavy_positions,
    needle_position,
    prefill_unit,
    prefill_batch,
    prefill_batch_fast,
    step_unit,
    step_logits,
    step_pool,
    step_pool_fast,
)
