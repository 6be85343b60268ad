"""Seeded synthetic inputs for one continuous-batching attention step over a paged KV cache.

This module is shared by the fp64 oracle (``oracle/``) and by the CUDA path's tests and
benchmark.  It draws random numbers and lays out block tables and slot mappings; it holds none
of the method's arithmetic (no attention, no quantisation, no gather).
"""

from .workloads import (  # noqa: F401
    CONFIG_NAMES,
    Workload,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_config,
    make_workload,
)
