"""Seeded synthetic inputs for absorbed-MLA decode.

This package only draws random numbers and shapes them like the workloads of
the pages (V2-Lite and DeepSeek-V3 MLA layer shapes).  It holds none of the
attention arithmetic: both the CUDA path (through the tests and the bench)
and the CPU oracle take their inputs from here, and nothing here imports
either of them.
"""

from .workloads import (  # noqa: F401
    HIDDEN,
    WORKLOADS,
    Workload,
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    gen_hidden,
    gen_out_weights,
    gen_project_weights,
    gen_queries,
    gen_queries_multi,
    gen_seqlens,
    gen_sequence,
    gen_weights,
    get_workload,
    make_page_table,
    rope_interleaved,
)
