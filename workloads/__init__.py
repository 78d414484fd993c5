"""Seeded synthetic inputs for one paged GQA decode step and for decode traces.

This package draws numbers only: sequence lengths, page permutations and fp16 query/key/value contents. It holds
none of the attention arithmetic, so both the fp64 oracle (``oracle/``) and the CUDA path
(``serving_paged_gqa_gb300``) can take their inputs from it without sharing any computation.
"""

from .traces import (  # noqa: F401
    CONFIGS,
    D,
    HKV,
    HQ,
    PS,
    Trace,
    make_trace,
    normal_fp16,
    rng_for,
    zipf_lengths,
)
