"""fp64 CPU oracle for one paged GQA decode step. TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline / reference arm may import this
package. It shares no code with the CUDA path and never imports it.
"""

from .oracle import (  # noqa: F401
    attention,
    build,
    half_to_double,
    launch_counts,
    merge,
    merge_state_bytes,
    num_threads,
    split_states,
    worklist,
)
