"""Paged grouped-query decode attention for GB300 (sm_103a).

One decode step of attention over a block-table FP16 KV cache with three schedules (single-pass, rectangular
sequence split, compact device-built workqueue), a log-sum-exp merge, a device worklist builder and a host
roofline cost-model planner, all in libpkv.so (C ABI: include/pkv.h). This package is its Python binding.
"""

from ._lib import (EXPORTS, LIB_PATH, PKV_MAX_BATCH, PKV_MAX_ROWS_IN_DECODE, PKV_PLAN_INPUTS_AFTER_PREV,  # noqa: F401
                   PKV_PLAN_OVERLAP_PREV,
                   PKV_SESSION_GRAPHS, PKV_STATIC_SCRATCH_BYTES,
                   PKV_STATUS_BAD_LEN, PKV_STATUS_BAD_PAGE, PKV_STATUS_TASKS, PKV_STATUS_TIMEOUT, PKV_VARIANT_SINGLE,
                   PKV_VARIANT_SPLIT, PKV_VARIANT_WORKQUEUE, VARIANT_NAMES, PkvError, load)
from .binding import (Plan, Policy, Problem, alloc_workspace, decode, make_problem, pkv_build_worklist,  # noqa: F401
                      pkv_check_problem, pkv_decode, pkv_decode_step, pkv_decode_step_append, pkv_decode_step_static,
                      pkv_merge, pkv_plan, pkv_plan_fixed, pkv_plan_launches, pkv_policy_default, pkv_read_status,
                      pkv_serve_step, pkv_step_input_layout, pkv_strerror, pkv_version, pkv_workspace_init, ServeSession,
                      ServeStep)
