"""ctypes view of include/pkv.h and the loader of the in-tree libpkv.so.

There is no fallback: if the CUDA library is missing or fails to load, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libpkv.so")

PKV_OK = 0
PKV_E_INVAL = -1
PKV_E_UNSUPPORTED = -2
PKV_E_NULLPTR = -3
PKV_E_WS_TOO_SMALL = -4
PKV_E_ALIGN = -5
PKV_E_CUDA = -6

PKV_STATUS_BAD_PAGE = 0x1
PKV_STATUS_BAD_LEN = 0x2
PKV_STATUS_TIMEOUT = 0x4
PKV_STATUS_TASKS = 0x8

PKV_MAX_BATCH = 4096
PKV_MAX_ROWS_IN_DECODE = 256

PKV_PLAN_OVERLAP_PREV = 0x1
PKV_PLAN_INPUTS_AFTER_PREV = 0x2

PKV_VARIANT_SINGLE = 0
PKV_VARIANT_SPLIT = 1
PKV_VARIANT_WORKQUEUE = 2
VARIANT_NAMES = {PKV_VARIANT_SINGLE: "single", PKV_VARIANT_SPLIT: "split", PKV_VARIANT_WORKQUEUE: "workqueue"}

# every symbol include/pkv.h declares
EXPORTS = (
    "pkv_version", "pkv_strerror", "pkv_check_problem", "pkv_policy_default", "pkv_plan", "pkv_plan_fixed",
    "pkv_workspace_init", "pkv_build_worklist", "pkv_decode", "pkv_merge", "pkv_decode_step", "pkv_read_status",
    "pkv_plan_launches", "pkv_decode_step_static", "pkv_decode_step_append", "pkv_step_input_layout",
    "pkv_serve_step", "pkv_session_create", "pkv_session_step", "pkv_session_stats", "pkv_session_destroy",
)

PKV_SESSION_GRAPHS = 16

PKV_STATIC_SCRATCH_BYTES = 16 << 20


class Problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32)]


class Policy(ctypes.Structure):
    _fields_ = [("launch_us", ctypes.c_double), ("hbm_gbs", ctypes.c_double), ("cta_gbs", ctypes.c_double),
                ("wq_cta_gbs", ctypes.c_double), ("task_us", ctypes.c_double), ("tail", ctypes.c_double),
                ("merge_us", ctypes.c_double), ("merge_state_us", ctypes.c_double), ("fused_us", ctypes.c_double),
                ("fused_state_us", ctypes.c_double), ("build_us", ctypes.c_double), ("ctas_per_sm", ctypes.c_int32),
                ("max_splits", ctypes.c_int32), ("allow_variants", ctypes.c_int32), ("allow_fused", ctypes.c_int32),
                ("split_max_batch", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    CONSTANTS = ("launch_us", "hbm_gbs", "cta_gbs", "wq_cta_gbs", "task_us", "tail", "merge_us", "merge_state_us",
                 "fused_us", "fused_state_us", "build_us")


class Plan(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("chunk_pages", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("num_tasks", ctypes.c_int32), ("grid_ctas", ctypes.c_int32), ("group", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("fuse_merge", ctypes.c_int32), ("list_in_decode", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("problem", Problem),
                ("task_capacity", ctypes.c_int64), ("state_capacity", ctypes.c_int64),
                ("ws_bytes", ctypes.c_int64), ("off_counters", ctypes.c_int64), ("off_row_off", ctypes.c_int64),
                ("off_row_splits", ctypes.c_int64),
                ("off_tasks", ctypes.c_int64), ("off_ml", ctypes.c_int64), ("off_acc", ctypes.c_int64),
                ("predicted_us", ctypes.c_double), ("kv_bytes", ctypes.c_double)]

    def describe(self) -> dict:
        return {"variant": VARIANT_NAMES.get(self.variant, self.variant), "chunk_pages": self.chunk_pages,
                "num_splits": self.num_splits, "num_tasks": self.num_tasks, "grid_ctas": self.grid_ctas,
                "fuse_merge": self.fuse_merge, "list_in_decode": self.list_in_decode, "ws_bytes": self.ws_bytes,
                "predicted_us": self.predicted_us}


_lib = None
_lock = threading.Lock()
_P = ctypes.POINTER
_vp = ctypes.c_void_p


def load(path: str | None = None):
    """Loads libpkv.so (raises if it was not built: there is no non-CUDA path)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"libpkv.so not built ({path}); run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        lib.pkv_version.restype = ctypes.c_int
        lib.pkv_version.argtypes = []
        lib.pkv_strerror.restype = ctypes.c_char_p
        lib.pkv_strerror.argtypes = [ctypes.c_int]
        lib.pkv_check_problem.restype = ctypes.c_int
        lib.pkv_check_problem.argtypes = [_P(Problem)]
        lib.pkv_policy_default.restype = None
        lib.pkv_policy_default.argtypes = [_P(Policy)]
        lib.pkv_plan.restype = ctypes.c_int
        lib.pkv_plan.argtypes = [_P(Problem), _vp, ctypes.c_int32, _P(Policy), _P(Plan)]
        lib.pkv_plan_fixed.restype = ctypes.c_int
        lib.pkv_plan_fixed.argtypes = [_P(Problem), _vp, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_int32, _P(Plan)]
        lib.pkv_workspace_init.restype = ctypes.c_int
        lib.pkv_workspace_init.argtypes = [_vp, ctypes.c_size_t, _vp]
        lib.pkv_build_worklist.restype = ctypes.c_int
        lib.pkv_build_worklist.argtypes = [_P(Plan), _P(Problem), _vp, _vp, ctypes.c_size_t, _vp]
        dec = [_P(Plan), _P(Problem), _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, ctypes.c_size_t, _vp, _vp]
        lib.pkv_decode.restype = ctypes.c_int
        lib.pkv_decode.argtypes = dec
        lib.pkv_decode_step.restype = ctypes.c_int
        lib.pkv_decode_step.argtypes = dec
        lib.pkv_merge.restype = ctypes.c_int
        lib.pkv_merge.argtypes = [_P(Plan), _P(Problem), _vp, ctypes.c_size_t, _vp, _vp]
        lib.pkv_read_status.restype = ctypes.c_int
        lib.pkv_read_status.argtypes = [_vp, ctypes.c_size_t, _vp, _P(ctypes.c_uint32)]
        lib.pkv_plan_launches.restype = ctypes.c_int
        lib.pkv_plan_launches.argtypes = [_P(Plan)]
        lib.pkv_decode_step_append.restype = ctypes.c_int
        lib.pkv_decode_step_append.argtypes = [_P(Plan), _P(Problem), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                               ctypes.c_float, _vp, ctypes.c_size_t, _vp, _vp]
        lib.pkv_decode_step_static.restype = ctypes.c_int
        lib.pkv_decode_step_static.argtypes = [_P(Plan), _P(Problem), _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp,
                                               _vp, _vp]
        lib.pkv_step_input_layout.restype = ctypes.c_int
        lib.pkv_step_input_layout.argtypes = [_P(Problem), _P(ctypes.c_size_t), _P(ctypes.c_size_t)]
        lib.pkv_serve_step.restype = ctypes.c_int
        lib.pkv_serve_step.argtypes = [_P(Problem), _P(Policy), ctypes.c_int32, _vp, _vp, _vp, _vp, ctypes.c_float,
                                       _vp, ctypes.c_size_t, _vp, _vp, _vp, _P(Plan)]
        lib.pkv_session_create.restype = ctypes.c_int
        lib.pkv_session_create.argtypes = [_P(Problem), _P(Policy), ctypes.c_int32, _vp, _vp, _vp, _vp,
                                           ctypes.c_float, _vp, ctypes.c_size_t, _vp, _vp, _P(_vp)]
        lib.pkv_session_step.restype = ctypes.c_int
        lib.pkv_session_step.argtypes = [_vp, _vp, _P(Plan)]
        lib.pkv_session_stats.restype = ctypes.c_int
        lib.pkv_session_stats.argtypes = [_vp, _P(ctypes.c_int64), _P(ctypes.c_int64)]
        lib.pkv_session_destroy.restype = ctypes.c_int
        lib.pkv_session_destroy.argtypes = [_vp]
        _lib = lib
        return lib


class PkvError(RuntimeError):
    def __init__(self, code: int, what: str):
        msg = load().pkv_strerror(code).decode()
        super().__init__(f"{what}: {msg} ({code})")
        self.code = code


def check(code: int, what: str) -> None:
    if code != PKV_OK:
        raise PkvError(code, what)
