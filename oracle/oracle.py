"""ctypes wrapper around ``pkv_oracle.c`` plus the oracle's scheduler counters. TEST INFRASTRUCTURE ONLY.

Source: "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity GPUs" (arXiv
2606.26666). The attention, split-state, merge and worklist definitions are documented in ``pkv_oracle.c``. The
counters below follow the gist.science technical summary, "Resultaten" ("Scheduling Overhead"), and the v2
abstract: the exact-length-bucket schedule launches once per distinct length, the workqueue schedule launches a
split kernel and a merge kernel.

Parity status: ``launch_counts`` is pinned by the pages' printed 16.00 / 2.00 launches per step on bimodal B8
(tests/golden/launch_fanout_b8_bimodal.txt). ``merge_state_bytes`` is pinned by byte counts derived by hand for
small cases (tests/test_golden_counters.py); the pages' ~37 % reduction cannot pin it, because the pages do not
state the split size it was measured at.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libpkv_oracle.so")
_lib = None
_lock = threading.Lock()

_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c with gcc (OpenMP when available). Returns the library path."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.pkv_oracle_half_to_double.restype = ctypes.c_double
            lib.pkv_oracle_half_to_double.argtypes = [ctypes.c_uint16]
            lib.pkv_oracle_num_threads.restype = ctypes.c_int
            shape = [ctypes.c_int] * 7
            lib.pkv_oracle_attention.restype = ctypes.c_int
            lib.pkv_oracle_attention.argtypes = shape + [_u16p, _u16p, _u16p, _i32p, _i32p, ctypes.c_double,
                                                         _i32p, ctypes.c_int64, _f64p]
            lib.pkv_oracle_split_state.restype = ctypes.c_int
            lib.pkv_oracle_split_state.argtypes = shape + [_u16p, _u16p, _u16p, _i32p, _i32p, ctypes.c_double,
                                                           ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                           _f64p, _f64p, _f64p]
            lib.pkv_oracle_merge.restype = None
            lib.pkv_oracle_merge.argtypes = [ctypes.c_int64, ctypes.c_int, _f64p, _f64p, _f64p, _f64p]
            lib.pkv_oracle_worklist.restype = ctypes.c_int64
            lib.pkv_oracle_worklist.argtypes = [ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                _i32p, ctypes.c_int64]
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype, ptr):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ptr)


def _bits(a: np.ndarray):
    a = np.ascontiguousarray(a, dtype=np.float16).view(np.uint16)
    return a, a.ctypes.data_as(_u16p)


def num_threads() -> int:
    return int(_load().pkv_oracle_num_threads())


def half_to_double(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    return np.array([lib.pkv_oracle_half_to_double(int(x)) for x in np.asarray(bits, dtype=np.uint16).ravel()])


def _shape_args(q, k_pool, block_table):
    B, Hq, d = q.shape
    num_pages, ps, Hkv, d2 = k_pool.shape
    if d2 != d:
        raise ValueError("head_dim mismatch")
    return [B, Hq, Hkv, d, ps, num_pages, block_table.shape[1]]


def attention(q, k_pool, v_pool, block_table, seq_lens, scale=None, pairs=None) -> np.ndarray:
    """fp64 attention output. Without ``pairs`` returns [B, Hq, d]; with ``pairs`` ([n, 2] of (b, hq)) [n, d]."""
    lib = _load()
    dims = _shape_args(q, k_pool, block_table)
    d = dims[3]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    qa, qp = _bits(q)
    ka, kp = _bits(k_pool)
    va, vp = _bits(v_pool)
    bt, btp = _c(block_table, np.int32, _i32p)
    sl, slp = _c(seq_lens, np.int32, _i32p)
    if pairs is None:
        n = dims[0] * dims[1]
        pa, pp = None, None
    else:
        pa, pp = _c(np.asarray(pairs).reshape(-1, 2), np.int32, _i32p)
        n = pa.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    rc = lib.pkv_oracle_attention(*dims, qp, kp, vp, btp, slp, float(scale), pp, n, out.ctypes.data_as(_f64p))
    if rc != 0:
        raise ValueError(f"oracle attention failed: {rc}")
    return out.reshape(dims[0], dims[1], d) if pairs is None else out


def split_states(q, k_pool, v_pool, block_table, seq_lens, b, hq, ranges, scale=None):
    """Partial (m, l, acc) states of pair (b, hq) over the given token ranges [(t0, t1), ...]."""
    lib = _load()
    dims = _shape_args(q, k_pool, block_table)
    d = dims[3]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    qa, qp = _bits(q)
    ka, kp = _bits(k_pool)
    va, vp = _bits(v_pool)
    bt, btp = _c(block_table, np.int32, _i32p)
    sl, slp = _c(seq_lens, np.int32, _i32p)
    S = len(ranges)
    m = np.zeros(S)
    l = np.zeros(S)
    acc = np.zeros((S, d))
    for i, (t0, t1) in enumerate(ranges):
        mi = ctypes.c_double()
        li = ctypes.c_double()
        row = np.zeros(d)
        rc = lib.pkv_oracle_split_state(*dims, qp, kp, vp, btp, slp, float(scale), int(b), int(hq), int(t0),
                                        int(t1), ctypes.byref(mi), ctypes.byref(li), row.ctypes.data_as(_f64p))
        if rc != 0:
            raise ValueError(f"oracle split state failed: {rc}")
        m[i], l[i], acc[i] = mi.value, li.value, row
    return m, l, acc


def merge(m, l, acc) -> np.ndarray:
    lib = _load()
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    S, d = acc.shape
    out = np.zeros(d)
    lib.pkv_oracle_merge(S, d, m.ctypes.data_as(_f64p), l.ctypes.data_as(_f64p), acc.ctypes.data_as(_f64p),
                         out.ctypes.data_as(_f64p))
    return out


def worklist(seq_lens, page_size: int, num_kv_heads: int, chunk_pages: int) -> np.ndarray:
    """Reference task list: int32 [count, 5] rows (b, h_kv, s, page_begin, page_end)."""
    lib = _load()
    sl, slp = _c(seq_lens, np.int32, _i32p)
    n = lib.pkv_oracle_worklist(len(sl), slp, page_size, num_kv_heads, chunk_pages, None, 0)
    if n < 0:
        raise ValueError("bad worklist arguments")
    tasks = np.zeros((max(n, 1), 5), dtype=np.int32)
    lib.pkv_oracle_worklist(len(sl), slp, page_size, num_kv_heads, chunk_pages, tasks.ctypes.data_as(_i32p), n)
    return tasks[:n]


def launch_counts(seq_lens) -> dict:
    """Kernel launches for one decode step under the two schedules the pages compare.

    Exact-length buckets: one split-decode launch and one merge launch for every distinct sequence length.
    Compact workqueue: one split-decode launch over the task list and one merge launch, whatever the lengths.
    """
    distinct = len(set(int(x) for x in np.asarray(seq_lens).ravel() if int(x) > 0))
    return {"exact_buckets": 2 * distinct, "workqueue": 2}


def merge_state_bytes(seq_lens, page_size: int, num_q_heads: int, num_kv_heads: int, chunk_pages: int,
                      head_dim: int = 128) -> dict:
    """Bytes of partial states written then read by the merge, rectangular split grid vs compact workqueue.

    A state is (m, l, acc[head_dim]) in fp32. The rectangular grid holds B*Hq*max_b(S_b) states (empty splits
    write neutral states); the workqueue holds sum_b Hq*S_b. Every state is written once and read once.
    """
    L = np.asarray(seq_lens, dtype=np.int64)
    P = (L + page_size - 1) // page_size
    S = (P + chunk_pages - 1) // chunk_pages
    per_state = 4 * (head_dim + 2)
    rect = int(len(L) * num_q_heads * (S.max() if len(S) else 0)) * per_state * 2
    wq = int(num_q_heads * S.sum()) * per_state * 2
    return {"rect": rect, "workqueue": wq}
