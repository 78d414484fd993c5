"""Python binding of libpkv.so: the C-ABI calls under the same names, taking torch tensors.

Argument marshalling only: every step of the decode path (worklist build, decode, merge) runs in the library's
CUDA kernels; the planner runs in the library's host code. PyTorch provides device memory and streams.
"""

from __future__ import annotations

import ctypes
import math

import numpy as np
import torch

from ._lib import (PKV_VARIANT_SINGLE, PKV_VARIANT_SPLIT, PKV_VARIANT_WORKQUEUE, Plan, Policy, Problem, check,
                   load)

__all__ = [
    "Problem", "Plan", "Policy", "pkv_version", "pkv_strerror", "pkv_check_problem", "pkv_policy_default",
    "pkv_plan", "pkv_plan_fixed", "pkv_workspace_init", "pkv_build_worklist", "pkv_decode", "pkv_merge",
    "pkv_decode_step", "pkv_read_status", "pkv_plan_launches", "pkv_decode_step_static", "pkv_decode_step_append",
    "pkv_step_input_layout", "pkv_serve_step", "ServeStep", "make_problem",
    "alloc_workspace", "decode",
    "PKV_VARIANT_SINGLE", "PKV_VARIANT_SPLIT", "PKV_VARIANT_WORKQUEUE",
]


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t: torch.Tensor | None, dtype=None, name: str = "tensor") -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _host_lens(seq_lens) -> np.ndarray:
    if isinstance(seq_lens, torch.Tensor):
        seq_lens = seq_lens.detach().cpu().numpy()
    if isinstance(seq_lens, np.ndarray) and seq_lens.dtype == np.int32 and seq_lens.flags.c_contiguous:
        return seq_lens
    return np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))


def pkv_version() -> int:
    return load().pkv_version()


def pkv_strerror(code: int) -> str:
    return load().pkv_strerror(code).decode()


def make_problem(batch, num_q_heads, num_kv_heads, head_dim, page_size, num_pages, max_pages_per_seq) -> Problem:
    return Problem(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim), int(page_size), int(num_pages),
                   int(max_pages_per_seq))


def pkv_check_problem(problem: Problem) -> int:
    return load().pkv_check_problem(ctypes.byref(problem))


def pkv_policy_default() -> Policy:
    pol = Policy()
    load().pkv_policy_default(ctypes.byref(pol))
    return pol


def pkv_plan(problem: Problem, seq_lens_host, num_sms: int, policy: Policy | None = None) -> Plan:
    lens = _host_lens(seq_lens_host)
    plan = Plan()
    pol = ctypes.byref(policy) if policy is not None else None
    check(load().pkv_plan(ctypes.byref(problem), lens.ctypes.data, int(num_sms),
                          pol, ctypes.byref(plan)), "pkv_plan")
    return plan


def pkv_plan_fixed(problem: Problem, seq_lens_host, num_sms: int, variant: int, chunk_pages: int = 1,
                   ctas_per_sm: int = 0) -> Plan:
    lens = _host_lens(seq_lens_host)
    plan = Plan()
    check(load().pkv_plan_fixed(ctypes.byref(problem), lens.ctypes.data,
                                int(num_sms), int(variant), int(chunk_pages), int(ctas_per_sm), ctypes.byref(plan)),
          "pkv_plan_fixed")
    return plan


def pkv_plan_launches(plan: Plan) -> int:
    return load().pkv_plan_launches(ctypes.byref(plan))


def alloc_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A uint8 CUDA tensor usable as workspace (torch's allocator returns 256-byte aligned blocks)."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")
    pkv_workspace_init(ws)
    return ws


def pkv_workspace_init(ws: torch.Tensor, stream=None) -> None:
    check(load().pkv_workspace_init(_ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "pkv_workspace_init")


def pkv_build_worklist(plan: Plan, problem: Problem, seq_lens: torch.Tensor, ws: torch.Tensor, stream=None) -> None:
    check(load().pkv_build_worklist(ctypes.byref(plan), ctypes.byref(problem), _ptr(seq_lens, torch.int32, "seq_lens"),
                                    _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "pkv_build_worklist")


def _decode_args(plan, problem, q, k_pool, v_pool, block_table, seq_lens, scale, ws, out, stream):
    return (ctypes.byref(plan), ctypes.byref(problem), _ptr(q, torch.float16, "q"), _ptr(k_pool, torch.float16, "k_pool"),
            _ptr(v_pool, torch.float16, "v_pool"), _ptr(block_table, torch.int32, "block_table"),
            _ptr(seq_lens, torch.int32, "seq_lens"), ctypes.c_float(scale), _ptr(ws, torch.uint8, "ws"), ws.numel(),
            _ptr(out, torch.float16, "out"), _stream(stream))


def pkv_decode(plan, problem, q, k_pool, v_pool, block_table, seq_lens, scale, ws, out=None, stream=None) -> None:
    check(load().pkv_decode(*_decode_args(plan, problem, q, k_pool, v_pool, block_table, seq_lens, scale, ws, out,
                                          stream)), "pkv_decode")


def pkv_merge(plan: Plan, problem: Problem, ws: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    check(load().pkv_merge(ctypes.byref(plan), ctypes.byref(problem), _ptr(ws, torch.uint8, "ws"), ws.numel(),
                           _ptr(out, torch.float16, "out"), _stream(stream)), "pkv_merge")


def pkv_decode_step(plan, problem, q, k_pool, v_pool, block_table, seq_lens, scale, ws, out, stream=None) -> None:
    check(load().pkv_decode_step(*_decode_args(plan, problem, q, k_pool, v_pool, block_table, seq_lens, scale, ws,
                                               out, stream)), "pkv_decode_step")


def pkv_decode_step_append(plan, problem, q, k_new, v_new, k_pool, v_pool, block_table, seq_lens, scale, ws, out,
                           stream=None) -> None:
    """pkv_decode_step with the new token's K/V ([B, Hkv, d] fp16) appended into the pools inside the decode."""
    check(load().pkv_decode_step_append(
        ctypes.byref(plan), ctypes.byref(problem), _ptr(q, torch.float16, "q"), _ptr(k_new, torch.float16, "k_new"),
        _ptr(v_new, torch.float16, "v_new"), _ptr(k_pool, torch.float16, "k_pool"),
        _ptr(v_pool, torch.float16, "v_pool"), _ptr(block_table, torch.int32, "block_table"),
        _ptr(seq_lens, torch.int32, "seq_lens"), ctypes.c_float(scale), _ptr(ws, torch.uint8, "ws"), ws.numel(),
        _ptr(out, torch.float16, "out"), _stream(stream)), "pkv_decode_step_append")


def pkv_decode_step_static(plan, problem, q, k_pool, v_pool, block_table, seq_lens, scale, out, status=None,
                           stream=None) -> None:
    """pkv_decode_step with the workspace in the library's fixed device array (no allocation by the call).

    ``status``, if given, is a CUDA int32/uint32-sized tensor of one element that receives the step's status bits.
    """
    if status is not None and (not status.is_cuda or status.numel() != 1 or status.element_size() != 4):
        raise ValueError("status must be a one-element 4-byte CUDA tensor")
    check(load().pkv_decode_step_static(
        ctypes.byref(plan), ctypes.byref(problem), _ptr(q, torch.float16, "q"), _ptr(k_pool, torch.float16, "k_pool"),
        _ptr(v_pool, torch.float16, "v_pool"), _ptr(block_table, torch.int32, "block_table"),
        _ptr(seq_lens, torch.int32, "seq_lens"), ctypes.c_float(scale), _ptr(out, torch.float16, "out"),
        _ptr(status, None, "status"), _stream(stream)), "pkv_decode_step_static")


def pkv_step_input_layout(problem: Problem) -> tuple[tuple[int, ...], int]:
    """Byte offsets of (q, k_new, v_new, block_table, seq_lens) in a packed step input, and its total size."""
    offs = (ctypes.c_size_t * 5)()
    total = ctypes.c_size_t(0)
    check(load().pkv_step_input_layout(ctypes.byref(problem), offs, ctypes.byref(total)), "pkv_step_input_layout")
    return tuple(int(x) for x in offs), int(total.value)


def _serve_args(problem, host_in, dev_in, k_pool, v_pool, scale, ws, dev_out, host_out, stream, policy, num_sms,
                plan_out):
    return _bind_args(problem, host_in, dev_in, k_pool, v_pool, scale, ws, dev_out, host_out, policy, num_sms) + (
        _stream(stream), ctypes.byref(plan_out))


def _bind_args(problem, host_in, dev_in, k_pool, v_pool, scale, ws, dev_out, host_out, policy, num_sms):
    if host_in.is_cuda or host_out.is_cuda:
        raise ValueError("host_in and host_out must be host (pinned) tensors")
    if not (host_in.is_contiguous() and host_out.is_contiguous()):
        raise ValueError("host_in and host_out must be contiguous")
    if host_out.dtype != torch.float16:
        raise ValueError("host_out must be float16")
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(dev_in.device).multi_processor_count
    return (ctypes.byref(problem), None if policy is None else ctypes.byref(policy), int(num_sms),
            ctypes.c_void_p(host_in.data_ptr()), _ptr(dev_in, torch.uint8, "dev_in"),
            _ptr(k_pool, torch.float16, "k_pool"), _ptr(v_pool, torch.float16, "v_pool"), ctypes.c_float(scale),
            _ptr(ws, torch.uint8, "ws"), ws.numel(), _ptr(dev_out, torch.float16, "dev_out"),
            ctypes.c_void_p(host_out.data_ptr()))


def pkv_serve_step(problem, host_in, dev_in, k_pool, v_pool, scale, ws, dev_out, host_out, stream=None, policy=None,
                   num_sms=None) -> Plan:
    """One serving step from host memory (include/pkv.h, pkv_serve_step): plan from the seq_lens in host_in, copy
    host_in (uint8, pinned, laid out by pkv_step_input_layout) into dev_in, decode with the new token's K/V appended,
    copy out into host_out (float16 [B, Hq, d], pinned). Asynchronous: synchronise the stream before reading host_out.
    Returns the plan the step ran."""
    plan = Plan()
    check(load().pkv_serve_step(*_serve_args(problem, host_in, dev_in, k_pool, v_pool, scale, ws, dev_out, host_out,
                                             stream, policy, num_sms, plan)), "pkv_serve_step")
    return plan


class ServeStep:
    """pkv_serve_step with its arguments marshalled once (a server's per-layer buffers do not change between steps):
    run() enqueues one step and returns the plan it ran; refill host_in between steps after synchronising."""

    def __init__(self, problem, host_in, dev_in, k_pool, v_pool, scale, ws, dev_out, host_out, stream=None,
                 policy=None, num_sms=None):
        self.plan = Plan()
        self._keep = (problem, host_in, dev_in, k_pool, v_pool, ws, dev_out, host_out, policy)
        self._args = _serve_args(problem, host_in, dev_in, k_pool, v_pool, scale, ws, dev_out, host_out, stream,
                                 policy, num_sms, self.plan)
        self._fn = load().pkv_serve_step

    def run(self) -> Plan:
        rc = self._fn(*self._args)
        if rc != 0:
            check(rc, "pkv_serve_step")
        return self.plan


class ServeSession:
    """A serving session (include/pkv.h, pkv_session_*): the buffers of pkv_serve_step bound once; run() plans the
    step from the seq_lens in host_in and replays the plan's captured CUDA graph (capturing it the first time the
    plan is seen) when both host buffers are mapped pinned memory, else enqueues the launches directly. Returns the
    plan it ran. Synchronise the stream before reading host_out or refilling host_in; close() when done."""

    def __init__(self, problem, host_in, dev_in, k_pool, v_pool, scale, ws, dev_out, host_out, policy=None,
                 num_sms=None):
        self.plan = Plan()
        self._keep = (problem, host_in, dev_in, k_pool, v_pool, ws, dev_out, host_out, policy)
        a = _bind_args(problem, host_in, dev_in, k_pool, v_pool, scale, ws, dev_out, host_out, policy, num_sms)
        self._lib = load()
        h = ctypes.c_void_p()
        check(self._lib.pkv_session_create(*a, ctypes.byref(h)), "pkv_session_create")
        self._h = h
        self._streams = {}

    def run(self, stream=None) -> Plan:
        """One step on `stream` (None: the current stream, looked up on every call)."""
        if stream is None:
            args = (self._h, _stream(None), ctypes.byref(self.plan))
        else:
            hit = self._streams.get(id(stream))
            if hit is None or hit[0] is not stream:  # the stream object is kept, so its id cannot be reused
                hit = self._streams[id(stream)] = (stream, (self._h, _stream(stream), ctypes.byref(self.plan)))
            args = hit[1]
        rc = self._lib.pkv_session_step(*args)
        if rc != 0:
            check(rc, "pkv_session_step")
        return self.plan

    def stats(self) -> tuple[int, int]:
        """(graphs captured, graph launches) so far."""
        c, n = ctypes.c_int64(0), ctypes.c_int64(0)
        check(self._lib.pkv_session_stats(self._h, ctypes.byref(c), ctypes.byref(n)), "pkv_session_stats")
        return int(c.value), int(n.value)

    def close(self):
        if getattr(self, "_h", None):
            h, self._h = self._h, None
            check(self._lib.pkv_session_destroy(h), "pkv_session_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pkv_read_status(ws: torch.Tensor, stream=None) -> int:
    v = ctypes.c_uint32(0)
    check(load().pkv_read_status(_ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream), ctypes.byref(v)),
          "pkv_read_status")
    return int(v.value)


def decode(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, block_table: torch.Tensor,
           seq_lens: torch.Tensor, seq_lens_host=None, out: torch.Tensor | None = None, plan: Plan | None = None,
           ws: torch.Tensor | None = None, scale: float | None = None, stream=None) -> torch.Tensor:
    """One decode step: plan (host), then build + decode + merge on the device. Returns out [B, Hq, d] fp16.

    q [B,Hq,d] fp16; k_pool / v_pool [num_pages, page_size, Hkv, d] fp16; block_table [B, max_pages] int32;
    seq_lens [B] int32 on the device; seq_lens_host, if given, must equal seq_lens (saves a device read).
    """
    B, Hq, d = q.shape
    num_pages, ps, Hkv, d2 = k_pool.shape
    problem = make_problem(B, Hq, Hkv, d, ps, num_pages, block_table.shape[1])
    if plan is None:
        host = seq_lens_host if seq_lens_host is not None else seq_lens
        plan = pkv_plan(problem, host, torch.cuda.get_device_properties(q.device).multi_processor_count)
    if ws is None or ws.numel() < plan.ws_bytes:
        ws = alloc_workspace(plan.ws_bytes, q.device)
    if out is None:
        out = torch.empty_like(q)
    pkv_decode_step(plan, problem, q, k_pool, v_pool, block_table, seq_lens,
                    1.0 / math.sqrt(d) if scale is None else float(scale), ws, out, stream)
    return out
