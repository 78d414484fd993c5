"""Helpers for the GPU parity tests: device copies of a trace step and the oracle comparison."""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import serving_paged_gqa_gb300 as pkv

ATOL, RTOL = 2e-3, 1e-2  # |gpu - fp64 oracle| <= ATOL + RTOL * |oracle|, elementwise


class Step:
    """Device tensors for step t of a trace. Unused pool pages and the slots past each row's length are NaN, so a
    kernel that reads outside the row's tokens produces NaN and fails the comparison."""

    def __init__(self, tr, t: int, dev="cuda", poison: bool = True):
        self.tr, self.t = tr, t
        ps, hkv, d = tr.ps, tr.hkv, tr.d
        kp = tr.k_pages.copy()
        vp = tr.v_pages.copy()
        if poison:
            dead = np.arange(ps)[None, :] >= tr.valid_slots(t)[:, None]
            kp[dead] = np.nan
            vp[dead] = np.nan
        fill = float("nan") if poison else 0.0
        self.k = torch.full((tr.num_pages, ps, hkv, d), fill, dtype=torch.float16, device=dev)
        self.v = torch.full((tr.num_pages, ps, hkv, d), fill, dtype=torch.float16, device=dev)
        idx = torch.from_numpy(tr.used_pages).to(dev)
        self.k.index_copy_(0, idx, torch.from_numpy(kp).to(dev))
        self.v.index_copy_(0, idx, torch.from_numpy(vp).to(dev))
        self.q_host = tr.q(t)
        self.bt_host = tr.block_table(t)
        self.lens_host = tr.seq_lens(t)
        self.q = torch.from_numpy(self.q_host).to(dev)
        self.bt = torch.from_numpy(self.bt_host).to(dev)
        self.lens = torch.from_numpy(self.lens_host).to(dev)
        self.problem = pkv.make_problem(tr.batch, tr.hq, tr.hkv, d, ps, tr.num_pages, tr.max_pages)
        self.scale = 1.0 / math.sqrt(d)
        self.sms = torch.cuda.get_device_properties(self.q.device).multi_processor_count
        self._ref = None

    def plan(self, variant=None, chunk=1, sms=None):
        sms = self.sms if sms is None else sms
        if variant is None:
            return pkv.pkv_plan(self.problem, self.lens_host, sms)
        return pkv.pkv_plan_fixed(self.problem, self.lens_host, sms, variant, chunk)

    def run(self, plan, ws=None):
        if ws is None:
            ws = pkv.alloc_workspace(plan.ws_bytes, self.q.device)
        out = torch.full_like(self.q, float("nan"))
        pkv.pkv_decode_step(plan, self.problem, self.q, self.k, self.v, self.bt, self.lens, self.scale, ws, out)
        torch.cuda.synchronize()
        status = pkv.pkv_read_status(ws)
        return out, ws, status

    def reference(self, pairs=None):
        kp, vp = self.tr.host_pools()
        if pairs is not None:
            return oracle.attention(self.q_host, kp, vp, self.bt_host, self.lens_host, self.scale, pairs=pairs)
        if self._ref is None:
            self._ref = oracle.attention(self.q_host, kp, vp, self.bt_host, self.lens_host, self.scale)
        return self._ref


def assert_close(got: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = got.float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    excess = np.abs(g - ref) - (ATOL + RTOL * np.abs(ref))
    i = int(np.argmax(excess))
    assert excess.flat[i] <= 0, (f"{what}: |gpu-oracle| = {np.abs(g - ref).flat[i]:.3e} at flat index {i} "
                                 f"(oracle {ref.flat[i]:.4e}) exceeds {ATOL} + {RTOL}*|oracle|")
    return float(np.abs(g - ref).max())


def read_worklist(plan, ws):
    torch.cuda.synchronize()
    hdr = ws[:256].view(torch.int32).cpu().numpy()
    count = int(hdr[1])
    tasks = ws[plan.off_tasks:plan.off_tasks + 16 * count].view(torch.int32).cpu().numpy().reshape(count, 4)
    out = np.zeros((count, 5), dtype=np.int32)
    out[:, 0] = tasks[:, 0]
    out[:, 1] = tasks[:, 1] >> 16
    out[:, 2] = tasks[:, 1] & 0xFFFF
    out[:, 3] = tasks[:, 2]
    out[:, 4] = tasks[:, 3]
    B = plan.problem.batch
    row_off = ws[plan.off_row_off:plan.off_row_off + 4 * B].view(torch.int32).cpu().numpy()
    row_splits = ws[plan.off_row_splits:plan.off_row_splits + 4 * B].view(torch.int32).cpu().numpy()
    return out, row_off, row_splits, int(hdr[0])
