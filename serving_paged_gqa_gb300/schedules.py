"""Comparison schedules for one decode step, built on the library's own calls.

"PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity GPUs", gist.science technical
summary: "Methodologie" 1, "Compact Workqueue" (exact-length bucketing fans out one launch group per distinct length;
the compact workqueue avoids it), "Row-Local Bounds" (coarse padded batches pad rows to a common length) and
"Calibrated Adaptive Policy" (B = 1 uses length buckets and sequence splitting); "Resultaten", "Scheduling Overhead"
(16.00 launches per step with exact buckets against 2.00 with the workqueue on held-out bimodal B8, merge-state
traffic about 37 % lower).

- ExactLengthBuckets: rows of equal length form a group; every group runs its own split-grid decode and merge, with
  the split size the planner picks for that group's length (length-bucketed split selection). Rows are stored
  sorted by length, as an exact-length-bucketing server keeps them, so each group is a contiguous window.
- padded_grid_plan: one rectangular split grid over the batch, every row cut into the splits of the longest row;
  rows shorter than that write neutral states for their empty splits (the merge state a padded batch carries).
- workqueue_plan: the compact workqueue the planner picks.

Counters (launches per step, partial-state bytes written and read) follow the same definitions as the oracle's.
"""

from __future__ import annotations

import numpy as np

STATE_BYTES = 4 * (128 + 2)  # (m, l, acc[128]) in fp32


def split_policy(pkv):
    """The planner restricted to the split grid for any batch size."""
    pol = pkv.pkv_policy_default()
    pol.allow_variants = 1 << pkv.PKV_VARIANT_SPLIT
    pol.split_max_batch = pkv.PKV_MAX_BATCH
    return pol


def state_bytes(plan) -> int:
    """Partial-state bytes a plan writes and its merge reads (0 for the single pass)."""
    if plan.variant == 0:
        return 0
    return 2 * int(plan.num_tasks) * int(plan.group) * STATE_BYTES


def padded_grid_plan(pkv, problem, lens, sms):
    return pkv.pkv_plan(problem, lens, sms, split_policy(pkv))


def workqueue_plan(pkv, problem, lens, sms):
    pol = pkv.pkv_policy_default()
    pol.allow_variants = 1 << pkv.PKV_VARIANT_WORKQUEUE
    return pkv.pkv_plan(problem, lens, sms, pol)


class ExactLengthBuckets:
    """One split-grid decode + merge per distinct row length, on a batch stored sorted by length."""

    def __init__(self, pkv, problem, lens_sorted, sms):
        lens_sorted = np.asarray(lens_sorted, dtype=np.int32)
        if np.any(np.diff(lens_sorted) < 0):
            raise ValueError("rows must be sorted by length")
        self.pkv = pkv
        pol = split_policy(pkv)
        self.groups = []  # (r0, r1, problem, plan)
        r0 = 0
        B = len(lens_sorted)
        while r0 < B:
            r1 = r0 + 1
            while r1 < B and lens_sorted[r1] == lens_sorted[r0]:
                r1 += 1
            if lens_sorted[r0] > 0:
                pr = pkv.make_problem(r1 - r0, problem.num_q_heads, problem.num_kv_heads, problem.head_dim,
                                      problem.page_size, problem.num_pages, problem.max_pages_per_seq)
                plan = pkv.pkv_plan(pr, lens_sorted[r0:r1], sms, pol)
                plan.fuse_merge = 0  # the split kernel and the merge kernel of the pages' schedule
                self.groups.append((r0, r1, pr, plan))
            r0 = r1
        self.ws_bytes = max([p.ws_bytes for _, _, _, p in self.groups], default=256)

    def launches(self) -> int:
        return sum(self.pkv.pkv_plan_launches(p) for _, _, _, p in self.groups)

    def state_bytes(self) -> int:
        return sum(state_bytes(p) for _, _, _, p in self.groups)

    def run(self, q, k_pool, v_pool, block_table, seq_lens, scale, ws, out, stream=None):
        """All groups on one stream; q, block_table, seq_lens and out hold the rows in sorted order. Rows of length
        0 (no group) get a zero output."""
        covered = np.zeros(q.shape[0], dtype=bool)
        for r0, r1, pr, plan in self.groups:
            self.pkv.pkv_decode_step(plan, pr, q[r0:r1], k_pool, v_pool, block_table[r0:r1], seq_lens[r0:r1], scale,
                                     ws, out[r0:r1], stream)
            covered[r0:r1] = True
        for r in np.nonzero(~covered)[0]:
            out[int(r)].zero_()
