"""pkv_decode_step_static: the decode step for callers that cannot allocate device memory.

Such callers (a plug-in whose host application owns every allocation, code inside another framework's memory
pool, a serving loop that must not allocate after start-up) cannot hand the library a workspace. This entry point
keeps the workspace in a fixed array in the library's own device memory instead. The test calls it through the C
ABI twice in a row on the same inputs and compares each result with pkv_decode_step on a caller-owned workspace,
within the tolerance every parity test here uses. The file name makes pytest collect it last.
"""

import numpy as np
import pytest
import torch

import serving_paged_gqa_gb300 as pkv
from workloads import make_trace

from gpu_harness import ATOL, RTOL, Step

pytestmark = pytest.mark.gpu

SINGLE, SPLIT, WQ = pkv.PKV_VARIANT_SINGLE, pkv.PKV_VARIANT_SPLIT, pkv.PKV_VARIANT_WORKQUEUE


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


def _close(a: torch.Tensor, b: torch.Tensor, what: str):
    x = a.float().cpu().numpy().astype(np.float64)
    y = b.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(x).all(), f"{what}: non-finite output"
    excess = np.abs(x - y) - (ATOL + RTOL * np.abs(y))
    assert excess.max() <= 0, f"{what}: max |static - workspace| = {np.abs(x - y).max():.3e}"


@pytest.mark.parametrize("name,seed,t,variant,chunk", [
    ("tiny", 0, 0, SPLIT, 8),
    ("tiny", 1, 0, SINGLE, 1),
    ("b1_bucketed", 6, 3, None, 1),
    ("b8_bimodal", 5, 0, WQ, 32),
    ("b8_zipf", 7, 2, SPLIT, 32),
])
def test_static_scratch_matches_workspace_path(name, seed, t, variant, chunk):
    tr = make_trace(name, seed, steps=t + 1)
    step = Step(tr, t)
    plan = step.plan(variant, chunk)
    assert plan.ws_bytes <= pkv.PKV_STATIC_SCRATCH_BYTES
    want, _, status = step.run(plan)
    assert status == 0
    st = torch.full((1,), -1, dtype=torch.int32, device=step.q.device)
    for call in range(2):
        out = torch.full_like(step.q, float("nan"))
        pkv.pkv_decode_step_static(plan, step.problem, step.q, step.k, step.v, step.bt, step.lens, step.scale, out,
                                   status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"call {call}: status {int(st.item()):#x}"
        _close(out, want, f"{name} {plan.describe()} call {call}")


def test_static_scratch_reports_and_clears_device_status():
    step = Step(make_trace("tiny", 1), 0, poison=False)
    plan = step.plan(SPLIT, 8)
    good = step.bt.clone()
    step.bt[0, 3] = step.tr.num_pages + 5  # a block-table entry outside the pool
    st = torch.zeros((1,), dtype=torch.int32, device=step.q.device)
    out = torch.empty_like(step.q)
    pkv.pkv_decode_step_static(plan, step.problem, step.q, step.k, step.v, step.bt, step.lens, step.scale, out,
                               status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & pkv.PKV_STATUS_BAD_PAGE
    # the next call starts from a cleared status word
    pkv.pkv_decode_step_static(plan, step.problem, step.q, step.k, step.v, good, step.lens, step.scale, out,
                               status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_static_scratch_rejects_plans_beyond_its_size():
    tr = make_trace("stress", 5, steps=1)
    lens = tr.seq_lens(0)
    problem = pkv.make_problem(tr.batch, tr.hq, tr.hkv, tr.d, tr.ps, tr.num_pages, tr.max_pages)
    plan = pkv.pkv_plan_fixed(problem, lens, 152, WQ, 1)  # about 95k tasks: far beyond the fixed array
    assert plan.ws_bytes > pkv.PKV_STATIC_SCRATCH_BYTES
    q = torch.zeros((tr.batch, tr.hq, tr.d), dtype=torch.float16, device="cuda")
    kv = torch.zeros((1, tr.ps, tr.hkv, tr.d), dtype=torch.float16, device="cuda")
    bt = torch.zeros((tr.batch, tr.max_pages), dtype=torch.int32, device="cuda")
    sl = torch.from_numpy(lens).cuda()
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_step_static(plan, problem, q, kv, kv, bt, sl, 1.0, torch.empty_like(q))
    assert e.value.code == -4
