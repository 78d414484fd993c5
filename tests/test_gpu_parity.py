"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded inputs.

Worklists must be bit-exact; outputs within 2e-3 absolute + 1e-2 relative of the oracle, elementwise.
"""

import numpy as np
import pytest
import torch

import oracle
import serving_paged_gqa_gb300 as pkv
from workloads import make_trace, normal_fp16, rng_for

from gpu_harness import Step, assert_close, read_worklist

pytestmark = pytest.mark.gpu

SINGLE, SPLIT, WQ = pkv.PKV_VARIANT_SINGLE, pkv.PKV_VARIANT_SPLIT, pkv.PKV_VARIANT_WORKQUEUE


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)


# ----------------------------------------------------------------------------------------------- worklist builder
def _check_worklist(step, chunk):
    plan = step.plan(WQ, chunk)
    ws = pkv.alloc_workspace(plan.ws_bytes)
    pkv.pkv_build_worklist(plan, step.problem, step.lens, ws)
    got, row_off, row_splits, head = read_worklist(plan, ws)
    want = oracle.worklist(step.lens_host, 16, step.tr.hkv, chunk)
    assert got.shape == want.shape and np.array_equal(got, want), f"worklist differs (c={chunk})"
    P = (step.lens_host.astype(np.int64) + 15) // 16
    S = (P + chunk - 1) // chunk
    assert np.array_equal(row_splits, S)
    assert np.array_equal(row_off, np.concatenate([[0], np.cumsum(step.tr.hkv * S)[:-1]]))
    assert head == 0 and pkv.pkv_read_status(ws) == 0


@pytest.mark.parametrize("name,seed,t", [
    ("tiny", 0, 0), ("b1_bucketed", 5, 0), ("b1_bucketed", 6, 63), ("b8_bimodal", 5, 0), ("b8_bimodal", 9, 63),
    ("b8_uniform", 5, 31), ("b8_zipf", 7, 63), ("b4_bimodal", 5, 10), ("stress", 5, 0),
])
def test_worklist_bit_exact_configs(name, seed, t):
    tr = make_trace(name, seed, steps=max(t + 1, 1))
    step = Step(tr, t, poison=False)
    for chunk in (1, 3, 8, 32, 64, 1000):
        _check_worklist(step, chunk)


class _Lens:
    """A step built from explicit lengths (edge cases)."""

    def __init__(self, lens, hkv=8, hq=32, seed=0, extra=5):
        from workloads.traces import Trace

        lens = np.asarray(lens, dtype=np.int64)
        r = rng_for(seed, 4242)
        P = (lens + 15) // 16
        n = int(P.sum())
        num_pages = n + extra
        perm = r.permutation(num_pages)
        max_pages = max(int(P.max()), 1)
        table = np.full((len(lens), max_pages), -1, dtype=np.int32)
        used, rows, logical = [], [], []
        k = 0
        for b, p in enumerate(P):
            for j in range(int(p)):
                table[b, j] = perm[k]
                used.append(perm[k])
                rows.append(b)
                logical.append(j)
                k += 1
        self.trace = Trace(name="edge", seed=seed, batch=len(lens), steps=1, num_pages=num_pages, start=lens,
                           table=table, used_pages=np.array(used, dtype=np.int64),
                           page_row=np.array(rows, dtype=np.int64), page_logical=np.array(logical, dtype=np.int64),
                           hq=hq, hkv=hkv)


def test_worklist_edge_lengths():
    step = Step(_Lens([1, 16, 17, 0, 32, 33, 255, 0]).trace, 0)
    for chunk in (1, 2, 3, 100):
        _check_worklist(step, chunk)
    empty = Step(_Lens([0, 0, 0]).trace, 0)
    _check_worklist(empty, 4)


# ------------------------------------------------------------------------------------------------- decode + merge
@pytest.mark.parametrize("seed", range(10))
def test_tiny_all_schedules(seed):
    step = Step(make_trace("tiny", seed), 0)
    ref = step.reference()
    outs = []
    for variant, chunk in ((SPLIT, 8), (WQ, 8), (SINGLE, 1), (SPLIT, 3), (WQ, 1), (SPLIT, 32), (None, 1)):
        out, _, status = step.run(step.plan(variant, chunk))
        assert status == 0
        assert_close(out, ref, f"tiny seed {seed} variant {variant} c={chunk}")
        outs.append(out.float())
    for o in outs[1:]:  # schedules agree with each other to fp32 round-off plus one fp16 rounding
        assert (o - outs[0]).abs().max().item() < 2e-3


@pytest.mark.parametrize("name,seed,steps", [
    ("b1_bucketed", 5, (0, 63)), ("b1_bucketed", 8, (17,)), ("b8_bimodal", 5, (0, 63)), ("b8_uniform", 6, (40,)),
    ("b8_zipf", 7, (0, 63)), ("b4_bimodal", 5, (5,)),
])
def test_traces_policy_and_forced_schedules(name, seed, steps):
    tr = make_trace(name, seed)
    for t in steps:
        step = Step(tr, t)
        ref = step.reference()
        plans = [step.plan()]
        pmax = int(tr.pages(t).max())
        for S in (8, 64):
            plans.append(step.plan(SPLIT, -(-pmax // S)))
        plans.append(step.plan(WQ, 32))
        if tr.batch > 1:
            plans.append(step.plan(SINGLE))
        for plan in plans:
            out, _, status = step.run(plan)
            assert status == 0, status
            assert_close(out, ref, f"{name} seed {seed} step {t} {plan.describe()}")


@pytest.mark.parametrize("sms", [1, 3])
def test_few_ctas_many_task_boundaries(sms):
    """A grid of 2 or 6 CTAs runs hundreds of tasks each, with page counts per task that are not multiples of the
    consumer-warp count, so the shared-memory page ring wraps across many task boundaries."""
    tr = make_trace("b8_zipf", 5, steps=1)
    step = Step(tr, 0)
    ref = step.reference()
    for variant, chunk in ((SPLIT, 5), (WQ, 3), (WQ, 7), (SPLIT, 1), (SINGLE, 1)):
        out, _, status = step.run(step.plan(variant, chunk, sms=sms))
        assert status == 0
        assert_close(out, ref, f"grid of {2 * sms} CTAs, variant {variant}, c={chunk}")


def test_stress_sampled_pairs():
    tr = make_trace("stress", 5, steps=1)
    step = Step(tr, 0)
    r = rng_for(5, 777)
    pairs = np.stack([np.arange(tr.batch), r.integers(0, tr.hq, tr.batch)], axis=1)
    ref = step.reference(pairs)
    for plan in (step.plan(), step.plan(WQ, 64)):
        out, _, status = step.run(plan)
        assert status == 0
        got = out[torch.from_numpy(pairs[:, 0]), torch.from_numpy(pairs[:, 1])]
        assert_close(got, ref, f"stress {plan.describe()}")


def test_edge_lengths_and_empty_rows():
    step = Step(_Lens([1, 15, 16, 17, 0, 31, 32, 33, 1000, 0]).trace, 0)
    ref = step.reference()
    for variant, chunk in ((SINGLE, 1), (SPLIT, 1), (SPLIT, 5), (WQ, 1), (WQ, 2), (None, 1)):
        out, _, status = step.run(step.plan(variant, chunk))
        assert status == 0
        assert_close(out, ref, f"edge {variant} {chunk}")
        assert not out[4].any() and not out[9].any()  # empty rows give 0
    allempty = Step(_Lens([0, 0]).trace, 0)
    for variant in (SINGLE, SPLIT, WQ):
        out, _, status = allempty.run(allempty.plan(variant, 2))
        assert status == 0


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 2), (16, 1), (32, 2)])
def test_group_sizes(hq, hkv):
    step = Step(_Lens([40, 300, 17], hkv=hkv, hq=hq, seed=hq * 10 + hkv).trace, 0)
    ref = step.reference()
    for variant, chunk in ((SINGLE, 1), (SPLIT, 4), (WQ, 2), (SPLIT, 1)):
        for fused in ((0,) if variant == SINGLE else (0, 1)):  # both merges: the merge task folds G heads per state
            plan = step.plan(variant, chunk)
            if variant != SINGLE:
                plan.fuse_merge = fused
            out, _, status = step.run(plan)
            assert status == 0
            assert_close(out, ref, f"G={hq // hkv} variant {variant} c={chunk} fused={fused}")


def test_partial_states_match_oracle_split_states():
    step = Step(make_trace("tiny", 2), 0)
    chunk = 8
    plan = step.plan(SPLIT, chunk)
    _, ws, status = step.run(plan)
    assert status == 0
    ml = ws[plan.off_ml:plan.off_ml + 8 * plan.state_capacity].view(torch.float32).cpu().numpy().reshape(-1, 2)
    acc = ws[plan.off_acc:plan.off_acc + 512 * plan.state_capacity].view(torch.float32).cpu().numpy()
    acc = acc.reshape(-1, 128)
    kp, vp = step.tr.host_pools()
    S, G = plan.num_splits, plan.group
    for hq in (0, 5, 31):
        h, g = hq // G, hq % G
        ranges = [(s * chunk * 16, (s + 1) * chunk * 16) for s in range(S)]
        m, l, a = oracle.split_states(step.q_host, kp, vp, step.bt_host, step.lens_host, 0, hq, ranges)
        for s in range(S):
            st = (h * S + s) * G + g
            assert abs(ml[st, 0] - m[s]) < 1e-3
            assert abs(ml[st, 1] - l[s]) <= 1e-3 * l[s]
            assert np.max(np.abs(acc[st] / ml[st, 1] - a[s] / l[s])) < 2e-3


def test_rect_empty_splits_write_neutral_states():
    step = Step(_Lens([16, 200]).trace, 0)
    plan = step.plan(SPLIT, 1)  # row 0 has 1 split, row 1 has 13: row 0's splits 1..12 are empty
    _, ws, status = step.run(plan)
    assert status == 0
    ml = ws[plan.off_ml:plan.off_ml + 8 * plan.state_capacity].view(torch.float32).cpu().numpy().reshape(-1, 2)
    acc = ws[plan.off_acc:plan.off_acc + 512 * plan.state_capacity].view(torch.float32).cpu().numpy()
    acc = acc.reshape(-1, 128)
    S, G = plan.num_splits, plan.group
    for h in range(8):
        for s in range(1, S):
            for g in range(G):
                st = ((0 * 8 + h) * S + s) * G + g
                assert ml[st, 0] == -np.inf and ml[st, 1] == 0 and not acc[st].any()


def test_workqueue_repeated_calls_reuse_workspace():
    tr = make_trace("b8_bimodal", 6, steps=3)
    ws = None
    for t in range(3):
        step = Step(tr, t)
        plan = step.plan(WQ, 16)
        if ws is None:
            ws = pkv.alloc_workspace(plan.ws_bytes * 2)
        out, _, status = step.run(plan, ws)
        assert status == 0
        assert_close(out, step.reference(), f"repeat step {t}")


def test_python_decode_api():
    step = Step(make_trace("b8_zipf", 9, steps=1), 0)
    out = pkv.decode(step.q, step.k, step.v, step.bt, step.lens, seq_lens_host=step.lens_host)
    torch.cuda.synchronize()
    assert_close(out, step.reference(), "pkv.decode")


# ------------------------------------------------------------------------------------------- device-side checks
def test_bad_block_table_entry_sets_status():
    step = Step(make_trace("tiny", 1), 0, poison=False)
    step.bt[0, 3] = step.tr.num_pages + 5
    for variant in (SPLIT, WQ, SINGLE):
        out, ws, status = step.run(step.plan(variant, 8))
        assert status & pkv.PKV_STATUS_BAD_PAGE
        assert pkv.pkv_read_status(ws) == 0  # reading clears it


def test_bad_length_sets_status():
    step = Step(make_trace("tiny", 1), 0, poison=False)
    plan = step.plan(WQ, 8)
    step.lens[0] = step.tr.max_pages * 16 + 1
    out, ws, status = step.run(plan)
    assert status & pkv.PKV_STATUS_BAD_LEN
    plan = step.plan(SPLIT, 8)
    out, ws, status = step.run(plan)
    assert status & pkv.PKV_STATUS_BAD_LEN


def test_api_rejects_bad_arguments_before_launch():
    step = Step(make_trace("tiny", 1), 0)
    plan = step.plan(SPLIT, 8)
    ws = pkv.alloc_workspace(plan.ws_bytes)
    out = torch.empty_like(step.q)
    small = pkv.alloc_workspace(plan.ws_bytes // 2)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_step(plan, step.problem, step.q, step.k, step.v, step.bt, step.lens, step.scale, small, out)
    assert e.value.code == -4
    other = pkv.make_problem(1, 32, 8, 128, 16, 65, 32)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_step(plan, other, step.q, step.k, step.v, step.bt, step.lens, step.scale, ws, out)
    assert e.value.code == -1
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_build_worklist(plan, step.problem, step.lens, ws)  # a split plan has no worklist
    assert e.value.code == -1
    mis = torch.empty(step.q.numel() + 8, dtype=torch.float16, device="cuda")[1:1 + step.q.numel()].view_as(step.q)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_step(plan, step.problem, mis, step.k, step.v, step.bt, step.lens, step.scale, ws, out)
    assert e.value.code == -5
    plan.flags = 0x4  # no such flag
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_decode_step(plan, step.problem, step.q, step.k, step.v, step.bt, step.lens, step.scale, ws, out)
    assert e.value.code == -1


# ------------------------------------------------------------------------------------------- fused vs separate merge
def _with_merge(plan, fused: int):
    plan.fuse_merge = fused
    return plan


@pytest.mark.parametrize("name,seed,t", [
    ("tiny", 3, 0), ("b1_bucketed", 7, 40), ("b8_bimodal", 8, 12), ("b8_uniform", 9, 63), ("b8_zipf", 6, 5),
    ("b4_bimodal", 7, 30),
])
def test_fused_and_separate_merge_match_oracle(name, seed, t):
    """Every config: the merge fused into the decode's last task and the separate merge kernel both match the
    oracle, for the rectangular split grid and the workqueue, at several split sizes."""
    tr = make_trace(name, seed, steps=t + 1)
    step = Step(tr, t)
    ref = step.reference()
    pmax = int(tr.pages(t).max())
    outs = []
    for variant, chunk in ((SPLIT, 1), (SPLIT, max(1, -(-pmax // 19))), (WQ, 2), (WQ, 16), (WQ, 64)):
        for fused in (1, 0):
            for in_decode in ((1, 0) if variant == WQ else (0,)):
                plan = _with_merge(step.plan(variant, chunk), fused)
                plan.list_in_decode = in_decode
                assert pkv.pkv_plan_launches(plan) == 1 + (1 - fused) + (variant == WQ and not in_decode)
                out, _, status = step.run(plan)
                assert status == 0, status
                assert_close(out, ref, f"{name} seed {seed} step {t} variant {variant} c={chunk} fused={fused} "
                                       f"list_in_decode={in_decode}")
                outs.append(out.float())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() < 2e-3


def test_workqueue_decode_runs_twice_on_one_build():
    """The last CTA to finish claiming re-arms the queue head, so a second pkv_decode on the same list repeats the
    step (fused merge: the arrival counters are back at zero as well)."""
    step = Step(make_trace("b8_bimodal", 5, steps=1), 0)
    ref = step.reference()
    plan = step.plan(WQ, 8)
    plan.list_in_decode = 0  # run the builder's list
    plan.fuse_merge = 1      # pkv_decode writes out itself
    ws = pkv.alloc_workspace(plan.ws_bytes)
    pkv.pkv_build_worklist(plan, step.problem, step.lens, ws)
    for call in range(3):
        out = torch.full_like(step.q, float("nan"))
        pkv.pkv_decode(plan, step.problem, step.q, step.k, step.v, step.bt, step.lens, step.scale, ws, out)
        torch.cuda.synchronize()
        assert_close(out, ref, f"decode call {call} on one build")
    assert pkv.pkv_read_status(ws) == 0
    hdr = ws[:16].view(torch.int32).cpu().numpy()
    assert hdr[0] == 0 and hdr[3] == 0  # queue head and finished-CTA count re-armed
    counters = ws[plan.off_counters:plan.off_counters + 4 * 64].view(torch.int32).cpu().numpy()
    assert not counters.any()


def test_rows_longer_than_the_plan_raise_the_tasks_status():
    """A plan made from shorter lengths than the device holds: the split grid's last split and the workqueue list
    cannot cover the grown row, and both say so in the status word instead of returning silently."""
    step = Step(_Lens([100, 300]).trace, 0)
    short = np.array([100, 250], dtype=np.int32)
    for variant in (SPLIT, WQ):
        plan = pkv.pkv_plan_fixed(step.problem, short, step.sms, variant, 4)
        _, ws, status = step.run(plan)
        assert status & pkv.PKV_STATUS_TASKS, (variant, status)
    # the same plans on lengths they cover are clean
    step2 = Step(_Lens([100, 250]).trace, 0)
    for variant in (SPLIT, WQ):
        plan = pkv.pkv_plan_fixed(step2.problem, short, step2.sms, variant, 4)
        out, _, status = step2.run(plan)
        assert status == 0
        assert_close(out, step2.reference(), f"covered lengths, variant {variant}")


def test_all_rows_empty_write_zero_outputs():
    step = Step(_Lens([0, 0, 0]).trace, 0)
    for variant in (SINGLE, SPLIT, WQ):
        for fused in (1, 0):
            plan = _with_merge(step.plan(variant, 2), fused if variant != SINGLE else 0)
            out, _, status = step.run(plan)
            assert status == 0 and not out.isnan().any() and not out.any(), (variant, fused)


@pytest.mark.parametrize("name,seed,chunk", [("b8_zipf", 5, 3), ("b8_uniform", 6, 16), ("stress", 5, 64),
                                             ("tiny", 0, 1)])
def test_list_derived_in_decode_matches_the_builder(name, seed, chunk):
    """With list_in_decode the decode kernel publishes the same row offsets, split counts and task count as the
    worklist builder (bit-exact), and both runs of the list give the oracle's output."""
    tr = make_trace(name, seed, steps=1)
    step = Step(tr, 0, poison=False)
    plan = step.plan(WQ, chunk)
    if tr.batch > pkv.PKV_MAX_ROWS_IN_DECODE:
        pytest.skip("B above the in-decode row limit")
    assert plan.list_in_decode == 1
    _, ws, status = step.run(plan)
    assert status == 0
    B = tr.batch
    got_off = ws[plan.off_row_off:plan.off_row_off + 4 * B].view(torch.int32).cpu().numpy()
    got_spl = ws[plan.off_row_splits:plan.off_row_splits + 4 * B].view(torch.int32).cpu().numpy()
    count = int(ws[:8].view(torch.int32).cpu().numpy()[1])
    built = pkv.alloc_workspace(plan.ws_bytes)
    pkv.pkv_build_worklist(plan, step.problem, step.lens, built)
    _, off, spl, _ = read_worklist(plan, built)
    assert np.array_equal(got_off, off) and np.array_equal(got_spl, spl)
    assert count == len(oracle.worklist(step.lens_host, 16, tr.hkv, chunk))


# ------------------------------------------------------------------------------------------- fused KV append
@pytest.mark.parametrize("name,seed,t", [("tiny", 0, 0), ("b8_bimodal", 5, 7), ("b1_bucketed", 9, 20),
                                         ("b8_zipf", 6, 3), ("b4_bimodal", 8, 16)])
def test_fused_kv_append_matches_oracle_and_fills_the_slot(name, seed, t):
    """pkv_decode_step_append with the new token's K/V only in k_new / v_new (its pool slots hold NaN): the output
    matches the oracle on the full pools and the slots end up holding the token bit for bit, for every schedule and
    both merges (t = 16 on B4 / t = 0 on tiny put the new token in a full page, others in a partial one)."""
    tr = make_trace(name, seed, steps=t + 1)
    step = Step(tr, t, poison=False)
    ref = step.reference()
    B = tr.batch
    rows = torch.arange(B)
    L = torch.from_numpy(step.lens_host.astype(np.int64))
    phys = step.bt.cpu()[rows, (L - 1) // 16].cuda().long()
    slot = ((L - 1) % 16).cuda()
    k_new = step.k[phys, slot].clone()
    v_new = step.v[phys, slot].clone()
    pmax = int(tr.pages(t).max())
    plans = [(SINGLE, 1, 0), (SPLIT, max(1, -(-pmax // 8)), 0), (SPLIT, max(1, -(-pmax // 8)), 1), (WQ, 4, 0),
             (WQ, 16, 1)]
    for variant, chunk, fused in plans:
        step.k[phys, slot] = float("nan")
        step.v[phys, slot] = float("nan")
        plan = step.plan(variant, chunk)
        if variant != SINGLE:
            plan.fuse_merge = fused
        ws = pkv.alloc_workspace(plan.ws_bytes)
        out = torch.full_like(step.q, float("nan"))
        pkv.pkv_decode_step_append(plan, step.problem, step.q, k_new, v_new, step.k, step.v, step.bt, step.lens,
                                   step.scale, ws, out)
        torch.cuda.synchronize()
        assert pkv.pkv_read_status(ws) == 0
        assert_close(out, ref, f"{name} append variant {variant} c={chunk} fused={fused}")
        assert torch.equal(step.k[phys, slot].view(torch.int16), k_new.view(torch.int16))
        assert torch.equal(step.v[phys, slot].view(torch.int16), v_new.view(torch.int16))


def test_exact_length_bucket_schedule_matches_oracle():
    """The exact-length-bucket comparison schedule (one split grid + merge per distinct length, rows sorted by
    length) computes the same attention."""
    from serving_paged_gqa_gb300 import schedules

    step = Step(_Lens([40, 300, 40, 17, 300, 0, 1000, 17]).trace, 0)
    ref = step.reference()
    order = np.argsort(step.lens_host, kind="stable")
    idx = torch.from_numpy(order).cuda()
    sched = schedules.ExactLengthBuckets(pkv, step.problem, step.lens_host[order], step.sms)
    assert sched.launches() == 2 * 4  # lengths 17, 40, 300, 1000
    ws = pkv.alloc_workspace(sched.ws_bytes)
    out = torch.full_like(step.q, float("nan"))
    sched.run(step.q[idx].contiguous(), step.k, step.v, step.bt[idx].contiguous(), step.lens[idx].contiguous(),
              step.scale, ws, out)
    torch.cuda.synchronize()
    assert pkv.pkv_read_status(ws) == 0
    assert_close(out, ref[order], "exact-length buckets")


# ------------------------------------------------------------------------------------------- serving step
@pytest.mark.parametrize("name,seed,t", [("b8_bimodal", 6, 9), ("b1_bucketed", 5, 3), ("tiny", 1, 0)])
def test_serve_step_from_host_memory_matches_oracle(name, seed, t):
    """pkv_serve_step: the packed host input (q, new K/V, block table, lengths) goes to the device, the step runs
    with the append fused, and out comes back into pinned host memory; it matches the oracle, the new token's slots
    hold its K/V, the plan is pkv_plan's, a workspace smaller than the plan is refused before anything runs, and a
    ServeStep run twice matches the oracle each time (bit-identical for static plans; a workqueue's dynamic claims
    change which consumer warp combines which page, hence the rounding)."""
    tr = make_trace(name, seed, steps=t + 1)
    step = Step(tr, t, poison=False)
    ref = step.reference()
    B, Hq, Hkv, d = tr.batch, tr.hq, tr.hkv, tr.d
    rows = torch.arange(B)
    L = torch.from_numpy(step.lens_host.astype(np.int64))
    phys = step.bt.cpu()[rows, (L - 1) // 16].cuda().long()
    slot = ((L - 1) % 16).cuda()
    k_new = step.k[phys, slot].clone()
    v_new = step.v[phys, slot].clone()
    step.k[phys, slot] = float("nan")
    step.v[phys, slot] = float("nan")
    offs, total = pkv.pkv_step_input_layout(step.problem)
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for i, part in enumerate((step.q.cpu(), k_new.cpu(), v_new.cpu(), torch.from_numpy(step.bt_host),
                              torch.from_numpy(step.lens_host))):
        raw = part.contiguous().view(torch.uint8).reshape(-1)
        host_in[offs[i]:offs[i] + raw.numel()] = raw
    dev_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    dev_out = torch.empty((B, Hq, d), dtype=torch.float16, device="cuda")
    host_out = torch.full((B, Hq, d), float("nan"), dtype=torch.float16).pin_memory()
    want = step.plan()
    small = pkv.alloc_workspace(256)
    with pytest.raises(pkv.PkvError) as err:
        pkv.pkv_serve_step(step.problem, host_in, dev_in, step.k, step.v, step.scale, small, dev_out, host_out)
    assert err.value.code == -4 and torch.isnan(host_out.float()).all()  # PKV_E_WS_TOO_SMALL, nothing ran
    ws = pkv.alloc_workspace(want.ws_bytes)
    plan = pkv.pkv_serve_step(step.problem, host_in, dev_in, step.k, step.v, step.scale, ws, dev_out, host_out)
    torch.cuda.synchronize()
    assert pkv.pkv_read_status(ws) == 0
    assert (plan.variant, plan.chunk_pages, plan.num_tasks, plan.fuse_merge) == \
        (want.variant, want.chunk_pages, want.num_tasks, want.fuse_merge)
    assert_close(host_out.cuda(), ref, f"{name} serve step")
    assert torch.equal(step.k[phys, slot].view(torch.int16), k_new.view(torch.int16))
    assert torch.equal(step.v[phys, slot].view(torch.int16), v_new.view(torch.int16))
    # ordinary (pageable) host buffers: the input and out go through cudaMemcpyAsync instead of the GPU's own loads
    # and stores
    pageable_out = torch.full((B, Hq, d), float("nan"), dtype=torch.float16)
    assert not pageable_out.is_pinned()
    pageable_in = torch.empty(host_in.shape, dtype=torch.uint8)
    pageable_in.copy_(host_in)
    assert not pageable_in.is_pinned()
    pkv.pkv_serve_step(step.problem, pageable_in, dev_in, step.k, step.v, step.scale, ws, dev_out, pageable_out)
    torch.cuda.synchronize()
    assert_close(pageable_out.cuda(), ref, f"{name} serve step, pageable host buffers")
    first = host_out.clone()
    runner = pkv.ServeStep(step.problem, host_in, dev_in, step.k, step.v, step.scale, ws, dev_out, host_out)
    for i in range(2):
        host_out.fill_(float("nan"))
        runner.run()
        torch.cuda.synchronize()
        assert_close(host_out.cuda(), ref, f"{name} ServeStep run {i}")
        if plan.variant != WQ:
            assert torch.equal(host_out.view(torch.int16), first.view(torch.int16))
    assert pkv.pkv_read_status(ws) == 0


@pytest.mark.parametrize("name,seed,t,variant,chunk,fused", [
    ("b1_bucketed", 5, 4, SPLIT, 8, 0), ("b8_bimodal", 6, 2, WQ, 16, 0), ("b8_zipf", 7, 9, WQ, 12, 1),
    ("tiny", 2, 0, SINGLE, 1, 0), ("b4_bimodal", 5, 3, SPLIT, 64, 1)])
def test_overlapping_layers_read_the_previous_layers_output(name, seed, t, variant, chunk, fused):
    """A layer loop with PKV_PLAN_OVERLAP_PREV: layer l + 1's query rows are layer l's output buffer (poisoned with
    NaN before the loop), so a step that read q before the previous layer's last kernel had finished would produce
    NaN or the wrong rows. Every layer matches the oracle run on the query rows the previous layer produced."""
    tr = make_trace(name, seed, steps=t + 1)
    step = Step(tr, t)
    plan = step.plan(variant, chunk)
    if variant != SINGLE:
        plan.fuse_merge = fused
    ws = pkv.alloc_workspace(plan.ws_bytes)
    layers = 4
    bufs = [step.q.clone()] + [torch.full_like(step.q, float("nan")) for _ in range(layers)]
    kp, vp = tr.host_pools()
    for layer in range(layers):
        plan.flags = pkv.PKV_PLAN_OVERLAP_PREV if layer else 0
        pkv.pkv_decode_step(plan, step.problem, bufs[layer], step.k, step.v, step.bt, step.lens, step.scale, ws,
                            bufs[layer + 1])
    torch.cuda.synchronize()
    assert pkv.pkv_read_status(ws) == 0
    for layer in range(layers):
        q_in = bufs[layer].cpu().numpy()
        ref = oracle.attention(q_in, kp, vp, step.bt_host, step.lens_host, step.scale)
        assert_close(bufs[layer + 1], ref, f"{name} layer {layer} variant {variant} fused {fused}")


# ------------------------------------------------------------------------------------------------ serving session
def _pack_step(problem, host_in, q, k_new, v_new, bt, lens):
    offs, _ = pkv.pkv_step_input_layout(problem)
    for i, part in enumerate((q, k_new, v_new, bt, lens)):
        raw = torch.as_tensor(np.ascontiguousarray(part)).view(torch.uint8).reshape(-1)
        host_in[offs[i]:offs[i] + raw.numel()] = raw


def _launch_key(plan):
    return tuple(getattr(plan, f) for f, _ in plan._fields_ if f not in ("predicted_us", "kv_bytes", "problem"))


def _session_loop(session, base, tr, kp, vp, host_in, host_out, steps, lens_of, bt_of, q_of=None):
    """Runs the session over `steps`; for each, the new token's pool slots are poisoned first and must hold its K/V
    afterwards, and out must match the oracle. Returns the plans."""
    B = tr.batch
    q_of = tr.q if q_of is None else q_of
    plans = []
    for t in steps:
        lens, bt, q = lens_of(t), bt_of(t), q_of(t)
        rows = np.arange(B)
        phys = bt[rows, (lens - 1) // tr.ps]
        slot = (lens - 1) % tr.ps
        k_new, v_new = kp[phys, slot], vp[phys, slot]
        pi, si = torch.from_numpy(phys.astype(np.int64)).cuda(), torch.from_numpy(slot.astype(np.int64)).cuda()
        base.k[pi, si] = float("nan")
        base.v[pi, si] = float("nan")
        _pack_step(base.problem, host_in, q, k_new, v_new, bt, lens)
        host_out.fill_(float("nan"))
        torch.cuda.synchronize()
        plan = session.run()
        torch.cuda.synchronize()
        plans.append(_launch_key(plan))
        ref = oracle.attention(q, kp, vp, bt, lens, base.scale)
        assert_close(host_out.cuda(), ref, f"session step t={t} lens={lens[:4]}")
        assert torch.equal(base.k[pi, si].cpu(), torch.from_numpy(k_new)), "new K not appended"
        assert torch.equal(base.v[pi, si].cpu(), torch.from_numpy(v_new)), "new V not appended"
    return plans


@pytest.mark.parametrize("name,seed,t0,n", [("b1_bucketed", 5, 0, 4), ("b8_bimodal", 6, 0, 6),
                                            ("b4_bimodal", 5, 10, 4), ("tiny", 1, 0, 3)])
def test_serve_session_decode_loop_replays_graphs(name, seed, t0, n):
    """A decode loop through one ServeSession (buffers bound once, host_in refilled every step): every step matches
    the oracle and appends its token; the session captures one CUDA graph per distinct plan and launches a graph on
    every step. With pageable host buffers it enqueues the launches directly (no graph) and still matches."""
    tr = make_trace(name, seed, steps=t0 + n)
    base = Step(tr, t0, poison=False)
    kp, vp = tr.host_pools()
    B, Hq, d = tr.batch, tr.hq, tr.d
    steps = list(range(t0, t0 + n))
    ws_bytes = max(pkv.pkv_plan(base.problem, tr.seq_lens(t), base.sms).ws_bytes for t in steps)
    ws = pkv.alloc_workspace(ws_bytes)
    _, total = pkv.pkv_step_input_layout(base.problem)
    dev_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    dev_out = torch.empty((B, Hq, d), dtype=torch.float16, device="cuda")
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    host_out = torch.empty((B, Hq, d), dtype=torch.float16).pin_memory()
    session = pkv.ServeSession(base.problem, host_in, dev_in, base.k, base.v, base.scale, ws, dev_out, host_out)
    plans = _session_loop(session, base, tr, kp, vp, host_in, host_out, steps, tr.seq_lens, tr.block_table)
    assert session.stats() == (len(set(plans)), n), (session.stats(), len(set(plans)))
    assert pkv.pkv_read_status(ws) == 0
    session.close()
    # pageable host buffers: no graph
    pin = torch.zeros(total, dtype=torch.uint8)
    pout = torch.empty((B, Hq, d), dtype=torch.float16)
    direct = pkv.ServeSession(base.problem, pin, dev_in, base.k, base.v, base.scale, ws, dev_out, pout)
    _session_loop(direct, base, tr, kp, vp, pin, pout, steps[:2], tr.seq_lens, tr.block_table)
    assert direct.stats() == (0, 0)
    direct.close()


def test_serve_session_evicts_the_least_recently_used_graph():
    """More distinct plans than the session keeps graphs for (B = 1 rows cut to 18 lengths, each a different split
    count): every step matches the oracle; the 17th and 18th plans evict the two oldest graphs, so rerunning the
    first length captures again while rerunning the last one replays."""
    tr = make_trace("b1_bucketed", 5, steps=1)
    base = Step(tr, 0, poison=False)
    kp, vp = tr.host_pools()
    L0 = int(tr.seq_lens(0)[0])
    cut = [np.array([L0 - 130 * k], dtype=np.int32) for k in range(pkv.PKV_SESSION_GRAPHS + 2)]
    plans = [pkv.pkv_plan(base.problem, c, base.sms) for c in cut]
    assert len({_launch_key(p) for p in plans}) == len(cut)
    ws = pkv.alloc_workspace(max(p.ws_bytes for p in plans))
    _, total = pkv.pkv_step_input_layout(base.problem)
    dev_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    dev_out = torch.empty((1, tr.hq, tr.d), dtype=torch.float16, device="cuda")
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    host_out = torch.empty((1, tr.hq, tr.d), dtype=torch.float16).pin_memory()
    session = pkv.ServeSession(base.problem, host_in, dev_in, base.k, base.v, base.scale, ws, dev_out, host_out)
    bt = tr.block_table(0)
    order = list(range(len(cut))) + [0, len(cut) - 1]
    _session_loop(session, base, tr, kp, vp, host_in, host_out, order, lambda i: cut[i], lambda i: bt,
                  lambda i: tr.q(0))
    n = len(cut)
    assert session.stats() == (n + 1, n + 2)
    assert pkv.pkv_read_status(ws) == 0
    session.close()


@pytest.mark.parametrize("name,seed,t,variant,chunk,fused", [
    ("b1_bucketed", 7, 3, None, 0, 0), ("b8_bimodal", 5, 4, None, 0, 0), ("b8_zipf", 8, 2, WQ, 12, 1),
    ("tiny", 4, 0, SINGLE, 1, 0), ("b4_bimodal", 6, 1, SPLIT, 32, 1)])
def test_inputs_written_by_the_kernel_before(name, seed, t, variant, chunk, fused):
    """PKV_PLAN_INPUTS_AFTER_PREV: q, the block table and the lengths are written by a kernel enqueued just before
    the step (their buffers poisoned first: NaN query rows, a block table of -1, zero lengths), and the step, which
    may start while that kernel runs, must read them only after it: the output matches the oracle, no status."""
    tr = make_trace(name, seed, steps=t + 1)
    step = Step(tr, t)
    plan = step.plan() if variant is None else step.plan(variant, chunk)
    if plan.variant != SINGLE:
        plan.fuse_merge = fused
    plan.flags = pkv.PKV_PLAN_INPUTS_AFTER_PREV
    ws = pkv.alloc_workspace(plan.ws_bytes)
    q = torch.full_like(step.q, float("nan"))
    bt = torch.full_like(step.bt, -1)
    lens = torch.zeros_like(step.lens)
    out = torch.full_like(step.q, float("nan"))
    for i in range(2):
        torch.cuda.synchronize()
        torch.add(step.q, 0, out=q)  # kernels (not copies), the last one immediately before the step
        torch.add(step.bt, 0, out=bt)
        torch.add(step.lens, 0, out=lens)
        pkv.pkv_decode_step(plan, step.problem, q, step.k, step.v, bt, lens, step.scale, ws, out)
        torch.cuda.synchronize()
        assert_close(out, step.reference(), f"{name} inputs after the kernel before, run {i}")
        assert pkv.pkv_read_status(ws) == 0
        q.fill_(float("nan"))
        bt.fill_(-1)
        lens.zero_()
        out.fill_(float("nan"))


def test_serve_session_inside_a_callers_capture():
    """A ServeSession step run while the caller captures the stream (torch.cuda.graph): the session enqueues the
    launches into the caller's capture instead of its own graph (its counters do not move), and replaying the caller's
    graph computes the step: out in host memory matches the oracle, the new token's K/V is appended."""
    tr = make_trace("b8_bimodal", 5, steps=1)
    base = Step(tr, 0, poison=False)
    kp, vp = tr.host_pools()
    B, Hq, d = tr.batch, tr.hq, tr.d
    lens, bt = tr.seq_lens(0), tr.block_table(0)
    ws = pkv.alloc_workspace(pkv.pkv_plan(base.problem, lens, base.sms).ws_bytes)
    _, total = pkv.pkv_step_input_layout(base.problem)
    dev_in = torch.empty(total, dtype=torch.uint8, device="cuda")
    dev_out = torch.empty((B, Hq, d), dtype=torch.float16, device="cuda")
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    host_out = torch.empty((B, Hq, d), dtype=torch.float16).pin_memory()
    session = pkv.ServeSession(base.problem, host_in, dev_in, base.k, base.v, base.scale, ws, dev_out, host_out)
    # one ordinary step first (the session captures its own graph of this plan)
    _session_loop(session, base, tr, kp, vp, host_in, host_out, [0], tr.seq_lens, tr.block_table)
    assert session.stats() == (1, 1)
    rows = np.arange(B)
    phys, slot = bt[rows, (lens - 1) // tr.ps], (lens - 1) % tr.ps
    pi, si = torch.from_numpy(phys.astype(np.int64)).cuda(), torch.from_numpy(slot.astype(np.int64)).cuda()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        session.run(s)
    assert session.stats() == (1, 1)
    base.k[pi, si] = float("nan")
    base.v[pi, si] = float("nan")
    host_out.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.attention(tr.q(0), kp, vp, bt, lens, base.scale)
    assert_close(host_out.cuda(), ref, "session step replayed from the caller's graph")
    assert torch.equal(base.k[pi, si].cpu(), torch.from_numpy(kp[phys, slot]))
    assert pkv.pkv_read_status(ws) == 0
    session.close()


@pytest.mark.parametrize("B", [pkv.PKV_MAX_ROWS_IN_DECODE, pkv.PKV_MAX_ROWS_IN_DECODE + 1, pkv.PKV_MAX_BATCH])
def test_batch_limits(B):
    """The largest batch whose workqueue the decode derives itself (256 rows), the first one that runs the worklist
    builder (257) and the largest batch the library takes (4096): seeded lengths of 0 to 200 tokens (empty rows,
    partial and exact pages); the policy's plan (the single pass, for rows this short) and the workqueue with the
    fused merge both match the oracle, the builder's list is bit-exact, no status."""
    r = rng_for(B, 777)
    lens = r.integers(0, 201, size=B)
    lens[::17] = 0
    lens[1::23] = 16
    step = Step(_Lens(lens, seed=B).trace, 0)
    ref = step.reference()
    plan = step.plan()  # short rows: the single pass
    out, ws, status = step.run(plan)
    assert status == 0
    assert_close(out, ref, f"B={B} policy plan {plan.describe()}")
    wq = step.plan(WQ, 4)
    assert wq.list_in_decode == (1 if B <= pkv.PKV_MAX_ROWS_IN_DECODE else 0)
    wq.fuse_merge = 1
    out, ws, status = step.run(wq)
    assert status == 0
    assert_close(out, ref, f"B={B} workqueue, fused merge")
    if not wq.list_in_decode:
        got, _, _, _ = read_worklist(wq, ws)
        want = oracle.worklist(step.lens_host, 16, step.tr.hkv, 4)
        assert got.shape == want.shape and np.array_equal(got, want)
