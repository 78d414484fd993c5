"""The C-ABI library on the CPU: it loads, exports every declared symbol, and its host-only logic is right.

No call here touches the GPU: only pkv_version, pkv_strerror, pkv_check_problem, pkv_policy_default, pkv_plan,
pkv_plan_fixed and pkv_plan_launches run; they are host code.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import serving_paged_gqa_gb300 as pkv
from serving_paged_gqa_gb300 import _lib
from workloads import make_trace

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from serving_paged_gqa_gb300 import build

    build.build()


def _declared():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|void|const char\*)\s+(pkv_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol():
    lib = ctypes.CDLL(_lib.LIB_PATH)
    names = _declared()
    assert len(names) >= 13
    assert sorted(_lib.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_errors():
    assert pkv.pkv_version() == 3
    assert "null" in pkv.pkv_strerror(-3)
    assert pkv.pkv_strerror(0) == "ok"


def _problem(B=8, Hq=32, Hkv=8, d=128, ps=16, num_pages=1 << 16, max_pages=2100):
    return pkv.make_problem(B, Hq, Hkv, d, ps, num_pages, max_pages)


def test_check_problem():
    assert pkv.pkv_check_problem(_problem()) == 0
    assert pkv.pkv_check_problem(_problem(d=64)) == -2
    assert pkv.pkv_check_problem(_problem(ps=32)) == -2
    assert pkv.pkv_check_problem(_problem(Hq=32, Hkv=6)) == -2  # Hq % Hkv != 0
    assert pkv.pkv_check_problem(_problem(Hq=96, Hkv=2)) == -2  # G = 48 unsupported
    assert pkv.pkv_check_problem(_problem(B=-1)) == -1
    assert pkv.pkv_check_problem(_problem(B=5000)) == -2


def test_plan_fixed_counts_match_oracle_worklist():
    tr = make_trace("b8_bimodal", 5, steps=3)
    lens = tr.seq_lens(2)
    pr = _problem(max_pages=tr.max_pages)
    for c in (1, 4, 32, 100):
        wq = pkv.pkv_plan_fixed(pr, lens, 152, pkv.PKV_VARIANT_WORKQUEUE, c)
        assert wq.num_tasks == len(oracle.worklist(lens, 16, 8, c))
        assert wq.task_capacity == wq.num_tasks and wq.state_capacity == 4 * wq.num_tasks
        sp = pkv.pkv_plan_fixed(pr, lens, 152, pkv.PKV_VARIANT_SPLIT, c)
        S = max(-(-(-(-int(L) // 16)) // c) for L in lens)
        assert sp.num_splits == S and sp.num_tasks == 8 * 8 * S
        for pl in (wq, sp):
            assert pl.grid_ctas == min(pl.num_tasks, 2 * 152)
            offs = [pl.off_counters, pl.off_row_off, pl.off_row_splits, pl.off_tasks, pl.off_ml, pl.off_acc,
                    pl.ws_bytes]
            assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
            assert pl.off_acc + 4 * 128 * pl.state_capacity <= pl.ws_bytes
            assert pl.off_counters == 256 and pl.off_counters + 4 * 8 * 8 <= pl.off_row_off
            assert abs(pl.kv_bytes - (4096 * int(lens.sum()) + 16384 * 8)) < 1
            assert pl.fuse_merge in (0, 1)
        # the workqueue derives its list inside the decode (B <= PKV_MAX_ROWS_IN_DECODE) and merges in its last
        # tasks: one launch per step; the separate merge kernel and the builder each add one
        wq.fuse_merge = sp.fuse_merge = 1
        assert wq.list_in_decode == 1 and sp.list_in_decode == 0
        assert pkv.pkv_plan_launches(wq) == 1 and pkv.pkv_plan_launches(sp) == 1
        wq.fuse_merge = 0
        sp.fuse_merge = 0
        assert pkv.pkv_plan_launches(wq) == 2 and pkv.pkv_plan_launches(sp) == 2
        wq.list_in_decode = 0
        assert pkv.pkv_plan_launches(wq) == 3
    single = pkv.pkv_plan_fixed(pr, lens, 152, pkv.PKV_VARIANT_SINGLE)
    assert single.num_tasks == 64 and single.num_splits == 1 and single.state_capacity == 0
    assert single.fuse_merge == 0 and pkv.pkv_plan_launches(single) == 1


def test_grid_is_one_wave_of_resident_ctas():
    """The persistent grid never holds more CTAs than the SMs' registers and shared memory keep resident: two per SM
    for group sizes up to 8, one for G = 16, whose per-CTA shared memory is above half of an SM's 228 KB."""
    lens = np.full(8, 20000, dtype=np.int32)
    for hq, hkv, per_sm in ((32, 8, 2), (32, 32, 2), (64, 8, 2), (128, 8, 1), (16, 1, 1)):
        pr = pkv.make_problem(8, hq, hkv, 128, 16, 1 << 16, 2048)
        pl = pkv.pkv_plan_fixed(pr, lens, 152, pkv.PKV_VARIANT_WORKQUEUE, 4)
        assert pl.grid_ctas == min(pl.num_tasks, per_sm * 152), (hq, hkv, pl.grid_ctas)
        pl = pkv.pkv_plan_fixed(pr, lens, 152, pkv.PKV_VARIANT_SPLIT, 4, ctas_per_sm=4)
        assert pl.grid_ctas == min(pl.num_tasks, per_sm * 152)


def test_plan_rejects_bad_input():
    pr = _problem(B=2, max_pages=4)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_plan_fixed(pr, [10, 65], 152, pkv.PKV_VARIANT_SPLIT, 2)  # 65 > 4 pages * 16
    with pytest.raises(pkv.PkvError):
        pkv.pkv_plan_fixed(pr, [10, 20], 152, pkv.PKV_VARIANT_SPLIT, 0)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_plan_fixed(pr, [10, 20], 0, pkv.PKV_VARIANT_SPLIT, 1)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_plan_fixed(pr, [10, 20], 152, 7, 1)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_plan(pr, [-1, 20], 152)


def test_plan_picks_the_model_minimum():
    """pkv_plan's choice has the lowest predicted time among all fixed plans it could have made."""
    for name, seed in (("b1_bucketed", 5), ("b8_bimodal", 6), ("b4_bimodal", 7), ("b8_zipf", 8), ("tiny", 0)):
        tr = make_trace(name, seed, steps=1)
        lens = tr.seq_lens(0)
        pr = _problem(B=tr.batch, max_pages=tr.max_pages, num_pages=tr.num_pages)
        best = pkv.pkv_plan(pr, lens, 152)
        pmax = int(tr.pages(0).max())
        cands = [pkv.pkv_plan_fixed(pr, lens, 152, pkv.PKV_VARIANT_SINGLE)]
        # the split grid is a candidate only for small batches (pkv_policy.split_max_batch)
        variants = (pkv.PKV_VARIANT_SPLIT, pkv.PKV_VARIANT_WORKQUEUE) if tr.batch <= 2 else (pkv.PKV_VARIANT_WORKQUEUE,)
        for v in variants:
            for c in range(max(1, -(-pmax // 256)), pmax + 1):
                cands.append(pkv.pkv_plan_fixed(pr, lens, 152, v, c))
        low = min(c.predicted_us for c in cands)
        # the planner searches a subset of split sizes; it may not beat the full sweep, and must be close to it
        assert best.predicted_us >= low - 1e-9
        assert best.predicted_us <= low * 1.15


def test_list_in_decode_only_up_to_its_row_limit():
    lens = np.full(300, 100, dtype=np.int32)
    for B, expect in ((pkv.PKV_MAX_ROWS_IN_DECODE, 1), (pkv.PKV_MAX_ROWS_IN_DECODE + 1, 0)):
        pl = pkv.pkv_plan_fixed(_problem(B=B, max_pages=8), lens[:B], 152, pkv.PKV_VARIANT_WORKQUEUE, 2)
        assert pl.list_in_decode == expect


def test_empty_batch_and_empty_rows_plan():
    pr = _problem(B=3, max_pages=8)
    pl = pkv.pkv_plan_fixed(pr, [0, 0, 0], 152, pkv.PKV_VARIANT_WORKQUEUE, 2)
    assert pl.num_tasks == 0
    pl = pkv.pkv_plan_fixed(pr, [0, 17, 0], 152, pkv.PKV_VARIANT_WORKQUEUE, 1)
    assert pl.num_tasks == 8 * 2
    pl = pkv.pkv_plan(_problem(B=0, max_pages=1), np.zeros(0, np.int32), 152)
    assert pl.num_tasks == 0


def test_calibration_model_mirrors_the_planner():
    """The calibration tool fits the constants of the same formula the planner evaluates: for every candidate plan
    of a few steps, its Python mirror reproduces pkv_plan_fixed's predicted step time, and pkv_plan returns the
    candidate the mirror ranks cheapest."""
    from serving_paged_gqa_gb300 import calibrate

    consts = calibrate.policy_constants(pkv)
    for name, seed in (("b1_bucketed", 5), ("b8_bimodal", 6), ("b8_zipf", 8), ("tiny", 0), ("stress", 5)):
        tr = make_trace(name, seed, steps=1)
        lens = tr.seq_lens(0)
        pr = _problem(B=tr.batch, max_pages=tr.max_pages, num_pages=tr.num_pages)
        best = None
        for pl in calibrate.candidates(pkv, pr, lens, 152):
            f = calibrate.features(pl, lens)
            got = calibrate.predict(consts, f)
            if pl.fuse_merge == pkv.pkv_plan_fixed(pr, lens, 152, pl.variant, pl.chunk_pages).fuse_merge:
                assert abs(got - pl.predicted_us) <= 1e-9 * max(1.0, got), (name, pl.describe())
            if calibrate.policy_candidate(f):
                best = got if best is None else min(best, got)
        chosen = pkv.pkv_plan(pr, lens, 152)
        assert chosen.predicted_us <= best * (1 + 1e-12)


def test_step_input_layout_parts_are_aligned_and_disjoint():
    """The packed serving input: q, k_new, v_new, block table, lengths, each on a 256-byte boundary, in that order,
    each part as large as its tensor."""
    B, Hq, Hkv, d, maxp = 5, 32, 8, 128, 37
    pr = pkv.make_problem(B, Hq, Hkv, d, 16, 1000, maxp)
    offs, total = pkv.pkv_step_input_layout(pr)
    sizes = [B * Hq * d * 2, B * Hkv * d * 2, B * Hkv * d * 2, B * maxp * 4, B * 4]
    assert offs[0] == 0 and all(o % 256 == 0 for o in offs) and total % 256 == 0
    for i in range(4):
        assert offs[i] + sizes[i] <= offs[i + 1] < offs[i] + sizes[i] + 256
    assert offs[4] + sizes[4] <= total < offs[4] + sizes[4] + 256
    with pytest.raises(pkv.PkvError):
        pkv.pkv_step_input_layout(pkv.make_problem(5, 32, 8, 64, 16, 1000, maxp))  # d = 64 unsupported


def test_serve_step_rejects_missing_buffers_before_any_work():
    """pkv_serve_step returns an error code for null buffers without touching the device."""
    lib = pkv.load()
    pr = pkv.make_problem(1, 32, 8, 128, 16, 64, 32)
    plan = pkv.Plan()
    rc = lib.pkv_serve_step(ctypes.byref(pr), None, 152, None, None, None, None, ctypes.c_float(0.1), None, 0, None,
                            None, None, ctypes.byref(plan))
    assert rc == -3  # PKV_E_NULLPTR


def test_session_rejects_bad_arguments_before_any_work():
    """pkv_session_create / _step / _stats / _destroy: error codes for missing or misaligned buffers, a missing
    handle and a non-positive SM count, with nothing created (the handle stays NULL) and no device call."""
    lib = pkv.load()
    pr = pkv.make_problem(1, 32, 8, 128, 16, 64, 32)
    h = ctypes.c_void_p(1)
    f32 = ctypes.c_float(0.1)
    vp = ctypes.c_void_p
    a256, a16 = vp(1 << 20), vp((1 << 20) + 16)  # aligned stand-ins, never dereferenced: validation fails first
    assert lib.pkv_session_create(ctypes.byref(pr), None, 152, None, a256, a256, a256, f32, a256, 1 << 20, a256,
                                  a256, ctypes.byref(h)) == -3  # PKV_E_NULLPTR (host_in)
    assert h.value is None
    assert lib.pkv_session_create(ctypes.byref(pr), None, 152, a256, a16, a256, a256, f32, a256, 1 << 20, a256,
                                  a256, ctypes.byref(h)) == -5  # PKV_E_ALIGN (dev_in not 256-byte aligned)
    assert lib.pkv_session_create(ctypes.byref(pr), None, 152, vp((1 << 20) + 8), a256, a256, a256, f32, a256,
                                  1 << 20, a256, a256, ctypes.byref(h)) == -5  # host_in not 16-byte aligned
    assert lib.pkv_session_create(ctypes.byref(pr), None, 0, a256, a256, a256, a256, f32, a256, 1 << 20, a256,
                                  a256, ctypes.byref(h)) == -1  # PKV_E_INVAL (num_sms)
    assert lib.pkv_session_create(ctypes.byref(pr), None, 152, a256, a256, a256, a256, f32, a256, 1 << 20, a256,
                                  a256, None) == -3
    bad = pkv.make_problem(1, 32, 8, 64, 16, 64, 32)  # d = 64
    assert lib.pkv_session_create(ctypes.byref(bad), None, 152, a256, a256, a256, a256, f32, a256, 1 << 20, a256,
                                  a256, ctypes.byref(h)) == -2  # PKV_E_UNSUPPORTED
    plan = pkv.Plan()
    assert lib.pkv_session_step(None, None, ctypes.byref(plan)) == -3
    n1, n2 = ctypes.c_int64(), ctypes.c_int64()
    assert lib.pkv_session_stats(None, ctypes.byref(n1), ctypes.byref(n2)) == -3
    assert lib.pkv_session_destroy(None) == 0


def test_session_with_an_empty_batch_runs_without_the_device():
    """A B = 0 session: create, a step (the plan has no task, nothing is enqueued), stats and destroy all succeed
    with no device work, and no graph is captured."""
    lib = pkv.load()
    pr = pkv.make_problem(0, 32, 8, 128, 16, 64, 32)
    vp = ctypes.c_void_p
    a256 = vp(1 << 20)  # aligned stand-ins: with no rows nothing is read or written
    h = vp()
    assert lib.pkv_session_create(ctypes.byref(pr), None, 152, a256, a256, a256, a256, ctypes.c_float(0.1), a256,
                                  1 << 20, a256, a256, ctypes.byref(h)) == 0
    plan = pkv.Plan()
    assert lib.pkv_session_step(h, None, ctypes.byref(plan)) == 0
    assert plan.num_tasks == 0
    n1, n2 = ctypes.c_int64(-1), ctypes.c_int64(-1)
    assert lib.pkv_session_stats(h, ctypes.byref(n1), ctypes.byref(n2)) == 0
    assert (n1.value, n2.value) == (0, 0)
    assert lib.pkv_session_destroy(h) == 0


def test_policy_refinement_never_ends_worse_than_the_constants_in_force():
    """calibrate.refine on a slice of the committed calibration sweep: its result's mean regret is at most that of
    the least-squares start and of the constants in force (`also`), whichever is lower."""
    from serving_paged_gqa_gb300 import calibrate

    rows = calibrate.load_rows(os.path.join(ROOT, "serving_paged_gqa_gb300", "policy", "calibration_sweep.json"))
    rows = [r for r in rows if r["seed"] == 0]
    in_force = calibrate.policy_constants(pkv)
    lsq, _ = calibrate.fit(rows, in_force)
    groups = calibrate.step_groups(rows)
    got, stats = calibrate.refine(rows, lsq, restarts=1, also=in_force)
    best_start = min(calibrate.mean_regret(lsq, groups), calibrate.mean_regret(in_force, groups))
    assert calibrate.mean_regret(got, groups) <= best_start + 1e-12
    assert abs(stats["calibration_regret_in_force"] - calibrate.mean_regret(in_force, groups)) < 1e-12


def test_session_step_refuses_a_workspace_smaller_than_the_plan():
    """A session bound to a workspace smaller than the step's plan: pkv_session_step plans from the lengths in
    host_in, returns PKV_E_WS_TOO_SMALL and enqueues nothing (the device pointers are never used)."""
    import numpy as np

    lib = pkv.load()
    pr = pkv.make_problem(1, 32, 8, 128, 16, 1024, 512)
    offs, total = pkv.pkv_step_input_layout(pr)
    raw = np.zeros(total + 64, dtype=np.uint8)
    base = (-raw.ctypes.data) % 64
    host_in = raw[base:base + total]
    host_in[offs[4]:offs[4] + 4] = np.array([4096], dtype=np.int32).view(np.uint8)
    vp = ctypes.c_void_p
    a256 = vp(1 << 20)  # aligned stand-ins for the device buffers
    h = vp()
    assert lib.pkv_session_create(ctypes.byref(pr), None, 152, vp(host_in.ctypes.data), a256, a256, a256,
                                  ctypes.c_float(0.1), a256, 256, a256, a256, ctypes.byref(h)) == 0
    plan = pkv.Plan()
    assert lib.pkv_session_step(h, None, ctypes.byref(plan)) == -4  # PKV_E_WS_TOO_SMALL
    assert plan.ws_bytes > 256 and plan.num_tasks > 0
    n1, n2 = ctypes.c_int64(-1), ctypes.c_int64(-1)
    assert lib.pkv_session_stats(h, ctypes.byref(n1), ctypes.byref(n2)) == 0 and (n1.value, n2.value) == (0, 0)
    assert lib.pkv_session_destroy(h) == 0
