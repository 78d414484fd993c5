"""Calibration of the planner's cost model (the "calibrated roofline-style policy" of the PersistentKV v2 abstract;
gist.science technical summary, "Calibrated Adaptive Policy": thresholds fixed on calibration traces, evaluated on
held-out traces).

    python -m serving_paged_gqa_gb300.calibrate sweep --seeds 0,1,2,3,4 --out SWEEP.json      (GPU)
    python -m serving_paged_gqa_gb300.calibrate fit SWEEP.json                                 (CPU)
    python -m serving_paged_gqa_gb300.calibrate evaluate --seeds 5,6,7,8,9 --out HELDOUT.json  (GPU)
    python -m serving_paged_gqa_gb300.calibrate report HELDOUT.json                            (CPU)

sweep: for every trace family and seed, a few steps spread over the trace; for every step, every candidate plan
(single pass; the split grid and the workqueue at several split sizes, each with the separate merge and, at small
split counts, the fused merge) is timed on the device: L2 flushed before the step, a GPU spin so the step's CUDA
events measure device time only, median of three.
fit: least-squares fit (relative error) of the model's constants on the near-optimal candidates, then a refinement
that minimises the calibration steps' regret (the policy ranks candidates; least squares alone leaves several % of
regret on the multi-row traces); writes policy/constants.json and csrc/policy_constants.h (rebuild the library to
make them pkv_policy_default).
evaluate: the same sweep on held-out seeds, plus the plan pkv_plan chooses; report: per trace, the policy's regret
against the best candidate of each step and against the best single fixed plan, and the model's prediction error.

The model (include/pkv.h, pkv_policy) is mirrored by `predict` below; a CPU test checks the two agree.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
POLICY_DIR = os.path.join(HERE, "policy")
HEADER = os.path.join(HERE, "csrc", "policy_constants.h")

TRACES = ("b1_bucketed", "b8_bimodal", "b8_uniform", "b8_zipf", "b4_bimodal", "stress")
STEPS_PER_SEED = {"stress": 1}
# the planner's candidate split sizes (powers of two and 1.5x powers of two) in the ranges it uses
SPLIT_CHUNKS = (2, 3, 4, 6, 8, 12, 16, 24, 32, 48, 64, 96, 128, 192, 256)
WQ_CHUNKS = (4, 6, 8, 12, 16, 24, 32, 48, 64, 96, 128)
FUSED_MAX_SPLITS = 48   # the fused merge is timed only where its one-CTA merge can pay off
MAX_SPLITS = 1024       # the planner's default bound on splits per row
L2_FLUSH_BYTES = 256 << 20
SPIN_US = 150.0
PAGE_SIZE, TOKEN_HEAD_BYTES = 16, 512  # K + V bytes of one token of one KV head (d = 128, fp16)

CONSTANTS = ("launch_us", "hbm_gbs", "cta_gbs", "wq_cta_gbs", "task_us", "tail", "merge_us", "merge_state_us",
             "fused_us", "fused_state_us", "build_us")
# launch_us is floored at the device-side cost of one kernel launch measured on this part (about 4 us): launch and
# merge costs are otherwise collinear, since every plan the policy can pick for B > 1 has a merge
BOUNDS = {"launch_us": (4.0, 60.0), "hbm_gbs": (3000.0, 6800.0), "cta_gbs": (5.0, 200.0), "wq_cta_gbs": (5.0, 200.0),
          "task_us": (0.05, 5.0), "tail": (0.0, 3.0), "merge_us": (0.0, 20.0), "merge_state_us": (0.0, 1.0),
          "fused_us": (0.0, 40.0), "fused_state_us": (0.0, 3.0), "build_us": (0.0, 40.0)}
NEAR_OPTIMAL = 2.0     # the fit uses the candidates within this factor of their step's best time
SPLIT_MAX_BATCH = 2    # the split grid is a candidate only for B <= this (pkv_policy.split_max_batch)
SINGLE, SPLIT, WQ = 0, 1, 2


# ------------------------------------------------------------------------------------------------ the model
def features(plan, lens) -> dict:
    """What the model needs from a plan and the step's host lengths."""
    lens = np.asarray(lens, dtype=np.int64)
    p_max = int(((lens + PAGE_SIZE - 1) // PAGE_SIZE).max()) if len(lens) else 0
    return {"variant": int(plan.variant), "chunk": int(plan.chunk_pages), "splits": int(plan.num_splits),
            "tasks": int(plan.num_tasks), "grid": int(plan.grid_ctas), "group": int(plan.group),
            "fused": int(plan.fuse_merge), "in_decode": int(plan.list_in_decode), "kv_bytes": float(plan.kv_bytes),
            "p_max": p_max, "batch": int(plan.problem.batch)}


def predict(c: dict, f: dict) -> float:
    """Step time in microseconds under constants c (the formula documented with pkv_policy in include/pkv.h)."""
    T = f["tasks"]
    if T <= 0:
        return c["launch_us"]
    W = max(1, f["grid"])
    A = min(T, W)
    pages = f["p_max"] if f["variant"] == SINGLE else min(f["chunk"], f["p_max"])
    task_bytes = pages * PAGE_SIZE * TOKEN_HEAD_BYTES
    if f["variant"] == WQ:
        stream = f["kv_bytes"] / (min(c["hbm_gbs"], A * c["wq_cta_gbs"]) * 1e3)
        makespan = math.ceil(T / W) * task_bytes / (c["wq_cta_gbs"] * 1e3)
        t = c["launch_us"] + stream + (T / W) * c["task_us"] + c["tail"] * max(0.0, makespan - stream)
    else:
        share = min(c["cta_gbs"], c["hbm_gbs"] / A) * 1e3
        t = c["launch_us"] + math.ceil(T / W) * (c["task_us"] + (f["kv_bytes"] / T) / share)
    if f["variant"] != SINGLE:
        s_max = f["splits"] if f["variant"] == SPLIT else math.ceil(f["p_max"] / max(1, f["chunk"]))
        if f["fused"]:
            t += c["fused_us"] + c["fused_state_us"] * s_max * f["group"]
        else:
            t += c["merge_us"] + c["merge_state_us"] * s_max
    if f["variant"] == WQ and not f["in_decode"]:
        t += c["build_us"]
    return t


def policy_candidate(f: dict) -> bool:
    """Whether pkv_plan may choose such a plan (the split grid only for small batches)."""
    return not (f["variant"] == SPLIT and f["batch"] > SPLIT_MAX_BATCH)


def policy_constants(pkv) -> dict:
    pol = pkv.pkv_policy_default()
    return {k: float(getattr(pol, k)) for k in CONSTANTS}


def make_policy(pkv, c: dict):
    pol = pkv.pkv_policy_default()
    for k in CONSTANTS:
        setattr(pol, k, float(c[k]))
    return pol


# ------------------------------------------------------------------------------------------------ GPU sweep
def _copy(plan):
    return type(plan).from_buffer_copy(plan)


def candidates(pkv, problem, lens, sms):
    """Every plan the sweep times for one step."""
    P = (np.asarray(lens, dtype=np.int64) + PAGE_SIZE - 1) // PAGE_SIZE
    pmax = max(1, int(P.max()))
    out = [pkv.pkv_plan_fixed(problem, lens, sms, SINGLE)]
    for variant, chunks in ((SPLIT, SPLIT_CHUNKS), (WQ, WQ_CHUNKS)):
        for c in chunks:
            if c > 2 * pmax:
                break
            s_max = math.ceil(pmax / c)
            if s_max > MAX_SPLITS:
                continue
            base = pkv.pkv_plan_fixed(problem, lens, sms, variant, c)
            for fused in (0, 1):
                if fused and s_max > FUSED_MAX_SPLITS:
                    continue
                pl = _copy(base)
                pl.fuse_merge = fused
                out.append(pl)
    return out


class _Timer:
    def __init__(self, torch, dev):
        self.torch = torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.spin = int(SPIN_US * 1e-6 * 2.0e9)

    def __call__(self, fn, reps=3):
        torch = self.torch
        ev = []
        for _ in range(reps):
            self.w.zero_()
            self.sink = self.r.sum()
            torch.cuda._sleep(self.spin)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            ev.append((e0, e1))
        torch.cuda.synchronize()
        return float(np.median([a.elapsed_time(b) * 1e3 for a, b in ev]))


def _step_fn(pkv, lib, plan, problem, tensors, scale, ws, out, stream):
    vp = ctypes.c_void_p
    q, k, v, bt, sl = tensors
    st = vp(stream.cuda_stream)
    args = (ctypes.byref(plan), ctypes.byref(problem), vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()),
            vp(bt.data_ptr()), vp(sl.data_ptr()), ctypes.c_float(scale), vp(ws.data_ptr()), ws.numel(),
            vp(out.data_ptr()), st)

    def fn():
        rc = lib.pkv_decode_step(*args)
        if rc != 0:
            raise RuntimeError(f"pkv_decode_step failed: {rc}")
    return fn


def sweep(seeds, traces=TRACES, with_policy=False, log=print):
    """Times every candidate plan on a few steps of every trace and seed; returns a list of measurement rows."""
    import torch

    sys.path.insert(0, ROOT)
    import serving_paged_gqa_gb300 as pkv
    from workloads import make_trace

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    lib = pkv.load()
    timer = _Timer(torch, dev)
    stream = torch.cuda.current_stream(dev)
    consts = policy_constants(pkv)
    rows = []
    for name in traces:
        for seed in seeds:
            t0 = time.time()
            tr = make_trace(name, seed)
            k = torch.empty((tr.num_pages, tr.ps, tr.hkv, tr.d), dtype=torch.float16, device=dev)
            v = torch.empty_like(k)
            idx = torch.from_numpy(tr.used_pages).to(dev)
            k.index_copy_(0, idx, torch.from_numpy(tr.k_pages).to(dev))
            v.index_copy_(0, idx, torch.from_numpy(tr.v_pages).to(dev))
            problem = pkv.make_problem(tr.batch, tr.hq, tr.hkv, tr.d, tr.ps, tr.num_pages, tr.max_pages)
            scale = 1.0 / math.sqrt(tr.d)
            n_steps = STEPS_PER_SEED.get(name, 6)
            for t in [(i * tr.steps) // n_steps for i in range(n_steps)]:
                lens = tr.seq_lens(t)
                tensors = (torch.from_numpy(tr.q(t)).to(dev), k, v, torch.from_numpy(tr.block_table(t)).to(dev),
                           torch.from_numpy(lens).to(dev))
                cands = candidates(pkv, problem, lens, sms)
                chosen = None
                if with_policy:
                    chosen = pkv.pkv_plan(problem, lens, sms)
                    cands.append(chosen)
                ws = pkv.alloc_workspace(max(p.ws_bytes for p in cands), dev)
                out = torch.empty((tr.batch, tr.hq, tr.d), dtype=torch.float16, device=dev)
                for i, plan in enumerate(cands):
                    fn = _step_fn(pkv, lib, plan, problem, tensors, scale, ws, out, stream)
                    fn()  # warm
                    us = timer(fn)
                    f = features(plan, lens)
                    rows.append({"trace": name, "seed": int(seed), "t": int(t), "sum_len": int(lens.sum()),
                                 "policy": bool(with_policy and i == len(cands) - 1), "us": us,
                                 "predicted_us": predict(consts, f), **f})
                torch.cuda.synchronize()
                if pkv.pkv_read_status(ws) != 0:
                    raise RuntimeError(f"device status set on {name} seed {seed} step {t}")
                del ws
            del k, v
            torch.cuda.empty_cache()
            log(f"{name} seed {seed}: {n_steps} steps, {time.time() - t0:.1f} s")
    return rows


# ------------------------------------------------------------------------------------------------ fit
def fit(rows, start: dict):
    """Least-squares fit of the constants on the policy's candidates that are near-optimal for their step (the
    policy has to rank those well; far-off candidates would only pull the constants towards plans it never picks).
    """
    from scipy.optimize import least_squares

    best_of = {}
    for r in rows:
        k = (r["trace"], r["seed"], r["t"])
        best_of[k] = min(best_of.get(k, float("inf")), r["us"])
    rows = [r for r in rows if policy_candidate(r) and not r.get("policy")
            and r["us"] <= NEAR_OPTIMAL * best_of[(r["trace"], r["seed"], r["t"])]]
    meas = np.array([r["us"] for r in rows])
    # constants no row depends on keep their starting value
    used = {"fused_us": any(r["fused"] for r in rows), "fused_state_us": any(r["fused"] for r in rows),
            "build_us": any(r["variant"] == WQ and not r["in_decode"] for r in rows)}
    free = [k for k in CONSTANTS if used.get(k, True)]
    x0 = np.array([start[k] for k in free])
    lo = np.array([BOUNDS[k][0] for k in free])
    hi = np.array([BOUNDS[k][1] for k in free])
    x0 = np.clip(x0, lo + 1e-9, hi - 1e-9)

    def consts(x):
        c = dict(start)
        c.update(zip(free, x))
        return c

    def resid(x):
        c = consts(x)
        return np.array([predict(c, r) for r in rows]) / meas - 1.0

    best = None
    for scale in (1.0, 0.6, 1.6):  # a few starts: the model is piecewise (min, ceil)
        xs = np.clip(x0 * scale, lo + 1e-9, hi - 1e-9)
        res = least_squares(resid, xs, bounds=(lo, hi), x_scale="jac", max_nfev=4000)
        if best is None or res.cost < best.cost:
            best = res
    c = {k: float(v) for k, v in consts(best.x).items()}
    err = np.abs(resid(best.x))
    return c, {"rows": len(rows), "mean_abs_rel_err": float(err.mean()), "p90_abs_rel_err": float(np.quantile(err, 0.9)),
               "fitted": free}


def step_groups(rows):
    """The timed candidates of every (trace, seed, step), without the policy's own row."""
    by = {}
    for r in rows:
        if not r.get("policy"):
            by.setdefault((r["trace"], r["seed"], r["t"]), []).append(r)
    return list(by.values())


def mean_regret(c: dict, groups) -> float:
    """Mean over the trace families of the policy's mean regret: per step, the candidate the model predicts fastest
    (among those pkv_plan may choose) against the fastest one measured."""
    per = {}
    for rs in groups:
        best = min(r["us"] for r in rs)
        chosen = min((r for r in rs if policy_candidate(r)), key=lambda r: predict(c, r))
        per.setdefault(rs[0]["trace"], []).append(chosen["us"] / best - 1.0)
    return float(np.mean([np.mean(v) for v in per.values()]))


def refine(rows, c: dict, seed: int = 0, restarts: int = 6, also: dict | None = None):
    """Refines least-squares constants towards the policy's purpose: ranking the candidates of a step. Nelder-Mead on
    the logarithms of the constants minimises the calibration steps' mean regret (mean_regret), from the better of
    the least-squares point and `also` (the constants in force), then from a few seeded perturbations of the best
    point so far."""
    from scipy.optimize import minimize

    groups = step_groups(rows)
    keys = [k for k in CONSTANTS if k != "build_us"]
    lo = np.log(np.array([BOUNDS[k][0] if BOUNDS[k][0] > 0 else 1e-4 for k in keys]))
    hi = np.log(np.array([BOUNDS[k][1] for k in keys]))

    def consts(x):
        out = dict(c)
        out.update(zip(keys, np.exp(np.clip(x, lo, hi))))
        return out

    def obj(x):
        return mean_regret(consts(x), groups)

    x0 = np.clip(np.log(np.array([max(c[k], 1e-4) for k in keys])), lo, hi)
    f0 = obj(x0)
    best_x, best_f = x0, f0
    if also is not None:
        xa = np.clip(np.log(np.array([max(also[k], 1e-4) for k in keys])), lo, hi)
        fa = obj(xa)
        if fa < best_f:
            best_x, best_f = xa, fa
    rng = np.random.default_rng(seed)
    for trial in range(restarts):
        xs = best_x + (rng.normal(0.0, 0.3, len(keys)) if trial else 0.0)
        res = minimize(obj, xs, method="Nelder-Mead", options={"maxiter": 1500, "xatol": 1e-3, "fatol": 1e-5})
        if res.fun < best_f:
            best_x, best_f = res.x, float(res.fun)
    stats = {"calibration_regret_lsq": f0, "calibration_regret": best_f}
    if also is not None:
        stats["calibration_regret_in_force"] = fa
    return consts(best_x), stats


def write_constants(c: dict, stats: dict, source: str):
    os.makedirs(POLICY_DIR, exist_ok=True)
    with open(os.path.join(POLICY_DIR, "constants.json"), "w") as f:
        json.dump({"constants": c, "fit": stats, "source": source}, f, indent=1)
    lines = ["// Cost-model constants of pkv_policy_default. Written by serving_paged_gqa_gb300/calibrate.py (fit) from",
             "// the calibration sweep; rebuild the library after changing them.", "#pragma once",
             f'#define PKV_FIT_SOURCE "{source}"']
    for k in CONSTANTS:
        lines.append(f"#define PKV_FIT_{k.upper()} {c[k]:.6g}")
    with open(HEADER, "w") as f:
        f.write("\n".join(lines) + "\n")


# ------------------------------------------------------------------------------------------------ storage
FIELDS = ("trace", "seed", "t", "sum_len", "policy", "us", "variant", "chunk", "splits", "tasks", "grid", "group",
          "fused", "in_decode", "kv_bytes", "p_max", "batch")


def save_rows(rows, path):
    """Measurements as a field list and one value list per row (about a third of the size of keyed rows)."""
    def val(r, k):
        v = r.get(k)
        return round(v, 2) if isinstance(v, float) and k == "us" else v
    with open(path, "w") as f:
        json.dump({"fields": FIELDS, "rows": [[val(r, k) for k in FIELDS] for r in rows]}, f, separators=(",", ":"))


def load_rows(path):
    from workloads import CONFIGS

    d = json.load(open(path))
    rows = [dict(zip(d["fields"], v)) for v in d["rows"]] if isinstance(d, dict) else d
    for r in rows:
        r.setdefault("batch", CONFIGS[r["trace"]].batch)
    return rows


# ------------------------------------------------------------------------------------------------ report
def report(rows) -> str:
    """Held-out evaluation table: regret of the policy's plan and of the best fixed plan, prediction error."""
    by = {}
    for r in rows:
        by.setdefault(r["trace"], {}).setdefault((r["seed"], r["t"]), []).append(r)
    key = lambda r: (r["variant"], r["chunk"], r["fused"])  # noqa: E731
    out = ["| trace | steps | policy regret mean | policy regret max | best fixed plan | its regret mean | "
           "policy choices | model error (policy plan) | model error (all) |", "|---|---|---|---|---|---|---|---|---|"]
    names = {SINGLE: "single", SPLIT: "split", WQ: "workqueue"}
    for trace, steps in by.items():
        regrets, perr = [], []
        totals = {}
        choices = {}
        allerr = []
        for st, rs in steps.items():
            cands = [r for r in rs if not r["policy"]]
            best = min(r["us"] for r in cands)  # over every timed plan, the ones the policy may not pick included
            pol = [r for r in rs if r["policy"]]
            for r in cands:
                totals.setdefault(key(r), []).append(r["us"] / best - 1.0)
                allerr.append(abs(r["predicted_us"] / r["us"] - 1.0))
            if pol:
                p = pol[0]
                regrets.append(p["us"] / best - 1.0)
                perr.append(abs(p["predicted_us"] / p["us"] - 1.0))
                nm = f'{names[p["variant"]]} c={p["chunk"]}{" fused" if p["fused"] else ""}'
                choices[nm] = choices.get(nm, 0) + 1
        n = len(steps)
        fixed = [(k, v) for k, v in totals.items() if len(v) == n]
        fk, fv = min(fixed, key=lambda kv: np.mean(kv[1])) if fixed else (None, [float("nan")])
        fname = "-" if fk is None else f'{names[fk[0]]} c={fk[1]}{" fused" if fk[2] else ""}'
        ch = ", ".join(f"{k} x{v}" for k, v in sorted(choices.items(), key=lambda kv: -kv[1]))
        out.append(f"| {trace} | {n} | {100 * np.mean(regrets):.1f} % | {100 * np.max(regrets):.1f} % | {fname} | "
                   f"{100 * np.mean(fv):.1f} % | {ch} | {100 * np.mean(perr):.1f} % | {100 * np.mean(allerr):.1f} % |")
    return "\n".join(out)


def main(argv=None):
    ap = argparse.ArgumentParser(prog="python -m serving_paged_gqa_gb300.calibrate")
    sub = ap.add_subparsers(dest="cmd", required=True)
    a = sub.add_parser("sweep")
    a.add_argument("--seeds", default="0,1,2,3,4")
    a.add_argument("--traces", default=",".join(TRACES))
    a.add_argument("--out", required=True)
    a = sub.add_parser("fit")
    a.add_argument("sweep")
    a = sub.add_parser("evaluate")
    a.add_argument("--seeds", default="5,6,7,8,9")
    a.add_argument("--traces", default=",".join(TRACES))
    a.add_argument("--out", required=True)
    a = sub.add_parser("report")
    a.add_argument("heldout")
    args = ap.parse_args(argv)
    sys.path.insert(0, ROOT)
    if args.cmd in ("sweep", "evaluate"):
        rows = sweep([int(s) for s in args.seeds.split(",")], args.traces.split(","),
                     with_policy=args.cmd == "evaluate")
        save_rows(rows, args.out)
        print(f"{len(rows)} measurements -> {args.out}")
    elif args.cmd == "fit":
        import serving_paged_gqa_gb300 as pkv

        rows = load_rows(args.sweep)
        in_force = policy_constants(pkv)
        c, stats = fit(rows, in_force)
        c, rstats = refine(rows, c, also=in_force)
        stats.update(rstats)
        seeds = sorted({r["seed"] for r in rows})
        write_constants(c, stats, f"least squares on {stats['rows']} timed candidate plans, then regret-refined on "
                                  f"every candidate, seeds {seeds}")
        print(json.dumps({"constants": c, "fit": stats}, indent=1))
    else:
        rows = load_rows(args.heldout)
        consts = policy_constants(__import__("serving_paged_gqa_gb300"))
        for r in rows:  # prediction error under the constants the library now holds
            r["predicted_us"] = predict(consts, r)
        print(report(rows))


if __name__ == "__main__":
    main()
