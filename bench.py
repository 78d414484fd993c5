"""Decode-step benchmark: paged GQA decode attention on one GB300 per rank.

One step = one decode step of a trace (plan, worklist build when the plan uses the workqueue, decode with the merge
fused into it) over one batch of synthetic inputs. Headline workload: the B1 bucketed long-context trace (B=1,
Hq=32, Hkv=8, d=128, page size 16, fp16 ~N(0,1), start length from {4096, 8192, 16384, 32768}, 64 steps of +1 token
per seed, pages shuffled in a 2^16-page pool) over the held-out seeds 5-9. The K timed steps are spread evenly over
all 5 x 64 steps of those traces (step j = k * 320 // K), so every length bucket the seeds drew is in the sample.
The same is then done for the B8 bimodal, uniform and Zipf-like traces, the B4 bimodal trace and (first held-out seed
only) the B = 64 stress step (sub-results under "traces").

Timing: between steps an L2 flush runs (a 256 MiB write, then a 256 MiB read of another buffer, both larger than
the 129 MB L2), so every step reads its KV from HBM, as it would after the other layers of a model ran. Then a GPU
spin of --spin-us keeps the GPU busy while the host enqueues the step, so the CUDA events around the step (and
around the decode kernel inside it) measure device time only, never a wait for the host. `value` = tokens / sum of
step times. `e2e` repeats the same steps through the public API from pinned host buffers, timed on the host wall
clock with a synchronize on both sides: per step one host->device copy of q, the block table, the lengths and the
new token's K/V, the step with that K/V appended into its page slot inside the decode, and the device->host copy
of out. `traces.multilayer_...` runs the decode loop of an 8-layer model's attention on the B8 bimodal trace (one
pkv_decode_step_append per layer per step, each layer with its own pools, no L2 flush: the layers' K/V exceed L2).
`cpu_baseline` times the fp64 oracle on the host on a bounded sample of the same steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config b1_bucketed] ...
Under torchrun (N > 1) every rank runs the same workload on its own GPU (replicas; no collective in the data
path); rank 0 prints one JSON line with value = tokens of all ranks / max over ranks of the timed time.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s per trace and KV-read HBM GB/s as % of GB300 peak"
L2_FLUSH_BYTES = 256 << 20
HELD_OUT = [5, 6, 7, 8, 9]
SUB_TRACES = ("b8_bimodal", "b8_uniform", "b8_zipf", "b4_bimodal", "stress")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_kernel_b1_bucketed.md")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="b1_bucketed")
    ap.add_argument("--traces", default=",".join(SUB_TRACES), help="sub-result traces ('none' to skip)")
    ap.add_argument("--seeds", default=",".join(map(str, HELD_OUT)))
    ap.add_argument("--variant", choices=["auto", "single", "split", "workqueue"], default="auto")
    ap.add_argument("--chunk", type=int, default=0, help="pages per split for a forced variant")
    ap.add_argument("--separate-merge", action="store_true", help="use the merge kernel instead of the fused merge")
    ap.add_argument("--spin-us", type=float, default=150.0, help="GPU spin before each timed step")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the oracle cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-wall", action="store_true")
    ap.add_argument("--pool-pages", type=int, default=0, help="override the page-pool size (small profiling runs)")
    ap.add_argument("--reference-budget", type=float, default=120.0, help="seconds for the reference arm's steps")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------------------------------- helpers
def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("decode.cu", "pkv_ptx.cuh", "pkv_internal.h"):
        with open(os.path.join(ROOT, "serving_paged_gqa_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic():
    """(DRAM bytes per KV token, kernel hash) from the committed ncu summary, if present."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None, None
    vals = {}
    for line in open(PROFILE_SUMMARY):
        line = line.strip()
        if line.startswith("- ") and "=" in line:
            k, v = line[2:].split("=", 1)
            vals[k.strip()] = v.strip().strip("`")
    try:
        return float(vals["dram_bytes_per_kv_token"]), vals["kernel_sha256_16"]
    except (KeyError, ValueError):
        return None, None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def max_over_ranks(x: float, dev) -> float:
    """The largest x over the ranks of the default process group (x itself without one)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, slowest_ms: float) -> float:
    """Units of all ranks (replicas, the same work each) over the slowest rank's timed milliseconds, per second."""
    return units_per_rank * world / (slowest_ms * 1e-3)


def strided(n: int, k: int) -> list[int]:
    """k step indices spread evenly over n steps."""
    return [(i * n) // k for i in range(k)]


class ClockSampler:
    """nvidia-smi clocks/throttle sampler (200 ms) around the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.proc = None
        if enabled:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None

    def finish(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


class L2Flush:
    """Evicts the L2 between steps: a write of one buffer larger than L2, then a read of another, which leaves
    only clean lines behind."""

    def __init__(self, torch, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        self.sink = self.r.sum()


# ------------------------------------------------------------------------------------------------ workload
class Workload:
    """Device tensors for every step of every seed's trace: a pool per seed holding every page the trace uses,
    per-step q, block table and lengths."""

    def __init__(self, torch, config: str, seeds, dev, pool_pages: int = 0):
        from workloads import make_trace

        self.config, self.seeds = config, list(seeds)
        self.traces, self.steps = [], []
        for seed in seeds:
            tr = make_trace(config, seed, pool_pages=pool_pages or None)
            ps, hkv, d = tr.ps, tr.hkv, tr.d
            k = torch.empty((tr.num_pages, ps, hkv, d), dtype=torch.float16, device=dev)
            v = torch.empty((tr.num_pages, ps, hkv, d), dtype=torch.float16, device=dev)
            idx = torch.from_numpy(tr.used_pages).to(dev)
            k.index_copy_(0, idx, torch.from_numpy(tr.k_pages).to(dev))
            v.index_copy_(0, idx, torch.from_numpy(tr.v_pages).to(dev))
            self.traces.append((tr, k, v))
            for t in range(tr.steps):
                lens = tr.seq_lens(t)
                bt = tr.block_table(t)
                q = tr.q(t)
                self.steps.append({"trace": len(self.traces) - 1, "seed": int(seed), "t": t, "lens_host": lens,
                                   "bt_host": bt, "q_host": q, "q": torch.from_numpy(q).to(dev),
                                   "bt": torch.from_numpy(bt).to(dev), "lens": torch.from_numpy(lens).to(dev)})
        tr0 = self.traces[0][0]
        self.B, self.Hq, self.Hkv, self.d, self.ps = tr0.batch, tr0.hq, tr0.hkv, tr0.d, tr0.ps

    def problem(self, pkv, i):
        tr = self.traces[i][0]
        return pkv.make_problem(tr.batch, tr.hq, tr.hkv, tr.d, tr.ps, tr.num_pages, tr.max_pages)


def make_plan(pkv, problem, lens, sms, args):
    if args.variant == "auto":
        plan = pkv.pkv_plan(problem, lens, sms)
    else:
        v = {"single": pkv.PKV_VARIANT_SINGLE, "split": pkv.PKV_VARIANT_SPLIT,
             "workqueue": pkv.PKV_VARIANT_WORKQUEUE}[args.variant]
        chunk = args.chunk
        if chunk <= 0:
            pmax = int(((lens.astype(np.int64) + 15) // 16).max())
            chunk = max(1, -(-pmax // 32))
        plan = pkv.pkv_plan_fixed(problem, lens, sms, v, chunk)
    if args.separate_merge and plan.variant != pkv.PKV_VARIANT_SINGLE:
        plan.fuse_merge = 0
    return plan


class Marshalled:
    """ctypes arguments of one step's C calls, built before the timed region."""

    def __init__(self, pkv, wl, j, plan, ws, out, scale, stream):
        s = wl.steps[j]
        _, kpool, vpool = wl.traces[s["trace"]]
        self.plan = plan
        self.problem = wl.problem(pkv, s["trace"])
        vp = ctypes.c_void_p
        st = vp(stream.cuda_stream)
        pr, pl = ctypes.byref(self.problem), ctypes.byref(self.plan)
        self.build = (pl, pr, vp(s["lens"].data_ptr()), vp(ws.data_ptr()), ws.numel(), st)
        self.decode = (pl, pr, vp(s["q"].data_ptr()), vp(kpool.data_ptr()), vp(vpool.data_ptr()),
                       vp(s["bt"].data_ptr()), vp(s["lens"].data_ptr()), ctypes.c_float(scale), vp(ws.data_ptr()),
                       ws.numel(), vp(out.data_ptr()), st)
        self.merge = (pl, pr, vp(ws.data_ptr()), ws.numel(), vp(out.data_ptr()), st)
        self.wq = plan.variant == pkv.PKV_VARIANT_WORKQUEUE and not plan.list_in_decode  # a builder launch
        self.separate_merge = plan.variant != pkv.PKV_VARIANT_SINGLE and not plan.fuse_merge


def _call(fn, args, what):
    rc = fn(*args)
    if rc != 0:
        raise SystemExit(f"{what} failed: {rc}")


def time_workload(pkv, torch, wl, K, W, args, sms, dev, flush, stream):
    """Times K steps spread over the workload (after W warm-up steps): events around each step and around the
    decode kernel inside it. Returns per-step arrays and the plans used."""
    lib = pkv.load()
    idx = strided(len(wl.steps), K)
    warm = strided(len(wl.steps), max(W, 1))[:W]
    scale = 1.0 / math.sqrt(wl.d)
    plans = {}
    for j in set(idx) | set(warm):
        s = wl.steps[j]
        plans[j] = make_plan(pkv, wl.problem(pkv, s["trace"]), s["lens_host"], sms, args)
    ws = pkv.alloc_workspace(max(p.ws_bytes for p in plans.values()), dev)
    out = torch.empty((wl.B, wl.Hq, wl.d), dtype=torch.float16, device=dev)
    calls = {j: Marshalled(pkv, wl, j, plans[j], ws, out, scale, stream) for j in plans}
    spin_cycles = int(args.spin_us * 1e-6 * 2.0e9)

    def step(c, ev=None, inner=False):
        # inner events split the step into its kernels; they also stop a dependent launch from overlapping the
        # kernel before it, so the step time is taken in a pass without them
        if ev is not None:
            ev[0].record(stream)
        if c.wq:
            _call(lib.pkv_build_worklist, c.build, "pkv_build_worklist")
        if inner:
            ev[1].record(stream)
        _call(lib.pkv_decode, c.decode, "pkv_decode")
        if inner:
            ev[2].record(stream)
        if c.separate_merge:
            _call(lib.pkv_merge, c.merge, "pkv_merge")
        if ev is not None:
            ev[3].record(stream)

    for j in warm:
        flush()
        step(calls[j])
    torch.cuda.synchronize()
    if pkv.pkv_read_status(ws) != 0:
        raise SystemExit("device status set during warm-up")

    def timed_pass(inner):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        torch.cuda.synchronize()
        for k, j in enumerate(idx):
            flush()
            torch.cuda._sleep(spin_cycles)
            step(calls[j], ev[k], inner)
        torch.cuda.synchronize()
        return ev

    ev = timed_pass(False)
    launches = sum(pkv.pkv_plan_launches(plans[j]) for j in idx)
    step_ms = np.array([e[0].elapsed_time(e[3]) for e in ev])
    ev = timed_pass(True)
    status = pkv.pkv_read_status(ws)
    copy_ms = copy_same_bytes(torch, dev, stream, flush, [plans[j].kv_bytes for j in idx], spin_cycles)
    dec_ms = np.array([e[1].elapsed_time(e[2]) for e in ev])
    merge_ms = np.array([e[2].elapsed_time(e[3]) for e in ev])  # zero-length pair unless the merge is separate
    build_ms = np.array([e[0].elapsed_time(e[1]) for e in ev])
    kv_bytes = np.array([plans[j].kv_bytes for j in idx])
    return {"idx": idx, "plans": [plans[j] for j in idx], "step_ms": step_ms, "dec_ms": dec_ms, "merge_ms": merge_ms,
            "build_ms": build_ms, "copy_ms": copy_ms,
            "kv_bytes": kv_bytes, "launches": launches, "status": status, "ws": ws, "out": out}


def wall_calls(pkv, wl, r, sms, args, stream):
    """Per timed step: the planner call (pkv_plan, or pkv_plan_fixed for a forced schedule) and the pkv_decode_step
    call with their ctypes arguments built once; both write / read the same Plan struct."""
    lib = pkv.load()
    vp = ctypes.c_void_p
    st = vp(stream.cuda_stream)
    scale = ctypes.c_float(1.0 / math.sqrt(wl.d))
    out = []
    for j in r["idx"]:
        s = wl.steps[j]
        _, kpool, vpool = wl.traces[s["trace"]]
        problem = wl.problem(pkv, s["trace"])
        plan = pkv.Plan()
        lens = np.ascontiguousarray(s["lens_host"], dtype=np.int32)
        if args.variant == "auto":
            plan_fn, plan_args = lib.pkv_plan, (ctypes.byref(problem), lens.ctypes.data_as(vp), int(sms), None,
                                                ctypes.byref(plan))
        else:
            v = {"single": pkv.PKV_VARIANT_SINGLE, "split": pkv.PKV_VARIANT_SPLIT,
                 "workqueue": pkv.PKV_VARIANT_WORKQUEUE}[args.variant]
            fixed = make_plan(pkv, problem, s["lens_host"], sms, args)  # the chunk the forced schedule uses
            plan_fn, plan_args = lib.pkv_plan_fixed, (ctypes.byref(problem), lens.ctypes.data_as(vp), int(sms), v,
                                                      int(fixed.chunk_pages), 0, ctypes.byref(plan))
        step_args = (ctypes.byref(plan), ctypes.byref(problem), vp(s["q"].data_ptr()), vp(kpool.data_ptr()),
                     vp(vpool.data_ptr()), vp(s["bt"].data_ptr()), vp(s["lens"].data_ptr()), scale,
                     vp(r["ws"].data_ptr()), r["ws"].numel(), vp(r["out"].data_ptr()), st)
        out.append((problem, plan, plan_fn, plan_args, step_args, lens))
    return out


def copy_same_bytes(torch, dev, stream, flush, sizes, spin_cycles):
    """The same protocol (L2 flushed, GPU spin, CUDA events) around one device-to-device torch copy that moves each
    step's algorithmic bytes (half read, half written), the operation the measured HBM peak is taken with: what moving
    those bytes in one call takes on this part at this size, launch and event costs included."""
    half = int(max(sizes)) // 2 + 256
    src = torch.zeros(half, dtype=torch.uint8, device=dev)
    dst = torch.empty(half, dtype=torch.uint8, device=dev)
    ms = []
    for nbytes in sizes:
        n = int(nbytes) // 2
        flush()
        torch.cuda._sleep(spin_cycles)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst[:n].copy_(src[:n])
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    del src, dst
    return np.array(ms)


def by_tokens(wl, r):
    """Mean step / decode time of the timed steps grouped by the step's token count rounded to a power of two."""
    groups = {}
    for k, j in enumerate(r["idx"]):
        key = str(int(2 ** round(math.log2(max(1, int(wl.steps[j]["lens_host"].sum()))))))
        groups.setdefault(key, []).append(k)
    return {key: {"steps": len(ks), "step_us": 1e3 * float(r["step_ms"][ks].mean()),
                  "decode_us": 1e3 * float(r["dec_ms"][ks].mean()),
                  "copy_same_bytes_us": 1e3 * float(r["copy_ms"][ks].mean()),
                  "bytes": float(r["kv_bytes"][ks].mean())} for key, ks in sorted(groups.items(), key=lambda x: int(x[0]))}


def merge_used(pkv, plans) -> dict:
    """How the timed steps' plans merge the split states: {"none (single pass)" | "separate kernel" | "fused": steps}."""
    used = {}
    for p in plans:
        k = ("none (single pass)" if p.variant == pkv.PKV_VARIANT_SINGLE
             else "fused" if p.fuse_merge else "separate kernel")
        used[k] = used.get(k, 0) + 1
    return used


def _mean_us(ms, has_kernel) -> float | None:
    """Mean of the event-timed kernel over the steps that launch it (None if none does: an event pair with no
    kernel between them reads ~2 us of event overhead, not a kernel)."""
    sel = np.asarray(ms)[np.asarray(has_kernel, dtype=bool)]
    return 1e3 * float(sel.mean()) if sel.size else None


def summarize(pkv, wl, r, peak):
    plans = r["plans"]
    K = len(plans)
    tok = K * wl.B
    return {"by_tokens": by_tokens(wl, r),"tokens_per_s": tok / (r["step_ms"].sum() * 1e-3), "step_us_mean": 1e3 * float(r["step_ms"].mean()),
            "decode_us_mean": 1e3 * float(r["dec_ms"].mean()),
            "merge_us_mean": _mean_us(r["merge_ms"], [p.variant != pkv.PKV_VARIANT_SINGLE and not p.fuse_merge
                                                      for p in plans]),
            "build_us_mean": _mean_us(r["build_ms"], [p.variant == pkv.PKV_VARIANT_WORKQUEUE and not p.list_in_decode
                                                      for p in plans]),
            "decode_frac": float(r["kv_bytes"].sum() / (r["dec_ms"].sum() * 1e-3)) / 1e9 / peak,
            "copy_same_bytes_us_mean": 1e3 * float(r["copy_ms"].mean()),
            "copy_same_bytes_frac": float(r["kv_bytes"].sum() / (r["copy_ms"].sum() * 1e-3)) / 1e9 / peak,
            "copy_over_decode_time": float(r["copy_ms"].sum() / r["dec_ms"].sum()),
            "step_frac": float(r["kv_bytes"].sum() / (r["step_ms"].sum() * 1e-3)) / 1e9 / peak,
            "algorithmic_bytes_per_step": float(r["kv_bytes"].mean()),
            "variants_used": sorted({pkv.VARIANT_NAMES[p.variant] for p in plans}),
            "merge_used": merge_used(pkv, plans),
            "chunk_pages_min_max": [int(min(p.chunk_pages for p in plans)), int(max(p.chunk_pages for p in plans))],
            "splits_min_max": [int(min(p.num_splits for p in plans)), int(max(p.num_splits for p in plans))],
            "launches_per_step": r["launches"] / K, "steps": K, "device_status": int(r["status"])}


# ------------------------------------------------------------------------------------------------ oracle legs
def oracle_baseline(wl, idx, budget_s):
    """Times the fp64 oracle on whole trace steps (all query heads) of the timed step set until the budget is
    spent."""
    import oracle

    pools = {}
    done_tokens, spent, n_steps = 0, 0.0, 0
    for j in idx:
        s = wl.steps[j]
        tr = wl.traces[s["trace"]][0]
        if s["trace"] not in pools:
            pools[s["trace"]] = tr.host_pools()
        kp, vp = pools[s["trace"]]
        t0 = time.perf_counter()
        oracle.attention(s["q_host"], kp, vp, s["bt_host"], s["lens_host"])
        spent += time.perf_counter() - t0
        done_tokens += tr.batch
        n_steps += 1
        if spent >= budget_s:
            break
    return {"value": done_tokens / spent, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"the first {n_steps} of the {len(idx)} timed {wl.config} steps (held-out seeds "
                      f"{wl.seeds}), all {wl.Hq} query heads per row, fp64, {spent:.1f} s"}


def run_reference(args):
    """The reference arm: the fp64 CPU oracle timed on the host cores, one bounded sample per step."""
    rank, world, _ = dist_info()
    if rank != 0:
        return
    import oracle
    from workloads import make_trace

    seeds = [int(s) for s in args.seeds.split(",")]
    traces = []
    for seed in seeds:
        tr = make_trace(args.config, seed)
        traces.append((tr, *tr.host_pools()))
    B, Hq = traces[0][0].batch, traces[0][0].hq
    pairs_all = np.array([(b, h) for b in range(B) for h in range(Hq)], dtype=np.int32)
    order = []
    for i, (tr, _, _) in enumerate(traces):
        order += [(i, t) for t in range(tr.steps)]
    pick = strided(len(order), args.steps)

    def one(k, npairs):
        i, t = order[pick[k % len(pick)]]
        tr, kp, vp = traces[i]
        sel = pairs_all[(np.arange(npairs) + k * npairs) % len(pairs_all)]
        t0 = time.perf_counter()
        oracle.attention(tr.q(t), kp, vp, tr.block_table(t), tr.seq_lens(t), pairs=sel)
        return time.perf_counter() - t0

    # size the per-step sample so that warmup + steps fit the budget
    probe = np.mean([one(k, 1) for k in range(3)])
    npairs = int(max(1, min(len(pairs_all), args.reference_budget / max(1, args.steps + args.warmup) / probe)))
    for k in range(args.warmup):
        one(k, npairs)
    spent = sum(one(k, npairs) for k in range(args.steps))
    tokens = args.steps * npairs / (B * Hq)
    value = tokens / spent
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * spent / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": args.config, "seeds": seeds, "batch": B, "num_q_heads": Hq,
                       "num_kv_heads": traces[0][0].hkv, "head_dim": traces[0][0].d, "page_size": traces[0][0].ps,
                       "timed_steps": f"{args.steps} steps spread over the {len(order)} trace steps"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{npairs} of {B * Hq} (row, query head) pairs of one trace step per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------------ our arm
def run_e2e(pkv, torch, wl, idx, args, sms, flush, stream, dev):
    """The same steps through the public serving call, host wall clock with a synchronize on both sides: each step's
    inputs (q, the new token's K/V, block table, lengths) sit packed in pinned host memory (pkv_step_input_layout);
    one pkv_serve_step call plans the step from the host lengths, copies the packed input to the device, runs the
    decode with the new token's K/V appended into its page slot, and copies out back to pinned host memory; then the
    stream is synchronised. The buffers are bound once per step buffer, as a server keeps its per-layer buffers:
    through a ServeSession (the step's launches replayed from the CUDA graph of its plan, captured in an untimed
    first run: a decode loop's plan repeats for chunk_pages * page_size steps) for the reported value, and through
    ServeStep (plan and launches enqueued by the call every step) for comparison."""
    B, Hq, Hkv, d, ps = wl.B, wl.Hq, wl.Hkv, wl.d, wl.ps
    scale = 1.0 / math.sqrt(d)
    out_d = torch.empty((B, Hq, d), dtype=torch.float16, device=dev)
    out_h = torch.empty((B, Hq, d), dtype=torch.float16).pin_memory()
    # the workspace is allocated once, before the timed steps, for the largest plan among them
    ws_bytes = max(make_plan(pkv, wl.problem(pkv, wl.steps[j]["trace"]), wl.steps[j]["lens_host"], sms, args).ws_bytes
                   for j in idx)
    ws = pkv.alloc_workspace(ws_bytes, dev)
    totals = [pkv.pkv_step_input_layout(wl.problem(pkv, wl.steps[j]["trace"]))[1] for j in idx]
    dev_in = torch.empty(max(totals), dtype=torch.uint8, device=dev)
    policy = None
    if args.variant != "auto" or args.separate_merge:
        return None  # the serving call runs the policy's plans only
    runners = []
    for j in idx:
        s = wl.steps[j]
        tr, kpool, vpool = wl.traces[s["trace"]]
        problem = wl.problem(pkv, s["trace"])
        lens = s["lens_host"]
        new_phys = s["bt_host"][np.arange(B), (lens - 1) // ps]
        new_slot = (lens - 1) % ps
        used_index = {int(p): i for i, p in enumerate(tr.used_pages)}
        k_new = np.stack([tr.k_pages[used_index[int(new_phys[b])], int(new_slot[b])] for b in range(B)])
        v_new = np.stack([tr.v_pages[used_index[int(new_phys[b])], int(new_slot[b])] for b in range(B)])
        offs, total = pkv.pkv_step_input_layout(problem)
        buf = np.zeros(total, dtype=np.uint8)
        for o, part in zip(offs, (s["q_host"], k_new, v_new, s["bt_host"], lens)):
            raw = np.ascontiguousarray(part).view(np.uint8).ravel()
            buf[o:o + raw.size] = raw
        host_in = torch.from_numpy(buf).pin_memory()
        runners.append((pkv.ServeSession(problem, host_in, dev_in, kpool, vpool, scale, ws, out_d, out_h, policy, sms),
                        pkv.ServeStep(problem, host_in, dev_in, kpool, vpool, scale, ws, out_d, out_h, stream,
                                      policy, sms), total))
    for session, _, _ in runners:  # graph capture, untimed
        session.run(stream)
    stream.synchronize()

    def timed(which):
        times = []
        for r in runners:
            flush()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            r[0].run(stream) if which == 0 else r[1].run()
            stream.synchronize()
            times.append(time.perf_counter() - t0)
        return np.array(times)

    times = timed(0)
    direct = timed(1)
    graphs = [r[0].stats() for r in runners]
    for r in runners:
        r[0].close()
    h2d, d2h = runners[-1][2], out_h.numel() * 2
    return {"value": B * len(times) / float(np.sum(times)), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": len(times), "us_per_step": 1e6 * float(np.mean(times)),
            "graph_replays_timed": int(sum(n - 1 for _, n in graphs)),
            "direct_us_per_step": 1e6 * float(np.mean(direct)),
            "direct_value": B * len(direct) / float(np.sum(direct)),
            "timing": "host wall clock per step, synchronize on both sides; one pkv_session_step call: pkv_plan on "
                      "the host lengths, then the plan's CUDA graph: the packed input read from pinned host memory "
                      "into the device, decode with the KV append fused, out stored into pinned host memory; "
                      "direct_*: the same step through pkv_serve_step, its launches enqueued by the call"}


def run_multilayer(pkv, torch, args, sms, dev, stream, peak, name="b8_bimodal", seed=5, layers=8):
    """Decode loop of a `layers`-layer model's attention: per step and layer, the new token's K/V appended into that
    layer's pools and the layer's attention, all inside pkv_decode_step_append, the layers' steps back to back on the
    stream with one event pair around the whole step. The layers share the trace's block table and lengths; each has
    its own pools (sized to the trace, pages drawn by the trace's permutation) and the same contents, so every layer
    reads its own K/V from HBM (the layers' K/V together exceed the L2)."""
    import math as _m

    from workloads import make_trace

    tr = make_trace(name, seed)
    B, Hq, Hkv, d, ps = tr.batch, tr.hq, tr.hkv, tr.d, tr.ps
    idx = torch.from_numpy(tr.used_pages).to(dev)
    kh, vh = torch.from_numpy(tr.k_pages).to(dev), torch.from_numpy(tr.v_pages).to(dev)
    pools = []
    for _ in range(layers):
        k = torch.empty((tr.num_pages, ps, Hkv, d), dtype=torch.float16, device=dev)
        v = torch.empty_like(k)
        k.index_copy_(0, idx, kh)
        v.index_copy_(0, idx, vh)
        pools.append((k, v))
    del kh, vh
    problem = pkv.make_problem(B, Hq, Hkv, d, ps, tr.num_pages, tr.max_pages)
    scale = 1.0 / _m.sqrt(d)
    K = min(args.steps, tr.steps)
    ts = strided(tr.steps, K)
    used_index = {int(p): i for i, p in enumerate(tr.used_pages)}
    steps = []
    for t in ts:
        lens = tr.seq_lens(t)
        bt = tr.block_table(t)
        phys = bt[np.arange(B), (lens - 1) // ps]
        slot = (lens - 1) % ps
        k_new = np.stack([tr.k_pages[used_index[int(phys[b])], int(slot[b])] for b in range(B)])
        v_new = np.stack([tr.v_pages[used_index[int(phys[b])], int(slot[b])] for b in range(B)])
        plan = pkv.pkv_plan(problem, lens, sms)
        steps.append((plan, torch.from_numpy(tr.q(t)).to(dev), torch.from_numpy(k_new).to(dev),
                      torch.from_numpy(v_new).to(dev), torch.from_numpy(bt).to(dev), torch.from_numpy(lens).to(dev),
                      float(plan.kv_bytes)))
    ws = pkv.alloc_workspace(max(st[0].ws_bytes for st in steps), dev)
    out = torch.empty((B, Hq, d), dtype=torch.float16, device=dev)
    lib = pkv.load()
    vp = ctypes.c_void_p
    calls = []
    for plan, q, kn, vn, bt, ln, _ in steps:
        calls.append([(ctypes.byref(plan), ctypes.byref(problem), vp(q.data_ptr()), vp(kn.data_ptr()),
                       vp(vn.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(bt.data_ptr()), vp(ln.data_ptr()),
                       ctypes.c_float(scale), vp(ws.data_ptr()), ws.numel(), vp(out.data_ptr()),
                       vp(stream.cuda_stream)) for k, v in pools])
    spin = int(args.spin_us * 4 * 1e-6 * 2.0e9)

    def run(overlap):
        # layers after the first may start while the previous layer's last kernel finishes (PKV_PLAN_OVERLAP_PREV):
        # their pools, block table and lengths are not written by it
        for st in steps:
            st[0].flags = pkv.PKV_PLAN_OVERLAP_PREV if overlap else 0
        for layer_calls in calls[:2]:
            for a in layer_calls:
                _call(lib.pkv_decode_step_append, a, "pkv_decode_step_append")
        torch.cuda.synchronize()
        ev = []
        for layer_calls in calls:
            torch.cuda._sleep(spin)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for a in layer_calls:
                _call(lib.pkv_decode_step_append, a, "pkv_decode_step_append")
            e1.record(stream)
            ev.append((e0, e1))
        torch.cuda.synchronize()
        return np.array([a.elapsed_time(b) * 1e3 for a, b in ev])

    step_us_plain = run(False)
    step_us = run(True)
    status = pkv.pkv_read_status(ws)
    kv = np.array([st[6] for st in steps]) * layers
    return {"layers": layers, "trace": name, "seed": seed, "steps": K, "tokens_per_s": B * K / (step_us.sum() * 1e-6),
            "step_us_mean": float(step_us.mean()), "layer_us_mean": float(step_us.mean()) / layers,
            "layer_us_mean_without_overlap": float(step_us_plain.mean()) / layers,
            "overlap": "layers after the first launched with PKV_PLAN_OVERLAP_PREV",
            "step_frac": float(kv.sum() / (step_us.sum() * 1e-6)) / 1e9 / peak,
            "launches_per_step": layers * pkv.pkv_plan_launches(steps[0][0]),
            "variants_used": sorted({pkv.VARIANT_NAMES[st[0].variant] for st in steps}),
            "l2": "not flushed: each step reads every layer's own pools", "device_status": int(status)}


def run_schedules(pkv, torch, args, sms, dev, flush, stream, name="b8_bimodal"):
    """The pages' comparison on held-out bimodal B8 steps: exact-length buckets (one split grid + merge per distinct
    length, rows sorted by length), the padded split grid and the compact workqueue, each as the planner sizes it:
    device time per step, launches per step and partial-state bytes per step."""
    from serving_paged_gqa_gb300 import schedules

    seeds = [int(x) for x in args.seeds.split(",")]
    wl = Workload(torch, name, seeds, dev, args.pool_pages)
    scale = 1.0 / math.sqrt(wl.d)
    spin = int(2 * args.spin_us * 1e-6 * 2.0e9)
    res = {k: {"us": [], "launches": [], "state_bytes": []} for k in ("exact_buckets", "padded_grid", "workqueue")}
    same_c = []  # partial-state bytes of the padded grid cut like the workqueue (the pages' like-for-like counter)
    for j in strided(len(wl.steps), args.steps):
        s = wl.steps[j]
        _, kpool, vpool = wl.traces[s["trace"]]
        problem = wl.problem(pkv, s["trace"])
        order = np.argsort(s["lens_host"], kind="stable")
        oi = torch.from_numpy(order).to(dev)
        q_s, bt_s, ln_s = s["q"][oi].contiguous(), s["bt"][oi].contiguous(), s["lens"][oi].contiguous()
        buckets = schedules.ExactLengthBuckets(pkv, problem, s["lens_host"][order], sms)
        padded = schedules.padded_grid_plan(pkv, problem, s["lens_host"], sms)
        work = schedules.workqueue_plan(pkv, problem, s["lens_host"], sms)
        same_c.append(schedules.state_bytes(pkv.pkv_plan_fixed(problem, s["lens_host"], sms, pkv.PKV_VARIANT_SPLIT,
                                                               work.chunk_pages)))
        ws = pkv.alloc_workspace(max(buckets.ws_bytes, padded.ws_bytes, work.ws_bytes), dev)
        out = torch.empty_like(s["q"])
        runs = {"exact_buckets": (lambda: buckets.run(q_s, kpool, vpool, bt_s, ln_s, scale, ws, out, stream),
                                  buckets.launches(), buckets.state_bytes()),
                "padded_grid": (lambda: pkv.pkv_decode_step(padded, problem, s["q"], kpool, vpool, s["bt"], s["lens"],
                                                            scale, ws, out, stream),
                                pkv.pkv_plan_launches(padded), schedules.state_bytes(padded)),
                "workqueue": (lambda: pkv.pkv_decode_step(work, problem, s["q"], kpool, vpool, s["bt"], s["lens"],
                                                          scale, ws, out, stream),
                              pkv.pkv_plan_launches(work), schedules.state_bytes(work))}
        for key, (fn, launches, sb) in runs.items():
            fn()
            ev = []
            for _ in range(3):
                flush()
                torch.cuda._sleep(spin)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                ev.append((e0, e1))
            torch.cuda.synchronize()
            res[key]["us"].append(float(np.median([a.elapsed_time(b) * 1e3 for a, b in ev])))
            res[key]["launches"].append(launches)
            res[key]["state_bytes"].append(sb)
        if pkv.pkv_read_status(ws) != 0:
            raise SystemExit("device status set in the schedule comparison")
    out = {k: {"us_per_step": float(np.mean(v["us"])), "launches_per_step": float(np.mean(v["launches"])),
               "state_mb_per_step": float(np.mean(v["state_bytes"])) / 1e6} for k, v in res.items()}
    out["workqueue_vs_exact_buckets_time"] = out["workqueue"]["us_per_step"] / out["exact_buckets"]["us_per_step"]
    out["padded_grid_at_workqueue_split_size_state_mb_per_step"] = float(np.mean(same_c)) / 1e6
    out["workqueue_vs_padded_state_traffic_same_split_size"] = (
        out["workqueue"]["state_mb_per_step"] / out["padded_grid_at_workqueue_split_size_state_mb_per_step"] - 1.0)
    out["pages"] = ("RTX 3060: 16.00 -> 2.00 launches per step (exact buckets -> workqueue), merge-state traffic "
                    "about -37 %")
    out["steps"] = args.steps
    return out


def run_ours(args):
    import torch

    rank, world, local = dist_info()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__

    __graft_entry__.build()
    import serving_paged_gqa_gb300 as pkv

    seeds = [int(s) for s in args.seeds.split(",")]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak, peak_kind = measured_peaks()
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)
    K, W = args.steps, args.warmup

    # ---- headline workload
    wl = Workload(torch, args.config, seeds, dev, args.pool_pages)
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    if not args.no_clocks:
        time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    r = time_workload(pkv, torch, wl, K, W, args, sms, dev, flush, stream)
    timed_wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.finish()
    total_ms = max_over_ranks(float(r["step_ms"].sum()), dev)
    head = summarize(pkv, wl, r, peak)

    # ---- synchronized wall time per step (the pages' protocol): plan + launches + sync, flush outside
    # (the C calls with their arguments marshalled before the loop, as a C caller makes them: pkv_plan on the host
    # lengths, then pkv_decode_step)
    wall_us = None
    if not args.no_wall:
        wall = []
        for problem, plan, plan_fn, plan_args, step_args, _keep in wall_calls(pkv, wl, r, sms, args, stream):
            flush()
            torch.cuda.synchronize()
            w0 = time.perf_counter()
            _call(plan_fn, plan_args, "pkv_plan")
            if args.separate_merge and plan.variant != pkv.PKV_VARIANT_SINGLE:
                plan.fuse_merge = 0
            _call(pkv.load().pkv_decode_step, step_args, "pkv_decode_step")
            torch.cuda.synchronize()
            wall.append(time.perf_counter() - w0)
        wall_us = 1e6 * float(np.mean(wall))

    e2e = None if args.no_e2e else run_e2e(pkv, torch, wl, r["idx"], args, sms, flush, stream, dev)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = oracle_baseline(wl, r["idx"], args.cpu_seconds)

    traffic_per_tok, traffic_hash = profile_traffic()
    traffic = None
    if traffic_per_tok is not None and traffic_hash == kernel_source_hash():
        mean_tokens = float(np.mean([int(wl.steps[j]["lens_host"].sum()) for j in r["idx"]]))
        traffic = traffic_per_tok * mean_tokens
    dec_gbs = float(r["kv_bytes"].sum() / (r["dec_ms"].sum() * 1e-3)) / 1e9
    B, Hq, Hkv, d = wl.B, wl.Hq, wl.Hkv, wl.d
    config = {"workload": args.config, "seeds": seeds, "batch": B, "num_q_heads": Hq, "num_kv_heads": Hkv,
              "head_dim": d, "page_size": wl.ps, "pool_pages": wl.traces[0][0].num_pages,
              "trace_steps": len(wl.steps),
              "timed_steps": f"{K} steps spread evenly over all {len(wl.steps)} steps of the seeds' traces",
              "l2": "flushed between steps outside the step events (256 MiB write, then 256 MiB read); "
                    f"a {args.spin_us:.0f} us GPU spin before each step keeps host enqueue out of the events",
              "variant": args.variant,
              "merge": ("separate kernel (forced)" if args.separate_merge else "the plan's choice per step") + ": "
                       + ", ".join(f"{k} x{v}" for k, v in head["merge_used"].items()),
              "variants_used": head["variants_used"], "chunk_pages_min_max": head["chunk_pages_min_max"],
              "splits_min_max": head["splits_min_max"], "parallelism": f"replicas x{world}"}
    line = {
        "metric": METRIC, "value": whole_job_rate(K * B, world, total_ms), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic", "impl": "ours", "config": config,
        "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peak, "unit": "GB/s", "frac": dec_gbs / peak,
                     "traffic": traffic, "kernel": "pkv decode_kernel",
                     "peak_source": f"hbm_gbs ({peak_kind})",
                     "algorithmic_bytes_per_launch": head["algorithmic_bytes_per_step"]},
        "decode_us_mean": head["decode_us_mean"], "step_us_mean": head["step_us_mean"],
        "merge_us_mean": head["merge_us_mean"], "build_us_mean": head["build_us_mean"],
        "step_frac": head["step_frac"], "launches_per_step": head["launches_per_step"], "by_tokens": head["by_tokens"],
        "copy_same_bytes": {"us_mean": head["copy_same_bytes_us_mean"], "frac": head["copy_same_bytes_frac"],
                            "copy_over_decode_time": head["copy_over_decode_time"],
                            "what": "one device-to-device torch copy moving each timed step's algorithmic bytes "
                                    "(half read, half written, as the measured peak), same flush / spin / event "
                                    "protocol"},
        "wall_us_per_step": wall_us, "wall_tokens_per_s": None if wall_us is None else B / (wall_us * 1e-6),
        "wall_timing": "host wall clock per step, synchronize on both sides, L2 flushed before: pkv_plan on the host "
                       "lengths then pkv_decode_step on the device-resident inputs, as C calls with their arguments "
                       "built before the loop",
        "timed_wall_s": timed_wall, "gpu_launches": r["launches"], "device_status": int(r["status"]),
        "e2e": e2e, "cpu_baseline": cpu, "clocks": clk,
    }
    del wl, r

    # ---- sub-results on the other traces (same protocol)
    subs = {}
    names = [] if args.traces in ("", "none") else [t for t in args.traces.split(",") if t != args.config]
    for name in names:
        torch.cuda.empty_cache()
        # the stress step (B = 64, ~6 GB of K/V) on the first held-out seed only: its trace takes seconds to draw
        wl = Workload(torch, name, seeds[:1] if name == "stress" else seeds, dev, args.pool_pages)
        r = time_workload(pkv, torch, wl, K, W, args, sms, dev, flush, stream)
        subs[name] = summarize(pkv, wl, r, peak)
        del wl, r
    if names:
        torch.cuda.empty_cache()
        subs["multilayer_b8_bimodal_8layers"] = run_multilayer(pkv, torch, args, sms, dev, stream, peak)
        for seed in (5, 7):  # B1 starting at 4096 and at 32768 tokens; 16 layers so that their K/V exceed the L2
            torch.cuda.empty_cache()
            subs[f"multilayer_b1_bucketed_seed{seed}_16layers"] = run_multilayer(
                pkv, torch, args, sms, dev, stream, peak, name="b1_bucketed", seed=seed, layers=16)
        torch.cuda.empty_cache()
        subs["schedules_b8_bimodal"] = run_schedules(pkv, torch, args, sms, dev, flush, stream)
    line["traces"] = subs
    if rank == 0:
        print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
