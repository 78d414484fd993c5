"""Decode-step benchmark: paged GQA decode attention on one GB300 per rank.

One step = one decode step of the trace (plan, worklist build when the plan uses the workqueue, decode, merge)
over one batch of synthetic inputs. Default workload: the B1 bucketed long-context trace (B=1, Hq=32, Hkv=8, d=128,
page size 16, fp16 ~N(0,1), start length from {4096, 8192, 16384, 32768}, 64 steps of +1 token per seed, pages
shuffled in a 2^16-page pool) over the held-out seeds 5-9, cycled until K steps have run.

Timing: every step is bracketed by CUDA events on the launching stream; the decode kernel alone by a second pair.
Between steps an L2 flush runs outside the step's events: a 256 MiB write (larger than the 129 MB L2), then a
256 MiB read of another buffer, so every step reads its KV from HBM, as it would after the other layers of a model
ran, and starts with an L2 that holds no dirty lines (the write-back of the flush buffer is not charged to the step). `value` = tokens / sum of step
times. `e2e` repeats the steps through the same C ABI from pinned host buffers: per step the host->device copies of
q, seq_lens, the block table and the new token's K/V, the step, and the device->host copy of out, all inside the
events. `cpu_baseline` times the fp64 oracle on the host on a bounded sample of the same trace steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config b1_bucketed] ...
Under torchrun (N > 1) every rank runs the same workload on its own GPU (replicas; no collective in the data
path); rank 0 prints one JSON line with value = tokens of all ranks / max over ranks of the timed time.
"""

from __future__ import annotations

import argparse
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
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_kernel_b1_bucketed.md")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="b1_bucketed")
    ap.add_argument("--seeds", default=",".join(map(str, HELD_OUT)))
    ap.add_argument("--variant", choices=["auto", "single", "split", "workqueue"], default="auto")
    ap.add_argument("--chunk", type=int, default=0, help="pages per split for a forced variant")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the oracle cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
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
    """(dram bytes per token of KV, kernel hash) from the committed ncu summary, if present."""
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


class ClockSampler:
    """nvidia-smi clocks/throttle sampler (200 ms) around the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True):
        self.proc = None
        self.gpu_index = gpu_index
        self.lines = []
        self.t_start = self.t_stop = None
        if enabled:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                     "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None

    def mark_start(self):
        self.t_start = time.time()

    def mark_stop(self):
        self.t_stop = time.time()

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
def build_workload(config: str, seeds, dev, pool_pages: int = 0):
    """Device tensors for every step of every trace: pools with all pages a trace will use, per-step q, block
    table and lengths. Returns a list of step records."""
    import torch

    from workloads import make_trace

    steps = []
    traces = []
    for seed in seeds:
        tr = make_trace(config, seed, pool_pages=pool_pages or None)
        ps, hkv, d = tr.ps, tr.hkv, tr.d
        k = torch.empty((tr.num_pages, ps, hkv, d), dtype=torch.float16, device=dev)
        v = torch.empty((tr.num_pages, ps, hkv, d), dtype=torch.float16, device=dev)
        idx = torch.from_numpy(tr.used_pages).to(dev)
        k.index_copy_(0, idx, torch.from_numpy(tr.k_pages).to(dev))
        v.index_copy_(0, idx, torch.from_numpy(tr.v_pages).to(dev))
        traces.append((tr, k, v))
        for t in range(tr.steps):
            lens = tr.seq_lens(t)
            bt = tr.block_table(t)
            q = tr.q(t)
            # the token appended at this step: row b's newest token (index L-1) and its page/slot
            new_phys = bt[np.arange(tr.batch), (lens - 1) // ps]
            new_slot = (lens - 1) % ps
            steps.append({"trace": len(traces) - 1, "t": t, "lens_host": lens, "bt_host": bt, "q_host": q,
                          "q": torch.from_numpy(q).to(dev), "bt": torch.from_numpy(bt).to(dev),
                          "lens": torch.from_numpy(lens).to(dev), "new_phys": new_phys, "new_slot": new_slot})
    return traces, steps


def decode_fit(kv_bytes, dec_ms):
    """Least-squares fit of decode time = fixed + bytes / bandwidth over the timed steps."""
    if len(set(np.round(kv_bytes / 1e6, 3))) < 2:
        return None
    slope, icpt = np.polyfit(kv_bytes, dec_ms * 1e3, 1)
    return {"fixed_us": float(icpt), "incremental_gbs": float(1e-3 / slope) if slope > 0 else None}


def make_plan(pkv, problem, lens, sms, args):
    if args.variant == "auto":
        return pkv.pkv_plan(problem, lens, sms)
    v = {"single": pkv.PKV_VARIANT_SINGLE, "split": pkv.PKV_VARIANT_SPLIT,
         "workqueue": pkv.PKV_VARIANT_WORKQUEUE}[args.variant]
    chunk = args.chunk
    if chunk <= 0:
        pmax = int(((lens.astype(np.int64) + 15) // 16).max())
        chunk = max(1, -(-pmax // 32))
    return pkv.pkv_plan_fixed(problem, lens, sms, v, chunk)


# ------------------------------------------------------------------------------------------------ oracle legs
def oracle_baseline(config, seeds, budget_s):
    """Times the fp64 oracle on whole trace steps (all query heads) until the budget is spent."""
    import oracle
    from workloads import make_trace

    done_tokens, spent, n_steps = 0, 0.0, 0
    for seed in seeds:
        tr = make_trace(config, seed)
        kp, vp = tr.host_pools()
        for t in range(0, tr.steps, 16):
            t0 = time.perf_counter()
            oracle.attention(tr.q(t), kp, vp, tr.block_table(t), tr.seq_lens(t))
            spent += time.perf_counter() - t0
            done_tokens += tr.batch
            n_steps += 1
            if spent >= budget_s:
                break
        if spent >= budget_s:
            break
    return {"value": done_tokens / spent, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n_steps} full {config} trace steps (every 16th step of the held-out seeds), all "
                      f"{make_trace(config, seeds[0]).hq} query heads per row, fp64, {spent:.1f} s"}


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

    def one(k, npairs):
        i, t = order[k % len(order)]
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
    spent = sum(one(args.warmup + k, npairs) for k in range(args.steps))
    tokens = args.steps * npairs / (B * Hq)
    value = tokens / spent
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * spent / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": args.config, "seeds": seeds, "batch": B, "num_q_heads": Hq,
                       "num_kv_heads": traces[0][0].hkv, "head_dim": traces[0][0].d, "page_size": traces[0][0].ps},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{npairs} of {B * Hq} (row, query head) pairs of one trace step per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------------ our arm
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
    traces, steps = build_workload(args.config, seeds, dev, args.pool_pages)
    tr0 = traces[0][0]
    B, Hq, Hkv, d = tr0.batch, tr0.hq, tr0.hkv, tr0.d
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    scale = 1.0 / math.sqrt(d)
    problems = [pkv.make_problem(B, Hq, Hkv, d, tr.ps, tr.num_pages, tr.max_pages) for tr, _, _ in traces]

    # plans for every trace step (host planning is timed separately, in the wall loop)
    t0 = time.perf_counter()
    plans = [make_plan(pkv, problems[s["trace"]], s["lens_host"], sms, args) for s in steps]
    plan_us = 1e6 * (time.perf_counter() - t0) / len(steps)
    ws = pkv.alloc_workspace(max(p.ws_bytes for p in plans), dev)
    out = torch.empty((B, Hq, d), dtype=torch.float16, device=dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream(dev)

    def launch(k):
        s = steps[k % len(steps)]
        tr, kpool, vpool = traces[s["trace"]]
        pkv.pkv_decode_step(plans[k % len(steps)], problems[s["trace"]], s["q"], kpool, vpool, s["bt"], s["lens"],
                            scale, ws, out, stream)

    for k in range(args.warmup):
        flush()
        launch(k)
    torch.cuda.synchronize()
    if pkv.pkv_read_status(ws) != 0:
        raise SystemExit("device status set during warm-up")

    # ---- timed region: K steps, events per step and around the decode kernel
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(local, enabled=not args.no_clocks)
    time.sleep(0.3 if not args.no_clocks else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.mark_start()
    wall0 = time.perf_counter()
    launches = 0
    for k in range(K):
        j = (args.warmup + k) % len(steps)
        s = steps[j]
        tr, kpool, vpool = traces[s["trace"]]
        plan, problem = plans[j], problems[s["trace"]]
        flush()
        e = ev[k]
        e[0].record(stream)
        if plan.variant == pkv.PKV_VARIANT_WORKQUEUE:
            pkv.pkv_build_worklist(plan, problem, s["lens"], ws, stream)
        e[1].record(stream)
        pkv.pkv_decode(plan, problem, s["q"], kpool, vpool, s["bt"], s["lens"], scale, ws, out, stream)
        e[2].record(stream)
        pkv.pkv_merge(plan, problem, ws, out, stream)
        e[3].record(stream)
        launches += pkv.pkv_plan_launches(plan)
    torch.cuda.synchronize()
    wall_timed = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clocks.mark_stop()
    step_ms = np.array([e[0].elapsed_time(e[3]) for e in ev])
    dec_ms = np.array([e[1].elapsed_time(e[2]) for e in ev])
    build_ms = np.array([e[0].elapsed_time(e[1]) for e in ev])
    merge_ms = np.array([e[2].elapsed_time(e[3]) for e in ev])
    kv_bytes = np.array([plans[(args.warmup + k) % len(steps)].kv_bytes for k in range(K)])
    tokens = K * B
    total_ms = float(step_ms.sum())
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    status = pkv.pkv_read_status(ws)

    # ---- synchronized wall time per step (pages' protocol): plan + launches + sync, no flush inside
    wall = []
    for k in range(min(K, 2 * len(steps))):
        j = k % len(steps)
        s = steps[j]
        tr, kpool, vpool = traces[s["trace"]]
        flush()
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        plan = make_plan(pkv, problems[s["trace"]], s["lens_host"], sms, args)
        pkv.pkv_decode_step(plan, problems[s["trace"]], s["q"], kpool, vpool, s["bt"], s["lens"], scale, ws, out,
                            stream)
        torch.cuda.synchronize()
        wall.append(time.perf_counter() - w0)
    wall_us = 1e6 * float(np.mean(wall))

    # ---- e2e through the C ABI from pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, pkv, torch, traces, steps, plans, problems, ws, flush, stream, scale, dev)

    peak, peak_kind = measured_peaks()
    achieved = float(kv_bytes.sum() / (dec_ms.sum() * 1e-3)) / 1e9
    traffic_per_tok, traffic_hash = profile_traffic()
    traffic = None
    if traffic_per_tok is not None and traffic_hash == kernel_source_hash():
        mean_tokens = float(np.mean([int(steps[(args.warmup + k) % len(steps)]["lens_host"].sum())
                                     for k in range(K)]))
        traffic = traffic_per_tok * mean_tokens
    clk = clocks.finish()

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world >= 1:
        cpu = oracle_baseline(args.config, seeds, args.cpu_seconds)
    variants = sorted({pkv.VARIANT_NAMES[plans[(args.warmup + k) % len(steps)].variant] for k in range(K)})
    splits = [plans[(args.warmup + k) % len(steps)].num_splits for k in range(K)]
    line = {
        "metric": METRIC, "value": tokens * world / (total_ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 in, f32 accumulate", "data": "synthetic",
        "impl": "ours",
        "config": {"workload": args.config, "seeds": seeds, "batch": B, "num_q_heads": Hq, "num_kv_heads": Hkv,
                   "head_dim": d, "page_size": tr0.ps, "pool_pages": tr0.num_pages, "trace_steps": len(steps),
                   "l2": "flushed between steps outside the step events (256 MiB write, then 256 MiB read)",
                   "variant": args.variant, "variants_used": variants,
                   "splits_min_max": [int(min(splits)), int(max(splits))], "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "kernel": "pkv decode_kernel", "peak_source": f"hbm_gbs ({peak_kind})",
                     "algorithmic_bytes_per_step": float(kv_bytes.mean())},
        "decode_us_mean": 1e3 * float(dec_ms.mean()), "step_us_mean": 1e3 * float(step_ms.mean()),
        "build_us_mean": 1e3 * float(build_ms.mean()), "merge_us_mean": 1e3 * float(merge_ms.mean()),
        "decode_fit": decode_fit(kv_bytes, dec_ms),
        "step_us_p50": 1e3 * float(np.median(step_ms)), "kv_gbs_step": float(kv_bytes.sum() / (step_ms.sum() * 1e-3)) / 1e9,
        "wall_us_per_step": wall_us, "wall_tokens_per_s": B / (wall_us * 1e-6), "plan_us": plan_us,
        "timed_wall_s": wall_timed, "gpu_launches": launches, "device_status": status,
        "e2e": e2e, "cpu_baseline": cpu, "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def run_e2e(args, pkv, torch, traces, steps, plans, problems, ws, flush, stream, scale, dev):
    """Steps through the C ABI with pinned host inputs/outputs; the copies are inside the events."""
    B = traces[0][0].batch
    nsteps = min(args.steps, len(steps))
    host = []
    for s in steps[:nsteps]:
        tr, kpool, vpool = traces[s["trace"]]
        ps = tr.ps
        rows = np.arange(tr.batch)
        # K/V of each row's newest token: [B, Hkv, d] from the trace's page contents
        used_index = {int(p): i for i, p in enumerate(tr.used_pages)}
        k_new = np.stack([tr.k_pages[used_index[int(s["new_phys"][b])], int(s["new_slot"][b])] for b in rows])
        v_new = np.stack([tr.v_pages[used_index[int(s["new_phys"][b])], int(s["new_slot"][b])] for b in rows])
        host.append({"q": torch.from_numpy(s["q_host"]).pin_memory(), "bt": torch.from_numpy(s["bt_host"]).pin_memory(),
                     "lens": torch.from_numpy(s["lens_host"]).pin_memory(),
                     "k_new": torch.from_numpy(k_new).pin_memory(), "v_new": torch.from_numpy(v_new).pin_memory()})
    out_host = torch.empty((B, traces[0][0].hq, traces[0][0].d), dtype=torch.float16).pin_memory()
    q_d = torch.empty_like(steps[0]["q"])
    bt_d = [torch.empty((B, tr.max_pages), dtype=torch.int32, device=dev) for tr, _, _ in traces]
    lens_d = torch.empty((B,), dtype=torch.int32, device=dev)
    out_d = torch.empty_like(q_d)
    times, h2d, d2h = [], 0, 0
    for k in range(nsteps):
        s, hs = steps[k], host[k]
        tr, kpool, vpool = traces[s["trace"]]
        plan = plans[k]
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        q_d.copy_(hs["q"], non_blocking=True)
        bt_view = bt_d[s["trace"]]
        bt_view.copy_(hs["bt"], non_blocking=True)
        lens_d.copy_(hs["lens"], non_blocking=True)
        for b in range(tr.batch):  # append the new token's K and V into its page slot
            kpool[int(s["new_phys"][b]), int(s["new_slot"][b])].copy_(hs["k_new"][b], non_blocking=True)
            vpool[int(s["new_phys"][b]), int(s["new_slot"][b])].copy_(hs["v_new"][b], non_blocking=True)
        pkv.pkv_decode_step(plan, problems[s["trace"]], q_d, kpool, vpool, bt_view, lens_d, scale, ws, out_d, stream)
        out_host.copy_(out_d, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
        h2d = hs["q"].numel() * 2 + hs["bt"].numel() * 4 + hs["lens"].numel() * 4 + 2 * hs["k_new"].numel() * 2
        d2h = out_host.numel() * 2
    return {"value": B * nsteps / (1e-3 * float(np.sum(times))), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": nsteps, "us_per_step": 1e3 * float(np.mean(times))}


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
