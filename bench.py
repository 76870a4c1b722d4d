#!/usr/bin/env python3
"""Tree decode-attention benchmark: one JSON line on stdout.

A step is one pst_decode_attn call over the whole batch (all PAC chunks of the
tree, every kv head, and the POR merge) on the document-QA workload: one
shared 32K-token prefix, 64 requests with unique suffixes of U{64..512}
tokens, 32 Q / 8 KV heads, d=128, bf16, 16-token pages (synthetic N(0,1)
data from a fixed seed). The metric is microseconds per step (lower is
better) with the achieved unique-KV bandwidth next to it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload document_qa|few_shot|speculative|tree_of_thought_gqa|...]

--impl reference times the fp64 CPU oracle (the only other implementation of
this computation; none of the pages ships code) on the host cores.
Under torchrun every rank runs its own replica (the path does not need a
collective); the JSON reports the slowest rank.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree decode-attn us/step (achieved unique-KV HBM GB/s vs GB300 ~8 TB/s peak)"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2**20

WORKLOADS = {
    "tiny_two_level": lambda s: s.tiny_two_level(),
    "document_qa": lambda s: s.document_qa(),
    "few_shot": lambda s: s.few_shot(),
    "speculative": lambda s: s.speculative(),
    "tree_of_thought_gqa": lambda s: s.tree_of_thought("gqa"),
    "tree_of_thought_mha": lambda s: s.tree_of_thought("mha"),
    "tree_of_thought_mqa": lambda s: s.tree_of_thought("mqa"),
    "document_qa_flat": lambda s: s.flat_control(s.document_qa()),
    "few_shot_flat": lambda s: s.flat_control(s.few_shot()),
}

DESCRIPTIONS = {
    "document_qa": "document QA: 32768-token shared prefix + 64 suffixes U{64..512}, 1 query each; "
                   "32 Q / 8 KV heads, d=128, bf16, page 16",
    "few_shot": "few-shot tree: 4000-token prefix, 16 branches x 256, 4 leaves x 32 each (64 queries); "
                "32/8 heads, d=128, bf16",
    "speculative": "speculative decoding: 8 x (8192-token prompt + 64-node draft tree, depth 6, all "
                   "drafts queried); 32/8 heads, d=128, bf16",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=30)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="document_qa", choices=sorted(WORKLOADS))
    ap.add_argument("--timed-steps", type=int, default=256, help="steps with per-kernel events")
    ap.add_argument("--cpu-sample-s", type=float, default=12.0)
    ap.add_argument("--ref-budget-s", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--plan-opt", action="append", default=[],
                    help="planner option key=value (split_policy, fixed_chunk, tc_min_rows, tc_engine, ...)")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_sources_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "prefix_shared_tree_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from a committed ncu summary, if its
    kernel sources are the ones built now."""
    p = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("sources_sha") != kernel_sources_sha():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(workload, budget_s, n_queries):
    """Time the fp64 oracle on queries of the workload in a single-threaded
    subprocess (BLAS pinned to one thread); returns the extrapolated us/step."""
    code = f"""
import os, sys, time, json
sys.path.insert(0, {ROOT!r})
import numpy as np
import synth
from oracle import attention as oa
sys.path.insert(0, {ROOT!r})
import bench
wl = bench.WORKLOADS[{workload!r}](synth)
K, V = wl.kv_pools()
Q = wl.q()
order = [(i * 37) % wl.n_queries for i in range(wl.n_queries)]
oa.decode_attention(wl, K, V, Q, [order[0]])          # warm-up
done, t0 = 0, time.perf_counter()
while time.perf_counter() - t0 < {budget_s}:
    oa.decode_attention(wl, K, V, Q, [order[(done + 1) % len(order)]])
    done += 1
    if done >= wl.n_queries:
        break
el = time.perf_counter() - t0
print(json.dumps({{"queries": done, "seconds": el}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=budget_s * 4 + 300)
    if r.returncode != 0:
        raise RuntimeError("cpu baseline failed: " + r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    per_q = d["seconds"] / d["queries"]
    return {"value": per_q * n_queries * 1e6, "unit": "us/step", "cores": 1, "kind": "oracle",
            "sample": f"{d['queries']} of {n_queries} queries (all heads, fp64) timed single-threaded "
                      f"in {d['seconds']:.1f} s, scaled to the full batch"}


def rotating_copies(U):
    """Device copies of the inputs the timed loop rotates over (their total exceeds L2)."""
    return max(2, math.ceil(3 * L2_BYTES / max(U, 1)))


def bench_config(args, wl, world):
    """The `config` object of a bench line (shared by both arms)."""
    U = wl.unique_kv_bytes()
    copies = rotating_copies(U)
    return {
        "workload": args.workload + (": " + DESCRIPTIONS[args.workload] if args.workload in DESCRIPTIONS else ""),
        "n_queries": wl.n_queries, "n_q_heads": wl.n_q_heads, "n_kv_heads": wl.n_kv_heads, "d": wl.d,
        "unique_kv_bytes": U, "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
        "l2": f"inputs rotate over {copies} device copies ({copies * U / 2**20:.0f} MiB > L2 129 MiB)",
    }


# ------------------------------------------------------------------ arms

def max_over_ranks(values, world, device="cpu"):
    """Per-rank timings -> their maximum over the ranks (every rank gets it).
    Replicas run independently; the job's step time is the slowest replica's.
    `device` is where the collective's tensor lives (cuda for NCCL, cpu for gloo)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def run_ours(args, rank, world):
    import numpy as np
    import torch

    import synth
    from prefix_shared_tree_gb300 import build as _build
    _build.build()
    from prefix_shared_tree_gb300 import pst
    from prefix_shared_tree_gb300.torch_api import TreeDecodeAttention, to_device

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = WORKLOADS[args.workload](synth)
    K_np, V_np = wl.kv_pools()
    Q_np = wl.q()
    U = wl.unique_kv_bytes()
    copies = rotating_copies(U)
    Kd = [to_device(K_np, wl.dtype, dev)]
    Vd = [to_device(V_np, wl.dtype, dev)]
    Qd = [to_device(Q_np, wl.dtype, dev)]
    for _ in range(copies - 1):
        Kd.append(Kd[0].clone())
        Vd.append(Vd[0].clone())
        Qd.append(Qd[0].clone())
    del K_np, V_np

    t0 = time.perf_counter()
    plan_opts = {}
    for kv in args.plan_opt:
        k, v = kv.split("=", 1)
        plan_opts[k] = int(v) if v.lstrip("-").isdigit() else v
    att = TreeDecodeAttention.from_workload(wl, device=dev, **plan_opts)
    plan_wall_us = (time.perf_counter() - t0) * 1e6
    st = att.plan.stats()
    # the next decode step's plan on the same tree (host only, not uploaded)
    update_us = pst.plan_update(att.plan, att.tree).stats()["plan_us"]
    ex = att.plan.export()
    O = [torch.empty((wl.n_queries, wl.n_q_heads, wl.d), dtype=torch.float32, device=dev) for _ in range(copies)]
    L = [torch.empty((wl.n_queries, wl.n_q_heads), dtype=torch.float32, device=dev) for _ in range(copies)]
    stream = torch.cuda.current_stream(dev)

    for i in range(max(3, args.warmup)):
        c = i % copies
        att(Qd[c], Kd[c], Vd[c], O[c], L[c])
    torch.cuda.synchronize(dev)
    if att.check_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    timer = pst.Timer(max(1, min(args.timed_steps, args.steps)))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        ev0.record(stream)
        for i in range(args.steps):
            c = i % copies
            att(Qd[c], Kd[c], Vd[c], O[c], L[c], timer=timer if i < args.timed_steps else None)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    total_ms = ev0.elapsed_time(ev1)
    kern_ms, kern_calls = timer.read()
    if att.check_status() != 0:
        raise RuntimeError("device status word set during the timed region")

    # e2e: per step, Q from pinned host -> device, decode, O and LSE back to pinned host
    Qh = torch.from_numpy(Q_np.view(np.int16) if wl.dtype == "bf16" else Q_np).pin_memory()
    Oh = torch.empty(O[0].shape, dtype=torch.float32).pin_memory()
    Lh = torch.empty(L[0].shape, dtype=torch.float32).pin_memory()
    Qstage = torch.empty(Qh.shape, dtype=Qh.dtype, device=dev)
    e2e_steps = max(10, args.steps // 4)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        c = i % copies
        Qstage.copy_(Qh, non_blocking=True)
        qv = Qstage.view(torch.bfloat16) if wl.dtype == "bf16" else Qstage
        att(qv, Kd[c], Vd[c], O[c], L[c])
        Oh.copy_(O[c], non_blocking=True)
        Lh.copy_(L[c], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_us = e0.elapsed_time(e1) * 1e3 / e2e_steps

    us = total_ms * 1e3 / args.steps
    us, e2e_us = max_over_ranks([us, e2e_us], world, dev)
    if rank != 0:
        return None

    peak, peak_src = measured_peaks()
    achieved_gbs = U / (us * 1e-6) / 1e9
    # per-kernel algorithmic bytes: unique KV of the chunks each PAC kernel reads
    per_tok = wl.n_kv_heads * 2 * wl.d * wl.elem_bytes
    ntok = np.diff(ex["chunk_tok_ptr"])
    kinds = ex["chunk_kind"]
    # tensor-core chunks shorter than p_bf16_min_tokens run in the exact-P launch (tcgen05 engine)
    thr = int(plan_opts.get("p_bf16_min_tokens", 0)) or 1024
    thr = np.inf if thr < 0 else thr
    tok_ptr = ex["chunk_tok_ptr"]
    node_tokens = np.array([wl.node_len[ex["chunk_tok_node"][tok_ptr[c]:tok_ptr[c + 1]]].max()
                            if len(set(ex["chunk_tok_node"][tok_ptr[c]:tok_ptr[c + 1]].tolist())) == 1 else 0
                            for c in range(len(ntok))])
    exact = (kinds == 1) & (node_tokens < thr) & (plan_opts.get("tc_engine", "tcgen05") == "tcgen05")
    alg = {"pac_tc": int(ntok[(kinds == 1) & ~exact].sum()) * per_tok,
           "pac_tc_exact": int(ntok[exact].sum()) * per_tok,
           "pac_thin": int(ntok[kinds == 0].sum()) * per_tok,
           "por": int(st["n_partial_rows"]) * (wl.d * 4 + 4) + wl.n_queries * wl.n_q_heads * (wl.d * 4 + 4)}
    shares = {k: v / max(1e-9, sum(kern_ms.values())) for k, v in kern_ms.items()}
    # the PAC launch groups start together; each group's time runs from the
    # call's start to its end. The dominant kernel is the one with the most bytes.
    dom = max(("pac_tc", "pac_tc_exact", "pac_thin"), key=lambda k: alg[k])
    dom_ms = kern_ms[dom] / max(1, kern_calls)
    dom_achieved = alg[dom] / (dom_ms * 1e-3) / 1e9
    traffic = recorded_traffic(dom, args.workload)
    clocks = clk.summary()
    line = {
        "metric": METRIC,
        "value": round(us, 3),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(us / 1e3, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded N(0,1) K/V/Q, shapes of the CoDec/DEFT workloads)",
        "config": bench_config(args, wl, world),
        "achieved_unique_kv_gbs": round(achieved_gbs, 1),
        "frac_of_8tbs": round(achieved_gbs / NOMINAL_HBM_GBS, 4),
        "frac_of_measured_hbm": round(achieved_gbs / peak, 4),
        "kernel_ms_share": {k: round(v, 4) for k, v in shares.items()},
        "kernel_us_per_call": {k: round(v * 1e3 / max(1, kern_calls), 3) for k, v in kern_ms.items()},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(dom_achieved, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(dom_achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": alg[dom]},
        "plan": {"plan_us": round(st["plan_us"], 1), "plan_wall_us": round(plan_wall_us, 1),
                 "plan_update_us": round(update_us, 1),
                 "predicted_makespan_us": round(st["predicted_makespan_us"], 2),
                 "n_chunks": st["n_chunks"], "n_items": st["n_items"], "n_tc_items": st["n_tc_items"],
                 "n_cc_items": st["n_cc_items"], "n_partial_rows": st["n_partial_rows"]},
        "e2e": {"value": round(e2e_us, 3), "unit": "us/step", "h2d_bytes_per_step": int(Qh.numel() * Qh.element_size()),
                "d2h_bytes_per_step": int(Oh.numel() * 4 + Lh.numel() * 4)},
        "gpu_launches": int(st["n_launches"]) * args.steps,
        "clocks": clocks,
    }
    return line, wl


def run_reference(args, rank):
    if rank != 0:
        return None
    import numpy as np  # noqa: F401

    import synth
    from oracle import attention as oa

    wl = WORKLOADS[args.workload](synth)
    K, V = wl.kv_pools()
    Q = wl.q()
    order = [(i * 37) % wl.n_queries for i in range(wl.n_queries)]
    oa.decode_attention(wl, K, V, Q, [order[0]])             # one untimed warm-up query
    t0 = time.perf_counter()
    done = 0
    while done < args.steps and time.perf_counter() - t0 < args.ref_budget_s:
        oa.decode_attention(wl, K, V, Q, [order[(done + 1) % len(order)]])
        done += 1
    el = time.perf_counter() - t0
    us = el / done * wl.n_queries * 1e6
    ncpu = 1
    try:
        import threadpoolctl  # noqa: F401
        ncpu = max(i.get("num_threads", 1) for i in threadpoolctl.threadpool_info()) or 1
    except Exception:
        ncpu = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    sample = (f"{done} of {args.steps} requested steps ran within {args.ref_budget_s:.0f} s; each timed one "
              f"query (all heads) of the batch; us/step = mean per query x {wl.n_queries} queries")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(us, 1),
        "unit": "us/step",
        "n_gpus": 1,
        "steps": done,
        "warmup": 1,
        "ms_per_step": round(us / 1e3, 3),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": bench_config(args, wl, 1),
        "cpu_baseline": {"value": round(us, 1), "unit": "us/step", "cores": ncpu, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(us, 1), "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    out = run_ours(args, rank, world)
    if out is not None:
        line, wl = out
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_sample_s, wl.n_queries)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
