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
    "speculative_flat": lambda s: s.flat_control(s.speculative()),
}

# configurations measured next to the headline in the same run (the other
# workloads of the pages, and the no-sharing flat controls of the shared ones)
PER_CONFIG = ["few_shot", "speculative", "tree_of_thought_gqa", "tree_of_thought_mha", "tree_of_thought_mqa",
              "tiny_two_level", "document_qa_flat", "few_shot_flat", "speculative_flat"]

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
    ap.add_argument("--timer-steps", type=int, default=64,
                    help="steps of a separate loop with the library's per-group events (after the timed loop)")
    ap.add_argument("--no-per-config", action="store_true", help="skip the other workloads")
    ap.add_argument("--per-config", default=",".join(PER_CONFIG), help="comma-separated workloads for per_config")
    ap.add_argument("--no-mla", action="store_true", help="leave the MLA entry out of per_config")
    ap.add_argument("--cpu-sample-s", type=float, default=12.0)
    ap.add_argument("--ref-budget-s", type=float, default=150.0,
                    help="host seconds the reference arm's warm-up and timed steps may take")
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
    """Digest of the sources that build the kernels (.cu, .cuh and .h under
    csrc). The host planner's sources are left out: what it produces enters a
    traffic record through the plan digest."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "prefix_shared_tree_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def plan_digest(plan):
    """Digest of a plan: its exported index, chunks and merge lists, and its
    stats without the host time. A launch's DRAM traffic depends on the
    kernels and on the items the plan gives them."""
    import numpy as np
    h = hashlib.sha256()
    ex = plan.export()
    for k in sorted(ex):
        h.update(k.encode())
        h.update(np.ascontiguousarray(ex[k]).tobytes())
    st = {k: v for k, v in plan.stats().items() if k != "plan_us"}
    h.update(json.dumps(st, sort_keys=True, default=float).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload, digest):
    """DRAM bytes per launch of `kernel` from a committed ncu summary, if it
    was taken with the kernels built now and with the same plan."""
    p = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("sources_sha") != kernel_sources_sha() or d.get("plan_digest") != digest:
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


def _plan_opts(args):
    plan_opts = {}
    for kv in args.plan_opt:
        k, v = kv.split("=", 1)
        plan_opts[k] = int(v) if v.lstrip("-").isdigit() else v
    return plan_opts


def device_inputs(name, dev, copies):
    """(workload, [K], [V], [Q], Q host array): `copies` device copies of the
    pools and queries. A flat control's pools are filled on the device from
    its shared workload's pools (a token's K/V depend on its logical id only)."""
    import numpy as np
    import torch

    import synth
    from prefix_shared_tree_gb300.torch_api import to_device
    if name.endswith("_flat"):
        base = WORKLOADS[name[:-len("_flat")]](synth)
        wl = synth.flat_control(base)
        Kb, Vb = base.kv_pools()
        src = torch.from_numpy(np.maximum(synth.source_rows(base, wl), 0)).to(dev)

        def gather(pool):
            P, H, S, D = pool.shape
            rows = to_device(pool, wl.dtype, dev).permute(0, 2, 1, 3).reshape(P * S, H, D)
            out = rows[src].reshape(wl.num_pages, S, H, D).permute(0, 2, 1, 3).contiguous()
            del rows
            return out
        Kd, Vd = [gather(Kb)], [gather(Vb)]
        del Kb, Vb
    else:
        wl = WORKLOADS[name](synth)
        K_np, V_np = wl.kv_pools()
        Kd, Vd = [to_device(K_np, wl.dtype, dev)], [to_device(V_np, wl.dtype, dev)]
        del K_np, V_np
    Q_np = wl.q()
    Qd = [to_device(Q_np, wl.dtype, dev)]
    for _ in range(copies - 1):
        Kd.append(Kd[0].clone())
        Vd.append(Vd[0].clone())
        Qd.append(Qd[0].clone())
    return wl, Kd, Vd, Qd, Q_np


def algorithmic_bytes(wl, ex, st, plan_opts):
    """Unique K/V bytes of the chunks each PAC launch group reads, and POR's
    partial-row traffic."""
    import numpy as np
    per_tok = wl.n_kv_heads * 2 * wl.d * wl.elem_bytes
    ntok = np.diff(ex["chunk_tok_ptr"])
    kinds = ex["chunk_kind"]
    # tensor-core chunks of nodes shorter than p_bf16_min_tokens run in the exact-P launch (tcgen05 engine)
    thr = int(plan_opts.get("p_bf16_min_tokens", 0)) or 1024
    thr = np.inf if thr < 0 else thr
    tok_ptr = ex["chunk_tok_ptr"]
    node_tokens = np.array([wl.node_len[ex["chunk_tok_node"][tok_ptr[c]:tok_ptr[c + 1]]].max()
                            if len(set(ex["chunk_tok_node"][tok_ptr[c]:tok_ptr[c + 1]].tolist())) == 1 else 0
                            for c in range(len(ntok))])
    exact = (kinds == 1) & (node_tokens < thr) & (plan_opts.get("tc_engine", "tcgen05") == "tcgen05")
    return {"pac_tc": int(ntok[(kinds == 1) & ~exact].sum()) * per_tok,
            "pac_tc_exact": int(ntok[exact].sum()) * per_tok,
            "pac_thin": int(ntok[kinds == 0].sum()) * per_tok,
            "por": int(st["n_partial_rows"]) * (wl.d * 4 + 4) + wl.n_queries * wl.n_q_heads * (wl.d * 4 + 4)}


def measure(name, args, dev, steps, warmup, timer_steps, plan_opts, e2e=False, world=1):
    """Times `steps` decode steps of workload `name` (after `warmup`), with no
    per-group events inside the timed loop; then `timer_steps` steps with the
    library's per-group events; optionally the end-to-end loop. Returns a dict
    (times in us)."""
    import numpy as np
    import torch

    from prefix_shared_tree_gb300 import pst
    from prefix_shared_tree_gb300.torch_api import TreeDecodeAttention

    peak, _ = measured_peaks()
    # rotate over device copies whose total exceeds L2 (the flat controls are far larger)
    probe = WORKLOADS[name[:-5] if name.endswith("_flat") else name]
    copies_hint = None
    wl0 = None
    if not name.endswith("_flat"):
        import synth
        wl0 = probe(synth)
        copies_hint = rotating_copies(wl0.unique_kv_bytes())
    wl, Kd, Vd, Qd, Q_np = device_inputs(name, dev, copies_hint or 2)
    U = wl.unique_kv_bytes()
    copies = len(Kd)
    t0 = time.perf_counter()
    att = TreeDecodeAttention.from_workload(wl, device=dev, **plan_opts)
    plan_wall_us = (time.perf_counter() - t0) * 1e6
    st = att.plan.stats()
    update_us = pst.plan_update(att.plan, att.tree).stats()["plan_us"]
    ex = att.plan.export()
    O = [torch.empty((wl.n_queries, wl.n_q_heads, wl.d), dtype=torch.float32, device=dev) for _ in range(copies)]
    L = [torch.empty((wl.n_queries, wl.n_q_heads), dtype=torch.float32, device=dev) for _ in range(copies)]
    stream = torch.cuda.current_stream(dev)
    for i in range(max(3, warmup)):
        c = i % copies
        att(Qd[c], Kd[c], Vd[c], O[c], L[c])
    torch.cuda.synchronize(dev)
    if att.check_status() != 0:
        raise RuntimeError(f"{name}: device status word set during warm-up")

    # ---- the timed loop: plain calls, CUDA events on the launching stream
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        ev0.record(stream)
        for i in range(steps):
            c = i % copies
            att(Qd[c], Kd[c], Vd[c], O[c], L[c])
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    us = ev0.elapsed_time(ev1) * 1e3 / steps
    if att.check_status() != 0:
        raise RuntimeError(f"{name}: device status word set during the timed region")

    # ---- the same steps replayed from CUDA graphs (one capture per input copy)
    graphs = [att.capture(Qd[c], Kd[c], Vd[c], O[c], L[c]) for c in range(copies)]
    torch.cuda.synchronize(dev)
    gv0, gv1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gv0.record(stream)
    for i in range(steps):
        graphs[i % copies].replay()
    gv1.record(stream)
    torch.cuda.synchronize(dev)
    graph_us = gv0.elapsed_time(gv1) * 1e3 / steps

    # ---- one step at a time from an idle GPU: the latency of a single call
    def _single(fn, n=30):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for i in range(n):
            torch.cuda.synchronize(dev)
            a.record(stream)
            fn(i)
            b.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b) * 1e3)
        return float(statistics.median(ts))
    single_us = _single(lambda i: att(Qd[i % copies], Kd[i % copies], Vd[i % copies], O[i % copies], L[i % copies]))
    single_graph_us = _single(lambda i: graphs[i % copies].replay())
    del graphs
    if att.check_status() != 0:
        raise RuntimeError(f"{name}: device status word set during the graph replays")

    # ---- per launch group: a separate loop with the library's events
    timer = pst.Timer(max(1, timer_steps))
    for i in range(max(1, timer_steps)):
        c = i % copies
        att(Qd[c], Kd[c], Vd[c], O[c], L[c], timer=timer)
    kern_ms, kern_calls = timer.read()
    group_us = {k: round(v * 1e3 / max(1, kern_calls), 3) for k, v in kern_ms.items()}

    alg = algorithmic_bytes(wl, ex, st, plan_opts)
    dom = max(("pac_tc", "pac_tc_exact", "pac_thin"), key=lambda k: alg[k])
    dom_us = group_us[dom]
    dom_achieved = alg[dom] / (dom_us * 1e-6) / 1e9 if dom_us > 0 else 0.0
    out = {
        "workload": name, "wl": wl, "us": us, "graph_us": graph_us, "U": U, "copies": copies,
        "single_us": single_us, "single_graph_us": single_graph_us,
        "clocks": clk.summary(),
        "plan": {"plan_us": round(st["plan_us"], 1), "plan_wall_us": round(plan_wall_us, 1),
                 "plan_update_us": round(update_us, 1),
                 "predicted_makespan_us": round(st["predicted_makespan_us"], 2),
                 "split_policy": {0: "cost_model", 1: "none", 2: "uniform", 3: "flatten"}[int(st["split_policy"])],
                 "fixed_chunk": int(st["fixed_chunk"]),
                 "n_chunks": st["n_chunks"], "n_items": st["n_items"], "n_tc_items": st["n_tc_items"],
                 "n_cc_items": st["n_cc_items"], "n_partial_rows": st["n_partial_rows"],
                 "digest": plan_digest(att.plan)},
        "n_launches": int(st["n_launches"]),
        "group_end_us": {k: v for k, v in group_us.items() if k != "por"},
        "por_us": group_us["por"],
        "alg": alg, "dom": dom, "dom_us": dom_us, "dom_achieved": dom_achieved, "peak": peak,
    }
    if e2e:
        # per step: Q from pinned host memory to the device, decode, O and LSE back to pinned host memory
        Qh = torch.from_numpy(Q_np.view(np.int16) if wl.dtype == "bf16" else Q_np).pin_memory()
        Oh = torch.empty(O[0].shape, dtype=torch.float32).pin_memory()
        Lh = torch.empty(L[0].shape, dtype=torch.float32).pin_memory()
        Qstage = torch.empty(Qh.shape, dtype=Qh.dtype, device=dev)
        e2e_steps = max(10, steps // 4)
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
        out["e2e_us"] = e0.elapsed_time(e1) * 1e3 / e2e_steps
        out["h2d"] = int(Qh.numel() * Qh.element_size())
        out["d2h"] = int(Oh.numel() * 4 + Lh.numel() * 4)
    del Kd, Vd, Qd, O, L, att
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return out


MLA_D_C = 512
MLA_HEADS = (16, 16)


def measure_mla(dev, steps: int, warmup: int):
    """Multi-head latent attention on the document-QA tree (16 heads, d=128,
    MHA after the rebuild, latent d_c = 512): per step the per-head K/V of
    every tree page are rebuilt from the latent pool (pst_mla_reconstruct) and
    the decode pipeline runs on them. Reports the step, the rebuild alone
    (CUDA events around it, on the launching stream) and the rebuild's
    tensor-core and HBM rates."""
    import numpy as np
    import torch
    import synth
    from prefix_shared_tree_gb300.torch_api import TreeDecodeAttention, to_device
    wl = synth.document_qa(heads=MLA_HEADS)
    C, Wk, Wv = wl.mla_inputs(MLA_D_C)
    att = TreeDecodeAttention.from_workload(wl, device=dev)
    Cd, Wkd, Wvd = (to_device(x, "bf16", dev) for x in (C, Wk, Wv))
    Qd = to_device(wl.q(), "bf16", dev)
    shape = (wl.num_pages, wl.n_kv_heads, wl.page_size, wl.d)
    Kd = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    Vd = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    O = torch.empty((wl.n_queries, wl.n_q_heads, wl.d), dtype=torch.float32, device=dev)
    L = torch.empty((wl.n_queries, wl.n_q_heads), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        att.mla_reconstruct(Cd, Wkd, Wvd, Kd, Vd)
        att(Qd, Kd, Vd, O, L)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ev[0].record(stream)
    for _ in range(steps):
        step()
    ev[1].record(stream)
    ev[2].record(stream)
    for _ in range(steps):
        att.mla_reconstruct(Cd, Wkd, Wvd, Kd, Vd)
    ev[3].record(stream)
    torch.cuda.synchronize(dev)
    if att.check_status() != 0:
        raise RuntimeError("mla: device status word set")
    step_us = ev[0].elapsed_time(ev[1]) * 1e3 / steps
    rebuild_us = ev[2].elapsed_time(ev[3]) * 1e3 / steps
    n_pages = len(np.unique(wl.page_ids))
    rows = n_pages * wl.page_size
    flops = 2.0 * rows * MLA_D_C * 2 * wl.n_kv_heads * wl.d
    bytes_ = rows * MLA_D_C * 2 + rows * 2 * wl.n_kv_heads * wl.d * 2
    try:
        tf_peak = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"])
    except Exception:
        tf_peak = 1900.0
    hbm, _ = measured_peaks()
    out = {"workload": "document_qa tree, 16 heads (MHA after the rebuild), d=128, latent d_c=512, bf16",
           "us_per_step": round(step_us, 3), "rebuild_us": round(rebuild_us, 3),
           "decode_us": round(step_us - rebuild_us, 3), "pages_rebuilt": int(n_pages),
           "rebuild_tflops": round(flops / (rebuild_us * 1e-6) / 1e12, 1),
           "rebuild_frac_of_bf16_peak": round(flops / (rebuild_us * 1e-6) / 1e12 / tf_peak, 4),
           "rebuild_hbm_gbs": round(bytes_ / (rebuild_us * 1e-6) / 1e9, 1),
           "rebuild_frac_of_hbm": round(bytes_ / (rebuild_us * 1e-6) / 1e9 / hbm, 4),
           "rebuild_flops": flops, "rebuild_bytes": int(bytes_), "steps": steps}
    del Cd, Wkd, Wvd, Kd, Vd, att
    torch.cuda.empty_cache()
    return out


def _config_entry(m):
    peak = m["peak"]
    gbs = m["U"] / (m["us"] * 1e-6) / 1e9
    return {
        "us_per_step": round(m["us"], 3), "graph_replay_us_per_step": round(m["graph_us"], 3),
        "single_step_us": {"call": round(m["single_us"], 3), "graph": round(m["single_graph_us"], 3)},
        "unique_kv_bytes": m["U"], "achieved_unique_kv_gbs": round(gbs, 1),
        "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4), "frac_of_measured_hbm": round(gbs / peak, 4),
        "dominant_kernel": {"kernel": m["dom"], "algorithmic_bytes": m["alg"][m["dom"]],
                            "group_end_us": m["dom_us"], "achieved_gbs": round(m["dom_achieved"], 1),
                            "frac": round(m["dom_achieved"] / peak, 4)},
        "group_end_us": m["group_end_us"], "por_us": m["por_us"], "n_launches": m["n_launches"],
        "plan_us": m["plan"]["plan_us"], "split_policy": m["plan"]["split_policy"], "sm_mhz": m["clocks"].get("sm_mhz"),
    }


def run_ours(args, rank, world):
    import torch

    from prefix_shared_tree_gb300 import build as _build
    _build.build()

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    plan_opts = _plan_opts(args)
    warm = max(3, args.warmup)
    h = measure(args.workload, args, dev, args.steps, warm, args.timer_steps, plan_opts, e2e=True, world=world)
    us, e2e_us = max_over_ranks([h["us"], h["e2e_us"]], world, dev)
    per_config = {}
    if world == 1 and not args.no_per_config:
        steps_pc = max(20, min(args.steps, 200))
        shared_us = {args.workload: h["us"]}
        for name in [n for n in args.per_config.split(",") if n and n != args.workload]:
            m = measure(name, args, dev, steps_pc, 5, min(args.timer_steps, 32), plan_opts)
            per_config[name] = _config_entry(m)
            shared_us[name] = m["us"]
            per_config[name]["steps"] = steps_pc
        if not args.no_mla:
            per_config["document_qa_mla"] = measure_mla(dev, min(steps_pc, 100), 5)
        for name, e in per_config.items():
            base = name[:-len("_flat")] if name.endswith("_flat") else None
            if base and base in shared_us:
                import synth
                U_shared = WORKLOADS[base](synth).unique_kv_bytes()
                e["vs_shared_tree"] = {"shared_us": round(shared_us[base], 3),
                                       "flat_over_shared_time": round(e["us_per_step"] / shared_us[base], 3),
                                       "flat_over_shared_unique_bytes": round(e["unique_kv_bytes"] / U_shared, 3)}
    if rank != 0:
        return None
    peak, peak_src = measured_peaks()
    U = h["U"]
    wl = h["wl"]
    achieved_gbs = U / (us * 1e-6) / 1e9
    traffic = recorded_traffic(h["dom"], args.workload, h["plan"]["digest"])
    line = {
        "metric": METRIC,
        "value": round(us, 3),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": warm,
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
        "graph_replay": {"value": round(h["graph_us"], 3), "unit": "us/step",
                         "note": "the same steps replayed from CUDA graphs of pst_decode_attn (one capture per "
                                 "input copy): no host work per step"},
        "single_step_us": {"call": round(h["single_us"], 3), "graph": round(h["single_graph_us"], 3),
                           "note": "median of 30 steps each launched on an idle GPU (synchronised before and "
                                   "after): the latency of one call, host launch work included"},
        "group_end_us": h["group_end_us"],
        "por_us": h["por_us"],
        "timer_note": f"group_end_us: from the call's start to the end of each PAC launch group (the groups run "
                      f"side by side), and POR alone, over a separate loop of {args.timer_steps} calls with the "
                      f"library's events; that timed entry point forks the groups onto side streams (events "
                      f"between chained launches would serialise them), while the timed loop above, the graph "
                      f"replays and e2e use the default chained launch and record no events",
        "roofline": {"bound": "hbm", "kernel": h["dom"], "achieved": round(h["dom_achieved"], 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(h["dom_achieved"] / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": h["alg"][h["dom"]]},
        "plan": h["plan"],
        "e2e": {"value": round(e2e_us, 3), "unit": "us/step", "h2d_bytes_per_step": h["h2d"],
                "d2h_bytes_per_step": h["d2h"]},
        "gpu_launches": h["n_launches"] * args.steps,
        "clocks": h["clocks"],
    }
    if per_config:
        line["per_config"] = per_config
    return line, wl


def run_reference(args, rank):
    """The oracle as it stands on the host cores. A step is the whole batch
    (every query and head) when W + K such steps fit in --ref-budget-s, else a
    fixed sample of queries per step with the full-batch time extrapolated
    (and said so in the line)."""
    if rank != 0:
        return None
    import numpy as np  # noqa: F401

    import synth
    from oracle import attention as oa

    wl = WORKLOADS[args.workload](synth)
    K, V = wl.kv_pools()
    Q = wl.q()
    nq = wl.n_queries
    order = [(i * 37) % nq for i in range(nq)]
    t0 = time.perf_counter()
    oa.decode_attention(wl, K, V, Q, order[:2])             # probe: two queries
    per_q = (time.perf_counter() - t0) / 2
    runs = max(1, args.steps) + max(1, args.warmup)
    per_step = max(1, min(nq, int(args.ref_budget_s / max(per_q * runs, 1e-9))))
    sampled = per_step < nq
    for w in range(max(1, args.warmup)):                    # untimed warm-up steps
        oa.decode_attention(wl, K, V, Q, [order[(w * per_step + i) % nq] for i in range(per_step)])
    times = []
    for st in range(max(1, args.steps)):
        qs = [order[(st * per_step + i) % nq] for i in range(per_step)]
        t0 = time.perf_counter()
        oa.decode_attention(wl, K, V, Q, qs)
        times.append(time.perf_counter() - t0)
    step_s = sum(times) / len(times)
    us = step_s / per_step * nq * 1e6
    ncpu = 1
    try:
        import threadpoolctl  # noqa: F401
        ncpu = max(i.get("num_threads", 1) for i in threadpoolctl.threadpool_info()) or 1
    except Exception:
        ncpu = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    if sampled:
        sample = (f"each of the {len(times)} timed steps ran {per_step} of the batch's {nq} queries (all heads, "
                  f"fp64); us/step is the full batch extrapolated from them")
    else:
        sample = f"each of the {len(times)} timed steps ran the whole batch ({nq} queries, all heads, fp64)"
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(us, 1),
        "unit": "us/step",
        "n_gpus": 1,
        "steps": len(times),
        "warmup": max(1, args.warmup),
        "ms_per_step": round(us / 1e3, 3),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": bench_config(args, wl, 1),
        "queries_per_step": per_step,
        "extrapolated": sampled,
        "executed_ms_per_step": round(step_s * 1e3, 3),
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
