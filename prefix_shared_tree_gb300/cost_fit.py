"""Measure the planner's cost tables C_est(rows, tokens) on the current GPU.

CoDec, "profile-based cost estimation": the partitioner needs the time of one
PAC thread block as a function of its aggregated query rows and KV tokens.
This script measures it for the four PAC kinds (0: CUDA-core PAC, 1: tcgen05
PAC with P rounded once to bf16, 2: tcgen05 PAC with exact P, 3: tcgen05 thin
PAC) on a grid of (rows, tokens): for each point it builds a forest of
identical independent nodes (one thread block each, no KV split), fills the
GPU with a few waves of them, times the PAC launch with the library's timer
and reports

    C_est = (launch time) x (number of SMs) / (number of blocks),

the time one block holds one of the planner's per-SM slots with every SM
busy (CUDA-core and thin-PAC blocks, several waves). Tensor-core blocks hold
a whole SM; they are timed as one wave on two thirds of the SMs, where C_est
is the launch time. Inputs are random bf16, d = 128, one KV head (blocks are
per KV head), eight for the thin PAC (a thin block covers eight kv heads;
rows are per head).

Writes ``cost_table_gb300.json`` and the C++ include ``cost_table_gb300.inc``
that libpst compiles in as its built-in tables:

    python -m prefix_shared_tree_gb300.cost_fit --out DIR
"""
from __future__ import annotations

import argparse
import json
import os
import time

import numpy as np

GRID = {
    0: ([1, 2, 4, 8], [64, 128, 256, 512, 1024, 2048, 4096, 8192]),
    1: ([16, 32, 64, 128, 256], [128, 256, 512, 1024, 2048, 4096, 8192]),
    2: ([16, 32, 64, 128, 256], [64, 128, 256, 512, 1024, 2048, 4096]),
    3: ([1, 2, 4, 8], [16, 32, 64, 128, 256, 512, 1024, 2048, 4096]),
}
SLOT = {0: "pac_thin", 1: "pac_tc", 2: "pac_tc_exact", 3: "pac_thin"}
PAGE = 16
D = 128


def measure_point(kind: int, rows: int, tokens: int, num_sms: int, seed: int, reps: int = 12,
                  thin_sms: int = 0) -> dict:
    import torch
    from . import pst
    from .torch_api import TreeDecodeAttention

    # CUDA-core blocks: a few waves, more when blocks are short so launch cost
    # amortises. Tensor-core blocks (one per SM): a single wave on about two
    # thirds of the SMs, the share they usually get beside CUDA-core work.
    hkv = 8 if kind == 3 else 1
    if kind == 3 and thin_sms > 0:
        n = thin_sms       # one wave on thin_sms SMs (HBM shared with fewer blocks)
    elif kind in (0, 3):
        n = 4 * num_sms
        n = max(n, min(16 * num_sms, (1 << 21) // max(tokens, 1)))
        n = min(n, max(num_sms, (6 << 20) // (tokens * hkv)))    # <= ~3 GiB per pool
    else:
        n = (2 * num_sms) // 3
    pages_per_node = (tokens + PAGE - 1) // PAGE
    num_pages = n * pages_per_node
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_pages).astype(np.int32)
    node_len = np.full(n, tokens, np.int32)
    parent = np.full(n, -1, np.int32)
    page_ptr = np.arange(n + 1, dtype=np.int64) * pages_per_node
    query_node = np.repeat(np.arange(n, dtype=np.int32), rows)       # G = 1: rows = queries
    opts = dict(split_policy="none", num_sms=num_sms)
    if kind == 0:
        opts["thin_engine"] = "cuda_core"
    elif kind == 3:
        opts["tc_min_rows"] = 1 << 20
    elif kind == 1:
        opts["p_bf16_min_tokens"] = 1
    elif kind == 2:
        opts["p_bf16_min_tokens"] = -1
    att = TreeDecodeAttention(node_len, parent, page_ptr, perm, None, PAGE, num_pages, query_node,
                              hkv, hkv, D, "bf16", **opts)
    st = att.plan.stats()
    blocks = st["n_tc_items"] if kind in (1, 2) else st["n_cc_items"]
    assert blocks == n, (kind, rows, tokens, blocks, n)
    g = torch.Generator(device="cuda").manual_seed(seed)
    K = torch.randn((num_pages, hkv, PAGE, D), generator=g, device="cuda").to(torch.bfloat16)
    V = torch.randn((num_pages, hkv, PAGE, D), generator=g, device="cuda").to(torch.bfloat16)
    Q = torch.randn((len(query_node), hkv, D), generator=g, device="cuda").to(torch.bfloat16)
    O = torch.empty((len(query_node), hkv, D), dtype=torch.float32, device="cuda")
    L = torch.empty((len(query_node), hkv), dtype=torch.float32, device="cuda")
    for _ in range(3):
        att(Q, K, V, O, L)
    timer = pst.Timer(reps)
    for _ in range(reps):
        att(Q, K, V, O, L, timer=timer)
    ms, calls = timer.read()
    if att.check_status() != 0:
        raise RuntimeError("device status word set")
    t_us = ms[SLOT[kind]] * 1e3 / calls
    del K, V, Q, O, L, att
    torch.cuda.empty_cache()
    # per slot: a wave of n blocks on n SMs holds each for the launch time
    per_slot = t_us * num_sms / n if (kind == 0 or (kind == 3 and thin_sms <= 0)) else t_us
    return {"kind": kind, "rows": rows, "tokens": tokens, "blocks": n, "launch_us": t_us, "us": per_slot}


def write_inc(tables: dict, path: str, note: str):
    lines = ["// Cost tables C_est(rows, tokens) in microseconds per PAC thread block with",
             "// every SM busy (one per PAC kind), measured by cost_fit.py.",
             f"// {note}",
             "struct BuiltinCostTable {", "    int n_r, n_n;", "    const double* rows;",
             "    const double* tokens;", "    const double* us;", "};"]
    entries = []
    for k in range(4):
        t = tables.get(k)
        if not t:
            entries.append("{0, 0, nullptr, nullptr, nullptr}")
            continue
        r, n, us = t["rows"], t["tokens"], t["us"]
        lines.append(f"static const double kCostRows{k}[] = {{{', '.join(f'{x:g}' for x in r)}}};")
        lines.append(f"static const double kCostTokens{k}[] = {{{', '.join(f'{x:g}' for x in n)}}};")
        flat = [u for row in us for u in row]
        lines.append(f"static const double kCostUs{k}[] = {{{', '.join(f'{x:.4g}' for x in flat)}}};")
        entries.append(f"{{{len(r)}, {len(n)}, kCostRows{k}, kCostTokens{k}, kCostUs{k}}}")
    lines.append("static const BuiltinCostTable kBuiltinCost[kCostKinds] = {" + ", ".join(entries) + "};")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=os.path.dirname(os.path.abspath(__file__)))
    ap.add_argument("--kinds", default="0,1,2,3")
    ap.add_argument("--thin-sms", type=int, default=0,
                    help="time thin-PAC points as one wave on this many SMs (0: waves on all SMs)")
    args = ap.parse_args()
    import torch
    props = torch.cuda.get_device_properties(0)
    num_sms = props.multi_processor_count
    # kinds not measured now keep the tables of the previous run in --out
    tables, points = {}, []
    prev = os.path.join(args.out, "cost_table_gb300.json")
    if os.path.exists(prev):
        with open(prev) as f:
            old = json.load(f)
        tables = {int(k): v for k, v in old.get("tables", {}).items()}
        points = old.get("points", [])
    t0 = time.time()
    new_points = []
    for kind in [int(k) for k in args.kinds.split(",")]:
        rows_g, tok_g = GRID[kind]
        us = [[0.0] * len(tok_g) for _ in rows_g]
        for i, r in enumerate(rows_g):
            for j, t in enumerate(tok_g):
                p = measure_point(kind, r, t, num_sms, seed=1000 * kind + 10 * i + j, thin_sms=args.thin_sms)
                us[i][j] = p["us"]
                new_points.append(p)
                print(json.dumps(p), flush=True)
        points = [p for p in points if p["kind"] != kind] + [p for p in new_points if p["kind"] == kind]
        tables[kind] = {"rows": rows_g, "tokens": tok_g, "us": us}
    note = f"{props.name}, {num_sms} SMs, measured in {time.time() - t0:.0f} s"
    with open(os.path.join(args.out, "cost_table_gb300.json"), "w") as f:
        json.dump({"device": props.name, "num_sms": num_sms, "tables": {str(k): v for k, v in sorted(tables.items())},
                   "points": points}, f, indent=1)
    write_inc(tables, os.path.join(args.out, "cost_table_gb300.inc"), note)
    print("wrote", args.out)


if __name__ == "__main__":
    main()
