"""ctypes binding of libpst (include/pst.h): argument marshalling only.

Every function mirrors a C entry point of the same name without the ``pst_``
prefix. Host arrays are numpy arrays (copied by the library during the call);
device buffers and streams are raw integers (pointers / cudaStream_t). The
library must be built (``prefix_shared_tree_gb300.build.build()``); importing
this module fails loudly if it is not.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import numpy as np

from . import build as _build

PST_OK = 0
ERRORS = {-1: "PST_EINVAL", -2: "PST_ECYCLE", -3: "PST_ERANGE", -4: "PST_EUNSUPPORTED",
          -5: "PST_EWORKSPACE", -6: "PST_ECUDA", -7: "PST_EDEVICE", -8: "PST_ENOMEM"}
DTYPES = {"bf16": 0, "f32": 1}
SPLIT = {"cost_model": 0, "none": 1, "uniform": 2, "flatten": 3}
KERNEL_SLOTS = 4


class PstError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class PlanOpts(C.Structure):
    _fields_ = [("split_policy", C.c_int32), ("fixed_chunk", C.c_int32), ("tc_min_rows", C.c_int32),
                ("pack_masks", C.c_int32), ("num_sms", C.c_int32), ("slots_per_sm", C.c_int32),
                ("tc_engine", C.c_int32), ("tc_block_rows", C.c_int32), ("p_bf16_min_tokens", C.c_int32),
                ("thin_engine", C.c_int32), ("debug_stall", C.c_int32), ("side_streams", C.c_int32),
                ("flatten_candidates", C.c_int32)]


class PlanStats(C.Structure):
    _fields_ = [("plan_us", C.c_double), ("predicted_makespan_us", C.c_double),
                ("cost_lower_bound_us", C.c_double), ("n_chunks", C.c_int64), ("n_items", C.c_int64),
                ("n_tc_items", C.c_int64), ("n_cc_items", C.c_int64), ("n_partial_rows", C.c_int64),
                ("unique_kv_tokens", C.c_int64), ("kv_tokens_read", C.c_int64),
                ("workspace_bytes", C.c_int64), ("num_slots", C.c_int32), ("n_launches", C.c_int32),
                ("split_policy", C.c_int32), ("fixed_chunk", C.c_int32)]


class ExportSizes(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("n_queries", "n_nodes", "n_chunks", "n_qpath", "n_nodeq",
                                          "n_chunk_q", "n_chunk_tok", "n_merge")]


_EXPORT_FIELDS = [("qpath_ptr", "i4", "n_queries", 1), ("qpath_node", "i4", "n_qpath", 0),
                  ("nodeq_ptr", "i4", "n_nodes", 1), ("nodeq", "i4", "n_nodeq", 0),
                  ("chunk_q_ptr", "i4", "n_chunks", 1), ("chunk_q", "i4", "n_chunk_q", 0),
                  ("chunk_q_mask", "u8", "n_chunk_q", 0), ("chunk_tok_ptr", "i4", "n_chunks", 1),
                  ("chunk_tok_node", "i4", "n_chunk_tok", 0), ("chunk_tok_t", "i4", "n_chunk_tok", 0),
                  ("chunk_kind", "i4", "n_chunks", 0), ("merge_ptr", "i4", "n_queries", 1),
                  ("merge_row", "i4", "n_merge", 0)]


class Export(C.Structure):
    _fields_ = [(n, C.POINTER(C.c_uint64) if t == "u8" else C.POINTER(C.c_int32))
                for n, t, _, _ in _EXPORT_FIELDS]


_lib = None


def lib() -> C.CDLL:
    """The loaded libpst (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libpst is not built ({path} missing): run prefix_shared_tree_gb300.build.build()")
    L = C.CDLL(path)
    vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
    sig = {
        "pst_tree_build": (C.c_int, [i32, vp, vp, vp, vp, vp, i32, i64, C.POINTER(vp)]),
        "pst_tree_destroy": (None, [vp]),
        "pst_plan_opts_default": (None, [C.POINTER(PlanOpts)]),
        "pst_plan_create": (C.c_int, [vp, i32, vp, i32, i32, i32, C.c_int, C.POINTER(PlanOpts), C.POINTER(vp)]),
        "pst_plan_update": (C.c_int, [vp, vp, C.POINTER(vp)]),
        "pst_plan_update_tree": (C.c_int, [vp, vp, i32, vp, vp, C.POINTER(vp)]),
        "pst_plan_destroy": (None, [vp]),
        "pst_plan_workspace_bytes": (i64, [vp]),
        "pst_plan_upload": (C.c_int, [vp, vp, i64, vp]),
        "pst_decode_attn": (C.c_int, [vp, vp, vp, vp, vp, vp, vp]),
        "pst_decode_attn_noalloc": (C.c_int, [vp, vp, vp, vp, vp, vp, vp]),
        "pst_noalloc_check_status": (C.c_int, [vp, C.POINTER(i32)]),
        "pst_mla_reconstruct": (C.c_int, [vp, vp, i32, vp, vp, vp, vp, vp]),
        "pst_plan_check_status": (C.c_int, [vp, vp, C.POINTER(i32)]),
        "pst_timer_create": (C.c_int, [i32, C.POINTER(vp)]),
        "pst_timer_destroy": (None, [vp]),
        "pst_decode_attn_timed": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, vp]),
        "pst_timer_read": (C.c_int, [vp, C.POINTER(C.c_float), i32, C.POINTER(i32)]),
        "pst_timer_kernel_name": (C.c_char_p, [i32]),
        "pst_plan_stats_get": (C.c_int, [vp, C.POINTER(PlanStats)]),
        "pst_plan_export_sizes": (C.c_int, [vp, C.POINTER(ExportSizes)]),
        "pst_plan_export": (C.c_int, [vp, C.POINTER(Export)]),
        "pst_cost_set_table": (C.c_int, [i32, i32, vp, i32, vp, vp]),
        "pst_cost_estimate": (C.c_double, [i32, C.c_double, C.c_double]),
        "pst_list_schedule": (C.c_int, [i32, vp, i32, vp, C.POINTER(C.c_double)]),
        "pst_last_error": (C.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def header_functions() -> list[str]:
    """Names of every function declared in include/pst.h."""
    src = open(os.path.join(_build.INCLUDE, "pst.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pst_[a-z0-9_]+)\s*\(", src)))


def _check(rc: int):
    if rc != PST_OK:
        raise PstError(rc, lib().pst_last_error().decode())


def _arr(x, dt):
    if x is None:
        return None, None
    a = np.ascontiguousarray(np.asarray(x), dtype=dt)
    return a, a.ctypes.data_as(C.c_void_p)


class Tree:
    def __init__(self, handle, n_nodes):
        self._h = handle
        self.n_nodes = n_nodes

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.pst_tree_destroy(self._h)
            self._h = None


def tree_build(node_len, parent, page_ptr, page_ids, first_offset=None, page_size=16,
               num_pages=None) -> Tree:
    nl, nlp = _arr(node_len, np.int32)
    pa, pap = _arr(parent, np.int32)
    pp, ppp = _arr(page_ptr, np.int64)
    pi, pip = _arr(page_ids, np.int32)
    fo, fop = _arr(first_offset, np.int32)
    if num_pages is None:
        num_pages = int(pi.max()) + 1 if pi.size else 0
    h = C.c_void_p()
    _check(lib().pst_tree_build(len(nl), nlp, pap, ppp, pip, fop, page_size, int(num_pages), C.byref(h)))
    return Tree(h, len(nl))


def plan_opts_default() -> PlanOpts:
    o = PlanOpts()
    lib().pst_plan_opts_default(C.byref(o))
    return o


class Plan:
    def __init__(self, handle, n_queries, hq, hkv, d, dtype):
        self._h = handle
        self.n_queries, self.hq, self.hkv, self.d, self.dtype = n_queries, hq, hkv, d, dtype
        self._ws = None  # keeps a caller-provided workspace object alive

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.pst_plan_destroy(self._h)
            self._h = None

    @property
    def workspace_bytes(self) -> int:
        return int(lib().pst_plan_workspace_bytes(self._h))

    def upload(self, d_workspace: int, nbytes: int, stream: int = 0, keepalive=None):
        _check(lib().pst_plan_upload(self._h, C.c_void_p(d_workspace), int(nbytes), C.c_void_p(stream)))
        self._ws = keepalive

    def stats(self) -> dict:
        s = PlanStats()
        _check(lib().pst_plan_stats_get(self._h, C.byref(s)))
        return {n: getattr(s, n) for n, _ in PlanStats._fields_}

    def export(self) -> dict:
        sz = ExportSizes()
        _check(lib().pst_plan_export_sizes(self._h, C.byref(sz)))
        out, e = {}, Export()
        for name, t, szname, extra in _EXPORT_FIELDS:
            n = getattr(sz, szname) + extra
            a = np.zeros(max(n, 1), dtype=np.uint64 if t == "u8" else np.int32)
            out[name] = a
            setattr(e, name, a.ctypes.data_as(C.POINTER(C.c_uint64 if t == "u8" else C.c_int32)))
        _check(lib().pst_plan_export(self._h, C.byref(e)))
        for name, t, szname, extra in _EXPORT_FIELDS:
            out[name] = out[name][:getattr(sz, szname) + extra]
        return out

    def check_status(self, stream: int = 0) -> int:
        code = C.c_int32(0)
        rc = lib().pst_plan_check_status(self._h, C.c_void_p(stream), C.byref(code))
        if rc not in (PST_OK, -7):
            _check(rc)
        return int(code.value)


def plan_create(tree: Tree, query_node, n_q_heads: int, n_kv_heads: int, d: int, dtype: str = "bf16",
                split_policy: str = "cost_model", fixed_chunk: int | None = None,
                tc_min_rows: int | None = None, pack_masks: bool | None = None, num_sms: int = 0,
                slots_per_sm: int = 0, tc_engine: str = "tcgen05", tc_block_rows: int = 256,
                p_bf16_min_tokens: int = 0, thin_engine: str = "tcgen05", debug_stall: bool = False,
                side_streams: bool = False, flatten_candidates: bool = True) -> Plan:
    o = plan_opts_default()
    o.split_policy = SPLIT[split_policy]
    if fixed_chunk is not None:
        o.fixed_chunk = fixed_chunk
    if tc_min_rows is not None:
        o.tc_min_rows = tc_min_rows
    if pack_masks is not None:
        o.pack_masks = int(bool(pack_masks))
    o.num_sms = num_sms
    o.slots_per_sm = slots_per_sm
    o.tc_engine = {"tcgen05": 0, "mma_sync": 1}[tc_engine]
    o.tc_block_rows = tc_block_rows
    o.p_bf16_min_tokens = p_bf16_min_tokens
    o.thin_engine = {"tcgen05": 0, "cuda_core": 1}[thin_engine]
    o.debug_stall = int(bool(debug_stall))
    o.side_streams = int(bool(side_streams))
    o.flatten_candidates = 0 if flatten_candidates else -1
    qn, qnp = _arr(query_node, np.int32)
    h = C.c_void_p()
    _check(lib().pst_plan_create(tree._h, len(qn), qnp, n_q_heads, n_kv_heads, d, DTYPES[dtype],
                                 C.byref(o), C.byref(h)))
    return Plan(h, len(qn), n_q_heads, n_kv_heads, d, dtype)


def plan_update(prev: Plan, tree: Tree) -> Plan:
    """Plan for the same queries on a tree whose node lengths (and pages)
    changed, keeping prev's KV-axis splits (no partition search)."""
    h = C.c_void_p()
    _check(lib().pst_plan_update(prev._h, tree._h, C.byref(h)))
    return Plan(h, prev.n_queries, prev.hq, prev.hkv, prev.d, prev.dtype)


def plan_update_tree(prev: Plan, tree: Tree, query_node, prev_node) -> Plan:
    """Plan for a tree whose shape changed (nodes kept, pruned or added; new
    queries): prev_node[n] is node n's id in prev's tree, or -1 if new. Kept
    nodes keep prev's KV-axis splits (no partition search)."""
    qn, qnp = _arr(query_node, np.int32)
    pn, pnp = _arr(prev_node, np.int32)
    if pn.size != tree.n_nodes:
        raise ValueError("prev_node needs one entry per node of the new tree")
    h = C.c_void_p()
    _check(lib().pst_plan_update_tree(prev._h, tree._h, len(qn), qnp, pnp, C.byref(h)))
    return Plan(h, len(qn), prev.hq, prev.hkv, prev.d, prev.dtype)


def decode_attn(plan: Plan, q: int, k_pool: int, v_pool: int, o: int, lse: int, stream: int = 0):
    _check(lib().pst_decode_attn(plan._h, C.c_void_p(q), C.c_void_p(k_pool), C.c_void_p(v_pool),
                                 C.c_void_p(o), C.c_void_p(lse), C.c_void_p(stream)))


NOALLOC_WORKSPACE_BYTES = 32 << 20


def decode_attn_noalloc(plan: Plan, q: int, k_pool: int, v_pool: int, o: int, lse: int, stream: int = 0):
    """pst_decode_attn without any workspace: for callers that cannot allocate
    device memory where they run attention (the scratch is a fixed array of
    NOALLOC_WORKSPACE_BYTES inside the library; overlapping calls race)."""
    _check(lib().pst_decode_attn_noalloc(plan._h, C.c_void_p(q), C.c_void_p(k_pool), C.c_void_p(v_pool),
                                         C.c_void_p(o), C.c_void_p(lse), C.c_void_p(stream)))


class Timer:
    def __init__(self, max_calls: int):
        h = C.c_void_p()
        _check(lib().pst_timer_create(max_calls, C.byref(h)))
        self._h = h

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.pst_timer_destroy(self._h)
            self._h = None

    def read(self):
        """(per-kernel summed ms as a dict, number of calls); resets the timer."""
        ms = (C.c_float * KERNEL_SLOTS)()
        calls = C.c_int32(0)
        _check(lib().pst_timer_read(self._h, ms, KERNEL_SLOTS, C.byref(calls)))
        names = [lib().pst_timer_kernel_name(i).decode() for i in range(KERNEL_SLOTS)]
        return dict(zip(names, list(ms))), int(calls.value)


def decode_attn_timed(plan: Plan, q: int, k_pool: int, v_pool: int, o: int, lse: int, stream: int,
                      timer: Timer):
    _check(lib().pst_decode_attn_timed(plan._h, C.c_void_p(q), C.c_void_p(k_pool), C.c_void_p(v_pool),
                                       C.c_void_p(o), C.c_void_p(lse), C.c_void_p(stream), timer._h))


def cost_set_table(kind: int, rows, tokens, us):
    """Install a measured table for PAC kind 0 (CUDA core), 1 (tcgen05, P
    rounded once), 2 (tcgen05, exact P) or 3 (tcgen05 thin PAC); rows=None
    selects the analytic model, rows="builtin" restores the built-in table."""
    if isinstance(rows, str) and rows == "builtin":
        _check(lib().pst_cost_set_table(kind, -1, None, 0, None, None))
        return
    if rows is None:
        _check(lib().pst_cost_set_table(kind, 0, None, 0, None, None))
        return
    r, rp = _arr(rows, np.float32)
    t, tp = _arr(tokens, np.float32)
    u, up = _arr(us, np.float32)
    assert u.size == r.size * t.size
    _check(lib().pst_cost_set_table(kind, r.size, rp, t.size, tp, up))


def cost_estimate(kind: int, rows: float, tokens: float) -> float:
    return float(lib().pst_cost_estimate(kind, rows, tokens))


def list_schedule(costs, m: int):
    """The planner's largest-first list schedule of `costs` onto m slots:
    (slot of each task, makespan)."""
    c, cp = _arr(costs, np.float64)
    n = 0 if c is None else c.size
    slot = np.zeros(max(n, 1), dtype=np.int32)
    mk = C.c_double(0.0)
    _check(lib().pst_list_schedule(n, cp, int(m), slot.ctypes.data_as(C.c_void_p), C.byref(mk)))
    return slot[:n], float(mk.value)


def mla_reconstruct(plan: Plan, c_pool: int, d_c: int, w_uk: int, w_uv: int, k_pool: int, v_pool: int,
                    stream: int = 0):
    """Rebuild the per-head K/V pools of the plan's tree pages from a latent
    pool (multi-head latent attention); device pointers."""
    _check(lib().pst_mla_reconstruct(plan._h, C.c_void_p(c_pool), int(d_c), C.c_void_p(w_uk), C.c_void_p(w_uv),
                                     C.c_void_p(k_pool), C.c_void_p(v_pool), C.c_void_p(stream)))


def noalloc_check_status(stream: int = 0) -> int:
    """Raw device status word of pst_decode_attn_noalloc's built-in scratch
    (read and cleared; 0 = clean)."""
    code = C.c_int32(0)
    rc = lib().pst_noalloc_check_status(C.c_void_p(stream), C.byref(code))
    if rc not in (PST_OK, -7):
        _check(rc)
    return int(code.value)
