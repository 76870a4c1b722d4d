"""torch glue for libpst: device memory and streams from torch, nothing else.

``TreeDecodeAttention`` builds the tree and the plan once, allocates the plan's
device workspace as a torch uint8 tensor, uploads the plan, and then runs
``pst_decode_attn`` on torch tensors on the current (or given) stream.
"""
from __future__ import annotations

import numpy as np
import torch

from . import pst

_TORCH_DTYPE = {"bf16": torch.bfloat16, "f32": torch.float32}


def to_device(x: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """Host array (uint16 bf16 bit patterns or float32) -> device tensor."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(device)


class TreeDecodeAttention:
    def __init__(self, node_len, parent, page_ptr, page_ids, first_offset, page_size, num_pages,
                 query_node, n_q_heads, n_kv_heads, d, dtype="bf16", device="cuda", **plan_opts):
        self.device = torch.device(device)
        if self.device.index is None:
            self.device = torch.device(self.device.type, torch.cuda.current_device())
        self.dtype = dtype
        self.n_q_heads, self.n_kv_heads, self.d = n_q_heads, n_kv_heads, d
        self.n_queries = len(query_node)
        self.num_pages, self.page_size = int(num_pages), int(page_size)
        self.tree = pst.tree_build(node_len, parent, page_ptr, page_ids, first_offset, page_size, num_pages)
        with torch.cuda.device(self.device):
            if "num_sms" not in plan_opts:
                plan_opts["num_sms"] = torch.cuda.get_device_properties(self.device).multi_processor_count
            self.plan = pst.plan_create(self.tree, query_node, n_q_heads, n_kv_heads, d, dtype, **plan_opts)
            self.workspace = torch.empty(max(256, self.plan.workspace_bytes), dtype=torch.uint8, device=self.device)
            stream = torch.cuda.current_stream(self.device)
            self.plan.upload(self.workspace.data_ptr(), self.workspace.numel(), stream.cuda_stream,
                             keepalive=self.workspace)

    def update_tree(self, node_len, parent, page_ptr, page_ids, first_offset, num_pages=None):
        """Next decode step on the same tree shape (leaves grown, pages added):
        rebuild the tree and derive the plan from the current one with
        pst_plan_update (no partition search), then upload it."""
        if num_pages is not None:
            self.num_pages = int(num_pages)
        tree = pst.tree_build(node_len, parent, page_ptr, page_ids, first_offset, self.page_size, self.num_pages)
        with torch.cuda.device(self.device):
            plan = pst.plan_update(self.plan, tree)
            if plan.workspace_bytes > self.workspace.numel():
                self.workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=self.device)
            stream = torch.cuda.current_stream(self.device)
            plan.upload(self.workspace.data_ptr(), self.workspace.numel(), stream.cuda_stream,
                        keepalive=self.workspace)
        self.tree, self.plan = tree, plan

    def update_shape(self, node_len, parent, page_ptr, page_ids, first_offset, num_pages, query_node, prev_node):
        """Next decode step on a tree whose shape changed (e.g. speculative
        drafts accepted and pruned, a new draft tree with new queries): rebuild
        the tree and derive the plan with pst_plan_update_tree, where
        prev_node[n] is node n's id in the current tree or -1, then upload."""
        self.num_pages = int(num_pages)
        tree = pst.tree_build(node_len, parent, page_ptr, page_ids, first_offset, self.page_size, self.num_pages)
        with torch.cuda.device(self.device):
            plan = pst.plan_update_tree(self.plan, tree, query_node, prev_node)
            if plan.workspace_bytes > self.workspace.numel():
                self.workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=self.device)
            stream = torch.cuda.current_stream(self.device)
            plan.upload(self.workspace.data_ptr(), self.workspace.numel(), stream.cuda_stream,
                        keepalive=self.workspace)
        self.tree, self.plan = tree, plan
        self.n_queries = len(query_node)

    @classmethod
    def from_workload(cls, wl, device="cuda", **plan_opts):
        return cls(wl.node_len, wl.parent, wl.page_ptr, wl.page_ids, wl.first_offset, wl.page_size,
                   wl.num_pages, wl.query_node, wl.n_q_heads, wl.n_kv_heads, wl.d, wl.dtype, device,
                   **plan_opts)

    def capture(self, Q, K_pool, V_pool, O, LSE):
        """One decode step captured as a CUDA graph (torch.cuda.CUDAGraph) on
        these tensors: replaying it reruns every launch of pst_decode_attn
        (the chained PAC launch groups and POR, or with side_streams the
        groups on their forked streams and the join) with
        no host work per step. The plan, its workspace and the tensors must
        stay alive and in place while the graph is used; a new plan needs a
        new capture. One ordinary call first sets up the kernels and the
        plan's streams outside the capture."""
        side = torch.cuda.Stream(self.device)
        side.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(side):
            self(Q, K_pool, V_pool, O, LSE)
        torch.cuda.current_stream(self.device).wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self(Q, K_pool, V_pool, O, LSE)
        return g

    def _check(self, Q, K, V):
        td = _TORCH_DTYPE[self.dtype]
        for name, t in (("Q", Q), ("K_pool", K), ("V_pool", V)):
            if t.dtype != td or t.device != self.device or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous {td} tensor on {self.device}")
        if tuple(Q.shape) != (self.n_queries, self.n_q_heads, self.d):
            raise ValueError(f"Q shape {tuple(Q.shape)}")
        want = (self.num_pages, self.n_kv_heads, self.page_size, self.d)
        if tuple(K.shape) != want or tuple(V.shape) != want:
            raise ValueError(f"pool shape must be {want}")

    def __call__(self, Q, K_pool, V_pool, O=None, LSE=None, stream=None, timer=None):
        self._check(Q, K_pool, V_pool)
        if O is None:
            O = torch.empty((self.n_queries, self.n_q_heads, self.d), dtype=torch.float32, device=self.device)
        if LSE is None:
            LSE = torch.empty((self.n_queries, self.n_q_heads), dtype=torch.float32, device=self.device)
        st = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        if timer is None:
            pst.decode_attn(self.plan, Q.data_ptr(), K_pool.data_ptr(), V_pool.data_ptr(), O.data_ptr(),
                            LSE.data_ptr(), st)
        else:
            pst.decode_attn_timed(self.plan, Q.data_ptr(), K_pool.data_ptr(), V_pool.data_ptr(),
                                  O.data_ptr(), LSE.data_ptr(), st, timer)
        return O, LSE

    def mla_reconstruct(self, C_pool, W_uk, W_uv, K_pool=None, V_pool=None, stream=None):
        """Multi-head latent attention: rebuild the per-head K/V pools of the
        tree's pages from the latent pool C_pool [num_pages][page_size][d_c]
        with up-projections W_uk, W_uv [Hkv][d][d_c] (bf16), into K_pool /
        V_pool (allocated when not given); then call this object on them."""
        td = torch.bfloat16
        for name, t in (("C_pool", C_pool), ("W_uk", W_uk), ("W_uv", W_uv)):
            if t.dtype != td or t.device != self.device or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous bf16 tensor on {self.device}")
        d_c = C_pool.shape[-1]
        if tuple(C_pool.shape) != (self.num_pages, self.page_size, d_c):
            raise ValueError(f"C_pool shape {tuple(C_pool.shape)}")
        want_w = (self.n_kv_heads, self.d, d_c)
        if tuple(W_uk.shape) != want_w or tuple(W_uv.shape) != want_w:
            raise ValueError(f"W_uk / W_uv shape must be {want_w}")
        shape = (self.num_pages, self.n_kv_heads, self.page_size, self.d)
        if K_pool is None:
            K_pool = torch.empty(shape, dtype=td, device=self.device)
        if V_pool is None:
            V_pool = torch.empty(shape, dtype=td, device=self.device)
        st = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        pst.mla_reconstruct(self.plan, C_pool.data_ptr(), d_c, W_uk.data_ptr(), W_uv.data_ptr(), K_pool.data_ptr(),
                            V_pool.data_ptr(), st)
        return K_pool, V_pool

    def check_status(self, stream=None) -> int:
        st = (stream or torch.cuda.current_stream(self.device)).cuda_stream
        return self.plan.check_status(st)
