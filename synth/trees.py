"""Seeded synthetic prefix-shared KV trees and their tensors.

The shapes follow the workloads the CoDec and DEFT write-ups evaluate:
document QA with one long shared prefix, few-shot prompt trees, speculative
draft-token trees and irregular tree-of-thought trees (the public datasets
they use are not available here; these generators stand in for them).

A workload is a forest of KV nodes (``parent == -1`` hangs a node under the
virtual root), a paged KV pool in the layout ``[num_pages][Hkv][page][d]``,
per-node page lists (CSR) with a first-token offset into the first page, and
the node each decode query sits on. Every token carries a *logical id*; the
value of K/V at (logical id, kv head, channel) is a fixed function of the seed,
so the same token has the same K/V whether it lives in a shared tree or in the
copied pages of the no-sharing flat control.

Input generation only; no attention arithmetic lives here.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import rng

PAGE = 16
JUNK_SCALE = 8.0   # unused page rows hold large finite values: a masking bug shows


@dataclasses.dataclass
class Workload:
    name: str
    n_q_heads: int
    n_kv_heads: int
    d: int
    dtype: str                      # "bf16" or "f32"
    page_size: int
    node_len: np.ndarray            # int32 [N]
    parent: np.ndarray              # int32 [N], -1 = child of the virtual root
    first_offset: np.ndarray        # int32 [N]
    page_ptr: np.ndarray            # int64 [N+1]
    page_ids: np.ndarray            # int32 [page_ptr[-1]]
    num_pages: int
    query_node: np.ndarray          # int32 [B]
    lid_ptr: np.ndarray             # int64 [N+1] token logical-id CSR
    lid: np.ndarray                 # int64 [sum(node_len)]
    seed: int
    meta: dict = dataclasses.field(default_factory=dict)

    # ----------------------------------------------------------------- sizes
    @property
    def n_nodes(self) -> int:
        return int(self.node_len.shape[0])

    @property
    def n_queries(self) -> int:
        return int(self.query_node.shape[0])

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def unique_kv_bytes(self) -> int:
        return int(self.node_len.sum()) * self.n_kv_heads * 2 * self.d * self.elem_bytes

    # ----------------------------------------------------------------- keys
    def _key(self, tag: int) -> int:
        return rng.stream_key(self.seed, tag, self.n_kv_heads, self.d)

    @property
    def key_k(self): return self._key(11)

    @property
    def key_v(self): return self._key(12)

    @property
    def key_q(self): return rng.stream_key(self.seed, 13, self.n_q_heads, self.d)

    @property
    def key_junk(self): return self._key(14)

    # ------------------------------------------------------------ rounding
    def _to_storage(self, x: np.ndarray) -> np.ndarray:
        if self.dtype == "bf16":
            return rng.round_to_bf16_bits(x)
        return x.astype(np.float32)

    # --------------------------------------------------------------- tensors
    def row_lids(self) -> np.ndarray:
        """int64 [num_pages * page_size]: logical id stored in each pool row, -1 if unused."""
        out = np.full(self.num_pages * self.page_size, -1, dtype=np.int64)
        for n in range(self.n_nodes):
            L = int(self.node_len[n])
            if L == 0:
                continue
            pages = self.page_ids[self.page_ptr[n]:self.page_ptr[n + 1]].astype(np.int64)
            pos = self.first_offset[n] + np.arange(L, dtype=np.int64)
            rows = pages[pos // self.page_size] * self.page_size + pos % self.page_size
            out[rows] = self.lid[self.lid_ptr[n]:self.lid_ptr[n + 1]]
        return out

    def kv_pools(self, workers: int | None = None):
        """(K_pool, V_pool): uint16 bf16 bits or float32, shape [P, Hkv, page, d]."""
        P, H, S, D = self.num_pages, self.n_kv_heads, self.page_size, self.d
        st = np.uint16 if self.dtype == "bf16" else np.float32
        K = np.empty((P, H, S, D), dtype=st)
        V = np.empty((P, H, S, D), dtype=st)
        lids = self.row_lids().reshape(P, S)
        hh = np.arange(H, dtype=np.uint64)[None, :, None, None]
        ee = np.arange(D, dtype=np.uint64)[None, None, None, :]
        kk, kv, kj = self.key_k, self.key_v, self.key_junk

        def fill(p0, p1):
            lid = lids[p0:p1]
            used = (lid >= 0)[:, None, :, None]
            l64 = np.where(lid >= 0, lid, 0).astype(np.uint64)[:, None, :, None]
            cnt = (l64 * np.uint64(H) + hh) * np.uint64(D) + ee
            pr = np.arange(p0, p1, dtype=np.uint64)[:, None, None, None]
            rr = np.arange(S, dtype=np.uint64)[None, None, :, None]
            jc = ((pr * np.uint64(H) + hh) * np.uint64(S) + rr) * np.uint64(D) + ee
            for key, out, jtag in ((kk, K, 0), (kv, V, 1)):
                val = rng.normal_at(key, cnt)
                junk = JUNK_SCALE * rng.normal_at(kj, jc * np.uint64(2) + np.uint64(jtag))
                out[p0:p1] = self._to_storage(np.where(used, val, junk))

        rng.parallel_fill(P, fill, workers=workers, min_chunk=16)
        return K, V

    def mla_inputs(self, d_c: int = 512, workers: int | None = None):
        """Latent KV inputs (multi-head latent attention), bf16 bits:
        C_pool [P, page, d_c] with N(0, 1) latents per logical token (junk in
        rows no node covers), and up-projections W_uk, W_uv [Hkv, d, d_c]
        drawn N(0, 1/d_c), so the rebuilt K and V are about N(0, 1)."""
        P, S, H, D = self.num_pages, self.page_size, self.n_kv_heads, self.d
        C = np.empty((P, S, d_c), dtype=np.uint16)
        lids = self.row_lids().reshape(P, S)
        kc = rng.stream_key(self.seed, 15, d_c)
        kj = rng.stream_key(self.seed, 16, d_c)
        cc = np.arange(d_c, dtype=np.uint64)[None, None, :]

        def fill(p0, p1):
            lid = lids[p0:p1]
            used = (lid >= 0)[:, :, None]
            l64 = np.where(lid >= 0, lid, 0).astype(np.uint64)[:, :, None]
            pr = np.arange(p0, p1, dtype=np.uint64)[:, None, None]
            rr = np.arange(S, dtype=np.uint64)[None, :, None]
            val = rng.normal_at(kc, l64 * np.uint64(d_c) + cc)
            junk = JUNK_SCALE * rng.normal_at(kj, (pr * np.uint64(S) + rr) * np.uint64(d_c) + cc)
            C[p0:p1] = rng.round_to_bf16_bits(np.where(used, val, junk))

        rng.parallel_fill(P, fill, workers=workers, min_chunk=16)
        scale = 1.0 / np.sqrt(d_c)
        W = [rng.round_to_bf16_bits(scale * rng.normal(rng.stream_key(self.seed, tag, H, D, d_c), 0, H * D * d_c))
             .reshape(H, D, d_c) for tag in (17, 18)]
        return C, W[0], W[1]

    def q(self) -> np.ndarray:
        B, H, D = self.n_queries, self.n_q_heads, self.d
        x = rng.normal(self.key_q, 0, B * H * D).reshape(B, H, D)
        return self._to_storage(x)

    def node_kv_logical(self, n: int):
        """Exact K_n, V_n of node n as float64 [len, Hkv, d], built from logical ids
        directly (no page tables involved)."""
        H, D = self.n_kv_heads, self.d
        lid = self.lid[self.lid_ptr[n]:self.lid_ptr[n + 1]].astype(np.uint64)
        cnt = (lid[:, None, None] * np.uint64(H) + np.arange(H, dtype=np.uint64)[None, :, None]) \
            * np.uint64(D) + np.arange(D, dtype=np.uint64)[None, None, :]
        out = []
        for key in (self.key_k, self.key_v):
            s = self._to_storage(rng.normal_at(key, cnt))
            if self.dtype == "bf16":
                f = (s.astype(np.uint32) << np.uint32(16)).view(np.float32)
            else:
                f = s
            out.append(f.astype(np.float64))
        return out[0], out[1]


# ---------------------------------------------------------------------------
# construction helpers
# ---------------------------------------------------------------------------

def _assemble(name, Hq, Hkv, d, dtype, node_len, parent, query_node, seed,
              first_offset=None, explicit_pages=None, permute=True, page_slack=0,
              lid=None, lid_ptr=None, meta=None) -> Workload:
    """Give every node its own pages (or the explicit logical page lists), then
    map logical pages to a seeded random permutation of physical pages."""
    N = len(node_len)
    node_len = np.asarray(node_len, dtype=np.int32)
    parent = np.asarray(parent, dtype=np.int32)
    fo = np.zeros(N, dtype=np.int32) if first_offset is None else np.asarray(first_offset, np.int32)
    if explicit_pages is None:
        lists, nxt = [], 0
        for n in range(N):
            L = int(node_len[n])
            cnt = 0 if L == 0 else -(-(int(fo[n]) + L) // PAGE)
            lists.append(list(range(nxt, nxt + cnt)))
            nxt += cnt
        n_logical = nxt
    else:
        lists = explicit_pages
        n_logical = 1 + max((p for l in lists for p in l), default=-1)
    num_pages = n_logical + page_slack
    if permute:
        perm = _permutation(rng.stream_key(seed, 21), num_pages)
    else:
        perm = np.arange(num_pages, dtype=np.int64)
    page_ptr = np.zeros(N + 1, dtype=np.int64)
    page_ptr[1:] = np.cumsum([len(l) for l in lists])
    flat = [p for l in lists for p in l]
    page_ids = perm[np.asarray(flat, dtype=np.int64)].astype(np.int32) if flat else \
        np.zeros(0, dtype=np.int32)
    if lid is None:
        lid_ptr = np.zeros(N + 1, dtype=np.int64)
        lid_ptr[1:] = np.cumsum(node_len.astype(np.int64))
        lid = np.arange(int(lid_ptr[-1]), dtype=np.int64)
    return Workload(name=name, n_q_heads=Hq, n_kv_heads=Hkv, d=d, dtype=dtype,
                    page_size=PAGE, node_len=node_len, parent=parent, first_offset=fo,
                    page_ptr=page_ptr, page_ids=page_ids, num_pages=num_pages,
                    query_node=np.asarray(query_node, dtype=np.int32),
                    lid_ptr=np.asarray(lid_ptr, np.int64), lid=np.asarray(lid, np.int64),
                    seed=seed, meta=meta or {})


def _permutation(key: int, n: int) -> np.ndarray:
    """Seeded permutation of range(n): argsort of one 64-bit draw per item."""
    z = rng.splitmix64(key, np.arange(n, dtype=np.uint64))
    return np.argsort(z, kind="stable").astype(np.int64)


def config_seed(cfg: int) -> int:
    return 0x5EED0000 + cfg


# ---------------------------------------------------------------------------
# the five workload shapes
# ---------------------------------------------------------------------------

def tiny_two_level(seed: int | None = None) -> Workload:
    """Root prefix of 256 tokens, 4 leaves x 32 tokens, one decode query per
    leaf; MHA 4 heads, d=64, fp32."""
    seed = config_seed(1) if seed is None else seed
    node_len = [256, 32, 32, 32, 32]
    parent = [-1, 0, 0, 0, 0]
    return _assemble("tiny_two_level", 4, 4, 64, "f32", node_len, parent, [1, 2, 3, 4], seed,
                     meta={"config": 1})


def document_qa(seed: int | None = None, prefix: int = 32768, n_req: int = 64,
                suffix_lo: int = 64, suffix_hi: int = 512, heads: tuple = (32, 8)) -> Workload:
    """One shared prefix of 32K tokens and 64 requests with unique suffixes of
    U{64..512} tokens, one query per request; 32 Q / 8 KV heads (`heads`),
    d=128, bf16."""
    seed = config_seed(2) if seed is None else seed
    key = rng.stream_key(seed, 31)
    suff = [rng.uniform_int(key, i, suffix_lo, suffix_hi) for i in range(n_req)]
    node_len = [prefix] + suff
    parent = [-1] + [0] * n_req
    return _assemble("document_qa", heads[0], heads[1], 128, "bf16", node_len, parent,
                     list(range(1, n_req + 1)), seed, meta={"config": 2})


def few_shot(seed: int | None = None, prefix: int = 4000, n_branch: int = 16,
             branch_len: int = 256, n_leaf: int = 4, leaf_len: int = 32) -> Workload:
    """Shared prefix of 4000 tokens, 16 branches x 256 tokens, each forking into
    4 leaves x 32 tokens (64 queries); 32 Q / 8 KV heads, d=128, bf16."""
    seed = config_seed(3) if seed is None else seed
    node_len, parent, qn = [prefix], [-1], []
    for b in range(n_branch):
        bi = len(node_len)
        node_len.append(branch_len)
        parent.append(0)
        for _ in range(n_leaf):
            qn.append(len(node_len))
            node_len.append(leaf_len)
            parent.append(bi)
    return _assemble("few_shot", 32, 8, 128, "bf16", node_len, parent, qn, seed,
                     meta={"config": 3})


def speculative(seed: int | None = None, batch: int = 8, prompt: int = 8192,
                n_draft: int = 64, depth: int = 6) -> Workload:
    """Batch of 8 trees: an 8K-token prompt and a 64-node single-token draft
    tree of depth exactly 6 under it; all draft nodes are queries.

    Level sizes n_1..n_6 >= 1 sum to 64 (a seeded composition); each draft's
    parent is uniform over the previous level, level 1 hangs off the prompt.
    Draft nodes are numbered level by level and their tokens sit one after the
    other in 4 pages shared between them (a node starts mid-page).
    """
    seed = config_seed(4) if seed is None else seed
    node_len, parent, qn, pages, fo = [], [], [], [], []
    nxt = 0
    levels_meta = []
    for t in range(batch):
        kt = rng.stream_key(seed, 41, t)
        # composition of n_draft into `depth` positive parts: 5 distinct cuts in 1..63
        cand = list(range(1, n_draft))
        for i in range(depth - 1):           # partial Fisher-Yates
            j = rng.uniform_int(kt, i, i, len(cand) - 1)
            cand[i], cand[j] = cand[j], cand[i]
        cuts = sorted(cand[:depth - 1])
        sizes = [b - a for a, b in zip([0] + cuts, cuts + [n_draft])]
        levels_meta.append(sizes)
        root = len(node_len)
        node_len.append(prompt)
        parent.append(-1)
        fo.append(0)
        npg = -(-prompt // PAGE)
        pages.append(list(range(nxt, nxt + npg)))
        nxt += npg
        draft_base_page = nxt
        nxt += -(-n_draft // PAGE)
        prev = [root]
        j = 0
        for lvl, sz in enumerate(sizes):
            cur = []
            for s in range(sz):
                pidx = rng.uniform_int(kt, 1000 + j, 0, len(prev) - 1)
                nid = len(node_len)
                node_len.append(1)
                parent.append(prev[pidx])
                fo.append(j % PAGE)
                pages.append([draft_base_page + j // PAGE])
                qn.append(nid)
                cur.append(nid)
                j += 1
            prev = cur
    return _assemble("speculative", 32, 8, 128, "bf16", node_len, parent, qn, seed,
                     first_offset=fo, explicit_pages=pages,
                     meta={"config": 4, "levels": levels_meta})


def tree_of_thought(variant: str = "gqa", seed: int | None = None) -> Workload:
    """Root + 4 levels; per-level branching b_1..b_4 in {2..8} drawn (by
    rejection) until their product is 256, so there are exactly 256 leaves with
    one query each; node lengths round(exp(U(ln 16, ln 8192))) clamped to
    [16, 8192]. Variants: MHA 32/32, GQA 32/8, MQA 32/1; d=128, bf16."""
    seed = config_seed(5) if seed is None else seed
    hkv = {"mha": 32, "gqa": 8, "mqa": 1}[variant]
    kt = rng.stream_key(seed, 51)
    c = 0
    while True:
        b = [rng.uniform_int(kt, 4 * c + l, 2, 8) for l in range(4)]
        c += 1
        if math.prod(b) == 256:
            break
    kl = rng.stream_key(seed, 52)
    node_len, parent = [], []
    lo, hi = math.log(16.0), math.log(8192.0)

    def length(i):
        u = rng.uniform_real(kl, i)
        return int(min(8192, max(16, round(math.exp(lo + u * (hi - lo))))))

    node_len.append(length(0))
    parent.append(-1)
    level = [0]
    for bl in b:
        nxt = []
        for p in level:
            for _ in range(bl):
                nid = len(node_len)
                node_len.append(length(nid))
                parent.append(p)
                nxt.append(nid)
        level = nxt
    return _assemble(f"tree_of_thought_{variant}", 32, hkv, 128, "bf16", node_len, parent,
                     level, seed, meta={"config": 5, "branching": b, "variant": variant})


def flat_control(wl: Workload) -> Workload:
    """The same batch with no sharing: one single-node tree per query holding its
    whole root-to-node sequence in freshly allocated (copied) pages."""
    node_len, lids = [], []
    for q in range(wl.n_queries):
        path = []
        n = int(wl.query_node[q])
        while n >= 0:
            path.append(n)
            n = int(wl.parent[n])
        seq = [wl.lid[wl.lid_ptr[m]:wl.lid_ptr[m + 1]] for m in reversed(path)]
        s = np.concatenate(seq) if seq else np.zeros(0, np.int64)
        lids.append(s)
        node_len.append(len(s))
    lid_ptr = np.zeros(len(node_len) + 1, dtype=np.int64)
    lid_ptr[1:] = np.cumsum(node_len)
    out = _assemble(wl.name + "_flat", wl.n_q_heads, wl.n_kv_heads, wl.d, wl.dtype,
                    node_len, [-1] * len(node_len), list(range(len(node_len))), wl.seed,
                    lid=np.concatenate(lids), lid_ptr=lid_ptr, meta=dict(wl.meta, flat=True))
    return out


def source_rows(src: Workload, dst: Workload) -> np.ndarray:
    """int64 [dst.num_pages * page_size]: for every pool row of `dst`, the pool
    row of `src` that holds the same logical token (-1 where `dst`'s row is
    unused or `src` lacks the token). With it, `dst`'s pools (e.g. the flat
    control of `src`) can be filled by copying `src`'s rows, since a token's
    K/V depend on its logical id only."""
    where = np.full(int(src.lid.max()) + 1 if src.lid.size else 1, -1, dtype=np.int64)
    srows = src.row_lids()
    used = np.nonzero(srows >= 0)[0]
    where[srows[used]] = used
    drows = dst.row_lids()
    out = np.full(drows.shape, -1, dtype=np.int64)
    ok = (drows >= 0) & (drows < where.size)
    out[ok] = where[drows[ok]]
    return out


def grow_query_nodes(wl: Workload, tokens: int = 1) -> Workload:
    """The next decode steps' tree: every node a query sits on gains `tokens`
    tokens (new logical ids), in free rows of its last page or in new pages
    appended to the pool; the shape, the other nodes and every existing row
    stay as they are."""
    ps = wl.page_size
    grow = np.zeros(wl.n_nodes, dtype=np.int64)
    grow[np.unique(wl.query_node)] = tokens
    node_len = wl.node_len.astype(np.int64) + grow
    next_lid = int(wl.lid.max()) + 1 if wl.lid.size else 0
    num_pages = wl.num_pages
    page_lists, lid_lists = [], []
    for n in range(wl.n_nodes):
        pages = [int(p) for p in wl.page_ids[wl.page_ptr[n]:wl.page_ptr[n + 1]]]
        need = (int(wl.first_offset[n]) + int(node_len[n]) + ps - 1) // ps if node_len[n] > 0 else len(pages)
        while len(pages) < need:
            pages.append(num_pages)
            num_pages += 1
        page_lists.append(pages)
        lids = wl.lid[wl.lid_ptr[n]:wl.lid_ptr[n + 1]]
        if grow[n]:
            lids = np.concatenate([lids, np.arange(next_lid, next_lid + grow[n], dtype=np.int64)])
            next_lid += int(grow[n])
        lid_lists.append(lids)
    page_ptr = np.zeros(wl.n_nodes + 1, dtype=np.int64)
    page_ptr[1:] = np.cumsum([len(p) for p in page_lists])
    lid_ptr = np.zeros(wl.n_nodes + 1, dtype=np.int64)
    lid_ptr[1:] = np.cumsum([len(x) for x in lid_lists])
    # the new rows must be free (a page shared with another node may not be)
    used = wl.row_lids()
    for n in np.flatnonzero(grow):
        pos = int(wl.first_offset[n]) + int(wl.node_len[n]) + np.arange(tokens)
        pages = np.array(page_lists[n], dtype=np.int64)
        rows = pages[pos // ps] * ps + pos % ps
        old = rows[rows < used.shape[0]]
        if np.any(used[old] >= 0):
            raise ValueError(f"node {n} cannot grow in place: its next page rows hold other tokens")
    return dataclasses.replace(
        wl, name=wl.name + f"+{tokens}", node_len=node_len.astype(np.int32), page_ptr=page_ptr,
        page_ids=np.array([p for pl in page_lists for p in pl], dtype=np.int32), num_pages=num_pages,
        lid_ptr=lid_ptr, lid=np.concatenate(lid_lists) if lid_lists else wl.lid)


def speculative_next_step(wl: Workload, seed: int, n_draft: int = 64, depth: int = 6):
    """The tree of the next speculative decoding step, and for each of its
    nodes the id of the same node in `wl` (-1 for a new node).

    In every tree (a top-level prompt node and its single-token draft nodes)
    one draft is accepted, together with the drafts on its path: those keep
    their tokens and pages and now form a chain under the prompt; every other
    draft is pruned (its page rows become unused). A new draft tree of
    `n_draft` single-token nodes and exactly `depth` levels (a seeded
    composition of the level sizes, parents uniform over the previous level)
    hangs off the last accepted draft, in new pages appended to the pool with
    new logical ids; the new drafts are the step's queries."""
    ps = wl.page_size
    kids = [[] for _ in range(wl.n_nodes)]
    for n in range(wl.n_nodes):
        if wl.parent[n] >= 0:
            kids[int(wl.parent[n])].append(n)
    next_lid = int(wl.lid.max()) + 1 if wl.lid.size else 0
    num_pages = wl.num_pages
    node_len, parent, fo, page_lists, lid_lists, prev_node, qn = [], [], [], [], [], [], []

    def keep(old, new_parent):
        prev_node.append(old)
        node_len.append(int(wl.node_len[old]))
        parent.append(new_parent)
        fo.append(int(wl.first_offset[old]))
        page_lists.append([int(p) for p in wl.page_ids[wl.page_ptr[old]:wl.page_ptr[old + 1]]])
        lid_lists.append(wl.lid[wl.lid_ptr[old]:wl.lid_ptr[old + 1]])
        return len(node_len) - 1

    roots = [n for n in range(wl.n_nodes) if wl.parent[n] < 0]
    for t, r in enumerate(roots):
        kt = rng.stream_key(seed, 51, t)
        drafts, stack = [], list(kids[r])
        while stack:
            n = stack.pop()
            drafts.append(n)
            stack.extend(kids[n])
        drafts.sort()
        # the accepted draft and its path below the prompt
        path = []
        if drafts:
            a = drafts[rng.uniform_int(kt, 0, 0, len(drafts) - 1)]
            while a != r:
                path.append(a)
                a = int(wl.parent[a])
            path.reverse()
        last = keep(r, -1)
        for a in path:
            last = keep(a, last)
        # the new draft tree
        cand = list(range(1, n_draft))
        for i in range(depth - 1):
            j = rng.uniform_int(kt, 1 + i, i, len(cand) - 1)
            cand[i], cand[j] = cand[j], cand[i]
        cuts = sorted(cand[:depth - 1])
        sizes = [b - a for a, b in zip([0] + cuts, cuts + [n_draft])]
        base_page = num_pages
        num_pages += -(-n_draft // ps)
        prev_level = [last]
        j = 0
        for sz in sizes:
            cur = []
            for _ in range(sz):
                pidx = rng.uniform_int(kt, 1000 + j, 0, len(prev_level) - 1)
                prev_node.append(-1)
                node_len.append(1)
                parent.append(prev_level[pidx])
                fo.append(j % ps)
                page_lists.append([base_page + j // ps])
                lid_lists.append(np.array([next_lid], dtype=np.int64))
                next_lid += 1
                qn.append(len(node_len) - 1)
                cur.append(len(node_len) - 1)
                j += 1
            prev_level = cur
    N = len(node_len)
    page_ptr = np.zeros(N + 1, dtype=np.int64)
    page_ptr[1:] = np.cumsum([len(p) for p in page_lists])
    lid_ptr = np.zeros(N + 1, dtype=np.int64)
    lid_ptr[1:] = np.cumsum([len(x) for x in lid_lists])
    nxt = dataclasses.replace(
        wl, name=wl.name + "+step", node_len=np.array(node_len, dtype=np.int32),
        parent=np.array(parent, dtype=np.int32), first_offset=np.array(fo, dtype=np.int32), page_ptr=page_ptr,
        page_ids=np.array([p for pl in page_lists for p in pl], dtype=np.int32), num_pages=num_pages,
        query_node=np.array(qn, dtype=np.int32), lid_ptr=lid_ptr, lid=np.concatenate(lid_lists))
    return nxt, np.array(prev_node, dtype=np.int32)


def random_tree(seed: int, max_nodes: int = 12, max_len: int = 70, max_depth: int = 4,
                heads=(4, 2), d: int = 64, dtype: str = "bf16", n_queries: int | None = None,
                allow_empty: bool = True, random_offsets: bool = True) -> Workload:
    """A small random forest for exhaustive parity checks: lengths 0..max_len
    (ragged pages), random first offsets, queries on random nodes (any depth)."""
    k = rng.stream_key(seed, 61)
    c = [0]

    def ri(lo, hi):
        c[0] += 1
        return rng.uniform_int(k, c[0], lo, hi)

    N = ri(1, max_nodes)
    parent, depth, node_len, fo = [], [], [], []
    for n in range(N):
        if n == 0 or ri(0, 4) == 0:
            parent.append(-1)
            depth.append(0)
        else:
            cands = [m for m in range(n) if depth[m] < max_depth - 1]
            p = cands[ri(0, len(cands) - 1)] if cands else -1
            parent.append(p)
            depth.append(0 if p < 0 else depth[p] + 1)
        L = ri(0 if allow_empty else 1, max_len)
        node_len.append(L)
        fo.append(ri(0, PAGE - 1) if (random_offsets and L > 0) else 0)
    # every query must see at least one token: sit queries on nodes whose path
    # has a token
    def path_len(n):
        s = 0
        while n >= 0:
            s += node_len[n]
            n = parent[n]
        return s
    ok = [n for n in range(N) if path_len(n) > 0]
    if not ok:
        node_len[0] = 1 + ri(0, max_len - 1)
        ok = [n for n in range(N) if path_len(n) > 0]
    B = n_queries if n_queries is not None else ri(1, 2 * N + 2)
    qn = [ok[ri(0, len(ok) - 1)] for _ in range(B)]
    Hq, Hkv = heads
    return _assemble(f"random_{seed}", Hq, Hkv, d, dtype, node_len, parent, qn, seed,
                     first_offset=fo, page_slack=ri(0, 3), meta={"random": True})


CONFIGS = {
    1: ("tiny_two_level", tiny_two_level),
    2: ("document_qa", document_qa),
    3: ("few_shot", few_shot),
    4: ("speculative", speculative),
    5: ("tree_of_thought_gqa", lambda seed=None: tree_of_thought("gqa", seed)),
}


def paged_example() -> Workload:
    """Two 100-token requests sharing a 96-token prefix (pages 0-5) with 4-token
    suffixes in pages 6 and 7, page size 16, identity page mapping -- the
    block-table example of the shared-prefix techniques blog (section 4.3)."""
    return _assemble("paged_example", 2, 1, 64, "bf16", [96, 4, 4], [-1, 0, 0], [1, 2],
                     seed=0x5EED00AA, permute=False)


def cascade_example(n: int = 7, prefix: int = 512 * 16) -> Workload:
    """n requests sharing one prefix, each with its own suffix (the cascade
    attention decode example): node 0 is the prefix, node i+1 request i's suffix."""
    return _assemble("cascade_example", 2, 1, 64, "bf16", [prefix] + [16 + 3 * i for i in range(n)],
                     [-1] + [0] * n, list(range(1, n + 1)), seed=0x5EED00AB)
