"""Oracle, integer side: the KV forest index, the page walk and IO counts.

TEST INFRASTRUCTURE (see the package docstring): plain Python over the tree
arrays, no shared code with the library.

Sources
  * CoDec, "KV cache management" -- the KV forest with a virtual root, edge
    p->c meaning "p is a prefix of c", and the index recording which queries
    share each node and which nodes make up each query's prefix.
  * DEFT, Algorithm 1 (DEFT-Node QKV preparation) -- QMapKV (per query, the
    KV nodes of all its prefixes) and KVMapQ (per node, the queries that
    share it): KV-guided grouping.
  * Shared-prefix techniques blog, section 4.3 -- block tables of paged KV
    (token t of a sequence lives at page table[t // page], row t % page).
  * CoDec, "complexity analysis" -- IO of the tree kernel is h*d*sum_i n[i]
    against h*d*sum_i n[i]*n_q[i] for per-query kernels.
"""
from __future__ import annotations

import numpy as np


def root_path(parent, node: int) -> list[int]:
    """Nodes from the top of the forest down to ``node`` (inclusive).

    Raises ValueError on a cycle (a walk longer than the number of nodes)."""
    out = []
    n = int(node)
    limit = len(parent) + 1
    while n >= 0:
        out.append(n)
        if len(out) > limit:
            raise ValueError("cycle in parent array")
        n = int(parent[n])
    out.reverse()
    return out


def query_paths(parent, query_node) -> list[list[int]]:
    """QMapKV: for each query, the nodes forming its prefix, root first."""
    return [root_path(parent, int(v)) for v in query_node]


def node_queries(parent, query_node, n_nodes: int) -> list[list[int]]:
    """KVMapQ: for each node, the ascending ids of the queries whose prefix
    contains it (the queries the node's KV is grouped with)."""
    out: list[list[int]] = [[] for _ in range(n_nodes)]
    for q, path in enumerate(query_paths(parent, query_node)):
        for n in path:
            out[n].append(q)
    return out


def token_location(tree, node: int, t: int) -> tuple[int, int]:
    """(physical page, row) holding token t of ``node``: the node's tokens run
    contiguously from ``first_offset`` in its first listed page."""
    ps = int(tree.page_size)
    pos = int(tree.first_offset[node]) + int(t)
    page = int(tree.page_ids[int(tree.page_ptr[node]) + pos // ps])
    return page, pos % ps


def node_rows(tree, node: int) -> tuple[np.ndarray, np.ndarray]:
    """Vector form of token_location over all tokens of ``node``."""
    ps = int(tree.page_size)
    L = int(tree.node_len[node])
    pos = int(tree.first_offset[node]) + np.arange(L, dtype=np.int64)
    base = int(tree.page_ptr[node])
    pages = np.asarray(tree.page_ids, dtype=np.int64)[base + pos // ps]
    return pages, pos % ps


def visible_tokens(tree, q: int) -> list[tuple[int, int]]:
    """(node, token) pairs query q attends to: every token on the path from the
    top of the forest to the query's node, inclusive, in path order."""
    out = []
    for n in root_path(tree.parent, int(tree.query_node[q])):
        out.extend((n, t) for t in range(int(tree.node_len[n])))
    return out


def block_table(tree, q: int) -> tuple[list[int], int]:
    """Flat page list of query q's sequence and the number of rows used in its
    last page, for trees whose nodes start on a page boundary (PagedAttention
    style block table)."""
    pages: list[int] = []
    last = 0
    for n in root_path(tree.parent, int(tree.query_node[q])):
        L = int(tree.node_len[n])
        if L == 0:
            continue
        if int(tree.first_offset[n]) != 0:
            raise ValueError("block_table needs page-aligned nodes")
        lo, hi = int(tree.page_ptr[n]), int(tree.page_ptr[n + 1])
        pages.extend(int(p) for p in tree.page_ids[lo:hi])
        last = (L - 1) % int(tree.page_size) + 1
    return pages, last


def kv_token_counts(tree) -> tuple[int, int]:
    """(unique tokens, flat tokens): tokens stored once in the tree vs. tokens a
    per-query (flat) kernel reads -- the sum over queries of their path lengths."""
    unique = int(np.sum(np.asarray(tree.node_len, dtype=np.int64)))
    flat = 0
    for q in range(len(tree.query_node)):
        flat += sum(int(tree.node_len[n]) for n in root_path(tree.parent, int(tree.query_node[q])))
    return unique, flat


def kv_bytes(tokens: int, n_kv_heads: int, d: int, elem_bytes: int) -> int:
    """K and V bytes of ``tokens`` tokens over all kv heads."""
    return int(tokens) * int(n_kv_heads) * 2 * int(d) * int(elem_bytes)


def q_tile_scan(groups, q_tile: int) -> tuple[int, int]:
    """Thread blocks and KV tokens scanned when each group's query rows are
    packed in order into tiles of ``q_tile`` rows and every tile scans as many
    KV tokens as its furthest-reaching row (FlashAttention execution model,
    shared-prefix techniques blog section 5.1).

    ``groups`` is a list of lists: per group, the KV span each row scans."""
    ctas = 0
    scanned = 0
    for g in groups:
        for i in range(0, len(g), q_tile):
            ctas += 1
            scanned += max(g[i:i + q_tile])
    return ctas, scanned
