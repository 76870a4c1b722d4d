"""Oracle, floating-point side: decode attention over a KV forest in fp64.

TEST INFRASTRUCTURE (see the package docstring).

Sources
  * CoDec, "background": O = softmax(Q K^T / sqrt(d)) V.
  * CoDec, "KV cache management": the node-local stabilised accumulators
    s_{r,n} = q_r K_n^T / sqrt(d_k), m_{r,n} = max_j s, d_{r,n} = sum_j e^{s-m},
    u_{r,n} = sum_j e^{s-m} V_n[j] -- see ``partial_attention``.
  * CoDec, "intra-block primitives", POR: m = max(m1, m2),
    s = s1 e^{m1-m} + s2 e^{m2-m}, O = (O1 s1 e^{m1-m} + O2 s2 e^{m2-m}) / s --
    see ``por``.
  * DEFT, section 3.2: LSE(q, k) = log sum exp(q k^T / sqrt(d)), natural log.

Readings where the pages leave a step open
  * A decode query attends every token on the path from the top of its tree
    down to the node it sits on, that node included.
  * GQA: q-head h reads kv head floor(h / (Hq / Hkv)).
  * bf16 inputs are taken at their exact values; all arithmetic is fp64.
"""
from __future__ import annotations

import math

import numpy as np

from . import tree as _tree


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns: they are the top half of an fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_to_f64(x)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def node_kv(tr, K_pool, V_pool, n):
    """K, V of node n's tokens in token order, read through the node's own
    pages: fp64 arrays [Hkv, len, d] (each kv head's block contiguous)."""
    pages, rows = _tree.node_rows(tr, n)
    k = to_f64(K_pool[pages, :, rows, :], tr.dtype)   # [len, Hkv, d]
    v = to_f64(V_pool[pages, :, rows, :], tr.dtype)
    return np.ascontiguousarray(k.transpose(1, 0, 2)), np.ascontiguousarray(v.transpose(1, 0, 2))


def path_kv(tr, K_pool, V_pool, path, cache=None) -> tuple[list, list]:
    """K, V of the path's nodes in path order (each node's tokens in token
    order, read through its own pages): two lists of fp64 blocks [Hkv, len, d],
    whose concatenation along the token axis is the path's K and V.

    ``cache`` (optional dict, node id -> node_kv result) keeps the blocks of
    nodes already read, so that queries sharing a prefix decode it once."""
    ks, vs = [], []
    for n in path:
        n = int(n)
        if int(tr.node_len[n]) == 0:
            continue
        if cache is not None and n in cache:
            k, v = cache[n]
        else:
            k, v = node_kv(tr, K_pool, V_pool, n)
            if cache is not None:
                cache[n] = (k, v)
        ks.append(k)
        vs.append(v)
    return ks, vs


def attention_definition(q: np.ndarray, K, V):
    """Query rows q [d] (or [R, d]) against K, V [L, d]: (o, lse) with
    o = softmax(q K^T / sqrt(d)) V and lse = ln sum_j exp(s_j) per row, in
    fp64; o is [d] (or [R, d]) and lse a float (or [R]).

    K and V may also be given as lists of row blocks [L_i, d] (a path's nodes
    in order) that stack to the full K and V: the scores are then the stacked
    blocks' scores, and o the sum of the blocks' weighted rows."""
    Ks = list(K) if isinstance(K, (list, tuple)) else [K]
    Vs = list(V) if isinstance(V, (list, tuple)) else [V]
    d = q.shape[-1]
    s = np.concatenate([Kb @ q.T for Kb in Ks], axis=0) / math.sqrt(d)   # s_j = q . k_j / sqrt(d)
    m = np.max(s, axis=0)
    total = np.sum(np.exp(s - m), axis=0)
    lse = m + np.log(total)
    p = np.exp(s - lse)                        # softmax weights, token axis first
    o = 0.0
    j = 0
    for Vb in Vs:
        o = o + p[j:j + Vb.shape[0]].T @ Vb
        j += Vb.shape[0]
    return o, (float(lse) if np.ndim(lse) == 0 else lse)


def decode_attention(tr, K_pool, V_pool, Q, queries=None):
    """O [B, Hq, d] and LSE [B, Hq] (fp64) for the listed queries (all if None).

    ``tr`` carries the tree arrays: node_len, parent, first_offset, page_ptr,
    page_ids, page_size, query_node, n_q_heads, n_kv_heads, d, dtype.
    Rows of queries not listed are NaN."""
    B, Hq, d = Q.shape
    Hkv = K_pool.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    O = np.full((B, Hq, d), np.nan)
    LSE = np.full((B, Hq), np.nan)
    qs = range(B) if queries is None else queries
    cache: dict = {}
    for qi in qs:
        path = _tree.root_path(tr.parent, int(tr.query_node[qi]))
        # keep only the decoded blocks of this query's path (queries listed in
        # tree order share most of theirs)
        on_path = set(int(n) for n in path)
        for n in list(cache):
            if n not in on_path:
                del cache[n]
        Kq, Vq = path_kv(tr, K_pool, V_pool, path, cache)
        if not Kq:
            raise ValueError(f"query {qi} sees no token")
        qf = to_f64(Q[qi], tr.dtype)
        for g in range(Hkv):
            # the q-heads h with h // G == g read kv head g
            O[qi, g * G:(g + 1) * G], LSE[qi, g * G:(g + 1) * G] = attention_definition(
                qf[g * G:(g + 1) * G], [k[g] for k in Kq], [v[g] for v in Vq])
    return O, LSE


# --------------------------------------------------------------------------
# node-local accumulators and the partial-output merge
# --------------------------------------------------------------------------

def partial_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, visible=None):
    """CoDec's per-node stabilised accumulation for one query row:
    (m, dsum, u) with s = q K^T / sqrt(d) (masked where ``visible`` is False),
    m = max s, dsum = sum e^{s-m}, u = sum e^{s-m} V[j]."""
    d = q.shape[-1]
    s = (K @ q) / math.sqrt(d)
    if visible is not None:
        s = np.where(visible, s, -np.inf)
    m = np.max(s)
    e = np.exp(s - m)
    return m, float(np.sum(e)), e @ V


def normalised(m, dsum, u):
    """Partial output O_i = u / dsum with its max m and sum s = dsum (POR inputs)."""
    return u / dsum, m, dsum


def por(o1, m1, s1, o2, m2, s2):
    """Merge two partial outputs of the same query (CoDec POR)."""
    m = max(m1, m2)
    w1 = s1 * math.exp(m1 - m)
    w2 = s2 * math.exp(m2 - m)
    s = w1 + w2
    o = (o1 * w1 + o2 * w2) / s
    return o, m, s


def lse_of(m, s) -> float:
    """Natural-log LSE of a partial with max m and sum s."""
    return m + math.log(s)
