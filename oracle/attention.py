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


def path_kv(tr, K_pool, V_pool, path) -> tuple[np.ndarray, np.ndarray]:
    """K, V of the concatenated path nodes (node order, then token order), read
    through each node's own pages: fp64 arrays [L, Hkv, d]."""
    ks, vs = [], []
    for n in path:
        if int(tr.node_len[n]) == 0:
            continue
        pages, rows = _tree.node_rows(tr, n)
        ks.append(to_f64(K_pool[pages, :, rows, :], tr.dtype))
        vs.append(to_f64(V_pool[pages, :, rows, :], tr.dtype))
    Hkv, d = K_pool.shape[1], K_pool.shape[3]
    if not ks:
        z = np.zeros((0, Hkv, d))
        return z, z.copy()
    return np.concatenate(ks), np.concatenate(vs)


def attention_definition(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """One query row q [d] against K, V [L, d]: (o [d], lse) with
    o = softmax(q K^T / sqrt(d)) V and lse = ln sum_j exp(s_j), both fp64."""
    d = q.shape[-1]
    s = (K @ q) / math.sqrt(d)
    m = np.max(s)
    e = np.exp(s - m)
    total = np.sum(e)
    lse = m + math.log(total)
    o = (np.exp(s - lse)) @ V
    return o, lse


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
    for qi in qs:
        path = _tree.root_path(tr.parent, int(tr.query_node[qi]))
        Kq, Vq = path_kv(tr, K_pool, V_pool, path)
        if Kq.shape[0] == 0:
            raise ValueError(f"query {qi} sees no token")
        qf = to_f64(Q[qi], tr.dtype)
        for h in range(Hq):
            g = h // G
            O[qi, h], LSE[qi, h] = attention_definition(qf[h], Kq[:, g, :], Vq[:, g, :])
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
