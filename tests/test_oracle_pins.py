"""Pins of the fp64 oracle to things other than itself.

* brute force: per-request flat attention on sequences materialised straight
  from the generator's logical node arrays (no page tables), with a
  pure-Python textbook softmax;
* closed forms: single-token KV, constant V, equal scores;
* POR algebra: random partial splits merged in random orders and tree shapes
  (associativity and commutativity of the CoDec merge);
* the FlashAttention online-softmax loop (KV-cache engineering blog, section 3)
  as a third fp64 path;
* planted mistakes: each plausible bug in the oracle fails one of the above.
"""
import json
import math
import os
import types

import numpy as np
import pytest

import oracle
from oracle import attention as oa
from oracle import tree as ot
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers

def brute_force(wl, q_idx):
    """Textbook attention in pure Python for one query, all heads, from the
    generator's logical per-node arrays."""
    path = []
    n = int(wl.query_node[q_idx])
    while n >= 0:
        path.append(n)
        n = int(wl.parent[n])
    path.reverse()
    Ks, Vs = [], []
    for n in path:
        k, v = wl.node_kv_logical(n)
        Ks.extend(k)
        Vs.extend(v)
    Qraw = wl.q()[q_idx]
    if wl.dtype == "bf16":
        Qf = (Qraw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        Qf = Qraw.astype(np.float64)
    Hq, Hkv, d = wl.n_q_heads, wl.n_kv_heads, wl.d
    G = Hq // Hkv
    outs, lses = [], []
    for h in range(Hq):
        g = h // G
        scores = []
        for kt in Ks:
            acc = 0.0
            for e in range(d):
                acc += float(Qf[h][e]) * float(kt[g][e])
            scores.append(acc / math.sqrt(d))
        mx = max(scores)
        den = sum(math.exp(s - mx) for s in scores)
        o = [0.0] * d
        for s, vt in zip(scores, Vs):
            w = math.exp(s - mx) / den
            for e in range(d):
                o[e] += w * float(vt[g][e])
        outs.append(o)
        lses.append(mx + math.log(den))
    return np.array(outs), np.array(lses)


def run_oracle(wl, queries=None):
    K, V = wl.kv_pools(workers=1)
    return oa.decode_attention(wl, K, V, wl.q(), queries)


def close(a, b, tol=1e-12):
    a, b = np.asarray(a, float), np.asarray(b, float)
    return np.all(np.abs(a - b) <= tol * np.maximum(1.0, np.abs(b)))


def pin_brute_force(wl, queries):
    O, L = run_oracle(wl, queries)
    for q in queries:
        bo, bl = brute_force(wl, q)
        if not (close(O[q], bo) and close(L[q], bl)):
            return False
    return True


# ------------------------------------------------------------ brute force

@pytest.mark.parametrize("seed,heads,d,dtype", [
    (1, (4, 2), 8, "bf16"), (2, (2, 2), 16, "f32"), (3, (4, 1), 8, "bf16"),
    (4, (6, 3), 8, "f32"), (5, (1, 1), 4, "bf16"),
])
def test_oracle_matches_brute_force(seed, heads, d, dtype):
    wl = synth.random_tree(seed, max_nodes=6, max_len=20, heads=heads, d=d, dtype=dtype)
    assert pin_brute_force(wl, list(range(wl.n_queries)))


# ------------------------------------------------------------ closed forms

def _tiny_tree(node_len, parent, query_node, Hq, Hkv, d, K, V, Q):
    """A hand-made tree with one page per 16 tokens, identity page ids."""
    ps = 16
    page_ptr = [0]
    ids = []
    nxt = 0
    for L in node_len:
        c = -(-L // ps)
        ids.extend(range(nxt, nxt + c))
        nxt += c
        page_ptr.append(len(ids))
    tr = types.SimpleNamespace(node_len=np.array(node_len), parent=np.array(parent),
                               first_offset=np.zeros(len(node_len), int),
                               page_ptr=np.array(page_ptr), page_ids=np.array(ids),
                               page_size=ps, query_node=np.array(query_node),
                               n_q_heads=Hq, n_kv_heads=Hkv, d=d, dtype="f32")
    Kp = np.zeros((nxt, Hkv, ps, d), np.float32)
    Vp = np.zeros((nxt, Hkv, ps, d), np.float32)
    t = 0
    for n, L in enumerate(node_len):
        for j in range(L):
            p, r = ot.token_location(tr, n, j)
            Kp[p, :, r] = K[t]
            Vp[p, :, r] = V[t]
            t += 1
    return tr, Kp, Vp, np.asarray(Q, np.float32)


def test_closed_form_single_token():
    r = np.random.default_rng(0)
    d = 8
    k, v, q = r.standard_normal((1, 1, d)), r.standard_normal((1, 1, d)), r.standard_normal((1, 1, d))
    tr, Kp, Vp, Q = _tiny_tree([1], [-1], [0], 1, 1, d, k, v, q)
    O, L = oa.decode_attention(tr, Kp, Vp, Q)
    kf, vf, qf = (x.astype(np.float32).astype(np.float64) for x in (k, v, q))
    assert close(O[0, 0], vf[0, 0])
    assert close(L[0, 0], float(qf[0, 0] @ kf[0, 0]) / math.sqrt(d))


def test_closed_form_constant_v():
    r = np.random.default_rng(1)
    d, n = 8, 37
    K = r.standard_normal((n, 2, d))
    c = r.standard_normal(d).astype(np.float32)
    V = np.broadcast_to(c, (n, 2, d)).copy()
    tr, Kp, Vp, Q = _tiny_tree([20, 17], [-1, 0], [1], 4, 2, d, K, V, r.standard_normal((1, 4, d)))
    O, _ = oa.decode_attention(tr, Kp, Vp, Q)
    for h in range(4):
        assert close(O[0, h], c.astype(np.float64))


def test_closed_form_equal_scores():
    r = np.random.default_rng(2)
    d, n = 8, 29
    V = r.standard_normal((n, 1, d))
    K = r.standard_normal((n, 1, d))
    tr, Kp, Vp, Q = _tiny_tree([9, 20], [-1, 0], [1], 1, 1, d, K, V, np.zeros((1, 1, d)))
    O, L = oa.decode_attention(tr, Kp, Vp, Q)          # q = 0: all scores 0
    assert close(O[0, 0], V.astype(np.float32).astype(np.float64)[:, 0].mean(0))
    assert close(L[0, 0], math.log(n))
    # identical keys, q != 0: all scores equal s
    k0 = r.standard_normal(d)
    K2 = np.broadcast_to(k0, (n, 1, d)).copy()
    q = r.standard_normal((1, 1, d))
    tr, Kp, Vp, Q = _tiny_tree([9, 20], [-1, 0], [1], 1, 1, d, K2, V, q)
    O, L = oa.decode_attention(tr, Kp, Vp, Q)
    s = float(q.astype(np.float32).astype(np.float64)[0, 0] @ k0.astype(np.float32).astype(np.float64)) / math.sqrt(d)
    assert close(O[0, 0], V.astype(np.float32).astype(np.float64)[:, 0].mean(0))
    assert close(L[0, 0], math.log(n) + s)


# ------------------------------------------------------------ POR algebra

def _random_partials(r, L, d):
    q = r.standard_normal(d) * 2
    K = r.standard_normal((L, d))
    V = r.standard_normal((L, d))
    cuts = sorted(r.choice(np.arange(1, L), size=r.integers(1, min(7, L - 1) + 1), replace=False))
    bounds = [0] + list(cuts) + [L]
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        m, s, u = oa.partial_attention(q, K[a:b], V[a:b])
        parts.append(oa.normalised(m, s, u))
    return q, K, V, parts


def _merge_random_tree(r, parts):
    parts = list(parts)
    while len(parts) > 1:
        i, j = sorted(r.choice(len(parts), size=2, replace=False))
        a, b = parts[i], parts[j]
        if r.random() < 0.5:
            a, b = b, a
        merged = oa.por(*a, *b)
        parts = [p for k, p in enumerate(parts) if k not in (i, j)] + [merged]
    return parts[0]


@pytest.mark.parametrize("seed", range(8))
def test_por_associative_commutative(seed):
    r = np.random.default_rng(100 + seed)
    q, K, V, parts = _random_partials(r, int(r.integers(8, 60)), 16)
    o_ref, lse_ref = oa.attention_definition(q, K, V)
    for _ in range(5):
        o, m, s = _merge_random_tree(r, parts)
        assert close(o, o_ref, 1e-13)
        assert close(oa.lse_of(m, s), lse_ref, 1e-13)
    # pairwise identities
    if len(parts) >= 3:
        a, b, c = parts[:3]
        ab_c = oa.por(*oa.por(*a, *b), *c)
        a_bc = oa.por(*a, *oa.por(*b, *c))
        assert close(ab_c[0], a_bc[0], 1e-14) and close(ab_c[2] * math.exp(ab_c[1] - a_bc[1]), a_bc[2], 1e-14)
        ab, ba = oa.por(*a, *b), oa.por(*b, *a)
        assert close(ab[0], ba[0], 0) and ab[1] == ba[1] and close(ab[2], ba[2], 0)


def test_partial_attention_visibility_mask():
    r = np.random.default_rng(7)
    q, K, V = r.standard_normal(8), r.standard_normal((10, 8)), r.standard_normal((10, 8))
    vis = np.array([1, 0, 1, 1, 0, 0, 1, 0, 1, 1], bool)
    m, s, u = oa.partial_attention(q, K, V, vis)
    o_ref, lse_ref = oa.attention_definition(q, K[vis], V[vis])
    assert close(u / s, o_ref) and close(oa.lse_of(m, s), lse_ref)


# ------------------------------------------------- FlashAttention loop (3rd path)

def flash_loop(q, K, V, block):
    d = q.shape[-1]
    o = np.zeros(V.shape[1])
    m, l = -np.inf, 0.0
    for a in range(0, K.shape[0], block):
        s = K[a:a + block] @ q / math.sqrt(d)
        m_new = max(m, float(np.max(s)))
        p = np.exp(s - m_new)
        scale = math.exp(m - m_new) if m > -np.inf else 0.0
        l = scale * l + float(np.sum(p))
        o = scale * o + p @ V[a:a + block]
        m = m_new
    return o / l, m + math.log(l)


@pytest.mark.parametrize("seed", range(4))
def test_oracle_matches_flash_loop(seed):
    wl = synth.random_tree(200 + seed, max_nodes=5, max_len=40, heads=(4, 2), d=16)
    K, V = wl.kv_pools(workers=1)
    O, L = oa.decode_attention(wl, K, V, wl.q())
    Qf = oa.to_f64(wl.q(), wl.dtype)
    for q in range(wl.n_queries):
        path = ot.root_path(wl.parent, int(wl.query_node[q]))
        Ks = np.concatenate([wl.node_kv_logical(n)[0] for n in path])
        Vs = np.concatenate([wl.node_kv_logical(n)[1] for n in path])
        for h in range(4):
            o, lse = flash_loop(Qf[q, h], Ks[:, h // 2], Vs[:, h // 2], block=7)
            assert close(O[q, h], o, 1e-12) and close(L[q, h], lse, 1e-12)


# ------------------------------------------------------------ integer pins

def test_paged_example_block_tables():
    g = json.load(open(os.path.join(GOLDEN, "paged_example.json")))
    wl = synth.trees.paged_example()
    assert list(wl.node_len) == g["node_len"] and list(wl.parent) == g["parent"]
    tables, last, indptr = [], [], [0]
    for q in range(wl.n_queries):
        t, lp = ot.block_table(wl, q)
        tables.append(t)
        last.append(lp)
        indptr.append(indptr[-1] + len(t))
    assert tables == g["block_tables"]
    assert indptr == g["paged_kv_indptr"]
    assert [p for t in tables for p in t] == g["paged_kv_indices"]
    assert last == g["paged_kv_last_page_len"]
    assert [len(ot.visible_tokens(wl, q)) for q in range(2)] == g["visible_tokens"]


def test_cascade_example_grouping():
    g = json.load(open(os.path.join(GOLDEN, "cascade_grouping.json")))
    wl = synth.trees.cascade_example(g["n_requests"])
    nq = ot.node_queries(wl.parent, wl.query_node, wl.n_nodes)
    shared = [0, len(nq[0])]
    unique = [0]
    for n in range(1, wl.n_nodes):
        unique.append(unique[-1] + len(nq[n]))
    assert [shared, unique] == g["qo_indptr_arr"]
    assert nq[0] == list(range(g["n_requests"]))
    assert all(nq[i + 1] == [i] for i in range(g["n_requests"]))


def test_q_tile_scan_table():
    g = json.load(open(os.path.join(GOLDEN, "q_tile_scan.json")))
    T, P, S = g["q_tile"], g["prefix"], g["suffix"]
    full = P + S
    causal_req = [i + 1 for i in range(full)]            # row i scans KV [0, i]
    schemes = {
        # each request prefilled on its own
        "naive": [causal_req, causal_req],
        # request 0 = [P, S0]; request 1 = only S1 (rows at positions P..P+S-1)
        "direct_ragged": [causal_req, [P + j + 1 for j in range(S)]],
        # prefix prefill, shared level (suffix queries over P), unique level per request
        "cascade": [[i + 1 for i in range(P)], [P] * (2 * S), [j + 1 for j in range(S)],
                    [j + 1 for j in range(S)]],
        # one logical request [P, S0, S1]; suffix rows scan up to their merged position
        "multi_item_scoring": [[i + 1 for i in range(P)] + [P + j + 1 for j in range(2 * S)]],
    }
    for name, groups in schemes.items():
        ctas, scanned = ot.q_tile_scan(groups, T)
        want = g["schemes"][name]
        assert (ctas, scanned) == (want["ctas"], want["kv_scanned"]), name


def test_kv_counts_closed_form():
    wl = synth.document_qa()
    u, f = ot.kv_token_counts(wl)
    suffix = int(wl.node_len[1:].sum())
    assert u == 32768 + suffix
    assert f == 64 * 32768 + suffix
    wl3 = synth.few_shot()
    u3, f3 = ot.kv_token_counts(wl3)
    assert u3 == 4000 + 16 * 256 + 64 * 32 == 10144
    assert f3 == 64 * (4000 + 256 + 32)
    assert ot.kv_bytes(u3, 8, 128, 2) == 41_549_824


def test_node_queries_brute_force():
    for seed in range(20):
        wl = synth.random_tree(300 + seed)
        nq = ot.node_queries(wl.parent, wl.query_node, wl.n_nodes)
        for n in range(wl.n_nodes):
            # a query shares node n iff n is the query's node or one of its ancestors
            want = []
            for q in range(wl.n_queries):
                m = int(wl.query_node[q])
                anc = set()
                while m >= 0:
                    anc.add(m)
                    m = int(wl.parent[m])
                if n in anc:
                    want.append(q)
            assert nq[n] == want


def test_cycle_detected():
    with pytest.raises(ValueError):
        ot.root_path(np.array([1, 0]), 0)


# ------------------------------------------------------------ planted mistakes

def _planted(monkeypatch, kind):
    if kind == "scale":
        def bad(q, K, V):
            K = np.concatenate(K) if isinstance(K, list) else K
            V = np.concatenate(V) if isinstance(V, list) else V
            s = (K @ q.T) / q.shape[-1]
            m = np.max(s, axis=0)
            lse = m + np.log(np.sum(np.exp(s - m), axis=0))
            return np.exp(s - lse).T @ V, lse
        monkeypatch.setattr(oa, "attention_definition", bad)
    elif kind == "gqa":
        orig = oa.decode_attention

        def bad(tr, K_pool, V_pool, Q, queries=None):
            O, L = orig(tr, K_pool, V_pool, Q, queries)
            Hq, Hkv = Q.shape[1], K_pool.shape[1]
            # recompute with h % Hkv (interleaved groups) instead of h // G
            for qi in (range(Q.shape[0]) if queries is None else queries):
                path = ot.root_path(tr.parent, int(tr.query_node[qi]))
                Kq, Vq = oa.path_kv(tr, K_pool, V_pool, path)
                qf = oa.to_f64(Q[qi], tr.dtype)
                for h in range(Hq):
                    O[qi, h], L[qi, h] = oa.attention_definition(qf[h], [k[h % Hkv] for k in Kq],
                                                                  [v[h % Hkv] for v in Vq])
            return O, L
        monkeypatch.setattr(oa, "decode_attention", bad)
    elif kind == "drop_own_node":
        orig = ot.root_path
        monkeypatch.setattr(ot, "root_path", lambda parent, node: orig(parent, node)[:-1]
                            if len(orig(parent, node)) > 1 else orig(parent, node))
    elif kind == "page_row":
        orig = ot.node_rows

        def bad(tr, n):
            p, r = orig(tr, n)
            return p, (r + 1) % int(tr.page_size)
        monkeypatch.setattr(ot, "node_rows", bad)
    elif kind == "transposed_v":
        orig = oa.path_kv

        def bad(tr, K, V, path, cache=None):
            k, v = orig(tr, K, V, path, cache)
            return v, k
        monkeypatch.setattr(oa, "path_kv", bad)


@pytest.mark.parametrize("kind", ["scale", "gqa", "drop_own_node", "page_row", "transposed_v"])
def test_planted_mistake_is_caught(monkeypatch, kind):
    wl = synth.random_tree(11, max_nodes=5, max_len=20, heads=(4, 2), d=8, allow_empty=False)
    assert pin_brute_force(wl, list(range(wl.n_queries)))
    _planted(monkeypatch, kind)
    assert not pin_brute_force(wl, list(range(wl.n_queries)))
