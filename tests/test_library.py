"""Host-side checks of libpst (no GPU needed): the library loads and exports
every function the header declares, tree_build rejects malformed trees, the
KV-guided index matches the oracle bit for bit, and every plan covers each
(query, KV token) pair exactly once."""
import ctypes

import numpy as np
import pytest

import synth
from oracle import tree as ot


def test_exports_every_header_symbol(lib):
    names = lib.header_functions()
    assert len(names) >= 18
    L = lib.lib()
    for n in names:
        assert hasattr(L, n), n
        assert ctypes.cast(getattr(L, n), ctypes.c_void_p).value


def _tree(lib, wl, **kw):
    return lib.tree_build(wl.node_len, wl.parent, wl.page_ptr, wl.page_ids, wl.first_offset,
                          wl.page_size, wl.num_pages, **kw)


def _plan(lib, wl, **kw):
    t = _tree(lib, wl)
    kw.setdefault("num_sms", 152)
    return lib.plan_create(t, wl.query_node, wl.n_q_heads, wl.n_kv_heads, wl.d, wl.dtype, **kw)


# ------------------------------------------------------------ validation

def test_tree_build_rejects_bad_input(lib):
    ok = dict(node_len=[20, 5], parent=[-1, 0], page_ptr=[0, 2, 3], page_ids=[0, 1, 2], num_pages=3)
    lib.tree_build(**ok)

    def code(**kw):
        args = dict(ok)
        args.update(kw)
        with pytest.raises(lib.PstError) as e:
            lib.tree_build(**args)
        return e.value.code

    assert code(parent=[1, 0]) == -2                        # cycle
    assert code(parent=[-1, 5]) == -3                       # parent out of range
    assert code(page_ids=[0, 1, 7]) == -3                   # page id >= num_pages
    assert code(node_len=[40, 5]) == -3                     # overruns its 2 pages
    assert code(first_offset=[0, 16]) == -3                 # offset >= page size
    assert code(first_offset=[0, 12]) == -3                 # 12 + 5 > 16
    assert code(page_size=24) == -4
    assert code(node_len=[-1, 5]) == -1
    assert code(page_ptr=[0, 3, 2]) == -1


def test_plan_rejects_bad_input(lib):
    wl = synth.random_tree(5)
    t = _tree(lib, wl)
    with pytest.raises(lib.PstError) as e:
        lib.plan_create(t, wl.query_node, 6, 4, 64, "bf16", num_sms=8)
    assert e.value.code == -4
    with pytest.raises(lib.PstError) as e:
        lib.plan_create(t, wl.query_node, 4, 2, 96, "bf16", num_sms=8)
    assert e.value.code == -4
    with pytest.raises(lib.PstError) as e:
        lib.plan_create(t, [wl.n_nodes], 4, 2, 64, "bf16", num_sms=8)
    assert e.value.code == -1
    # a query whose whole path is empty sees no token
    t2 = lib.tree_build([0, 3], [-1, -1], [0, 0, 1], [0], num_pages=1)
    with pytest.raises(lib.PstError) as e:
        lib.plan_create(t2, [0], 1, 1, 64, "f32", num_sms=8)
    assert e.value.code == -1


# ------------------------------------------------------------ index (bit-exact)

def _workloads():
    out = [synth.tiny_two_level(), synth.few_shot(), synth.document_qa(), synth.speculative(),
           synth.tree_of_thought("gqa"), synth.trees.paged_example(), synth.trees.cascade_example()]
    out += [synth.random_tree(1000 + s) for s in range(40)]
    return out


@pytest.mark.parametrize("wl", _workloads(), ids=lambda w: w.name)
def test_index_matches_oracle(lib, wl):
    e = _plan(lib, wl).export()
    paths = ot.query_paths(wl.parent, wl.query_node)
    want_ptr = np.cumsum([0] + [len(p) for p in paths])
    assert np.array_equal(e["qpath_ptr"], want_ptr)
    assert np.array_equal(e["qpath_node"], np.concatenate([np.array(p, np.int32) for p in paths]))
    nq = ot.node_queries(wl.parent, wl.query_node, wl.n_nodes)
    assert np.array_equal(e["nodeq_ptr"], np.cumsum([0] + [len(x) for x in nq]))
    assert np.array_equal(e["nodeq"], np.array([q for x in nq for q in x], np.int32))


def _covered_pairs(wl, e):
    """Multiset of (query, node, token) the plan's chunks cover, as int64 codes."""
    codes = []
    tok_base = np.zeros(wl.n_nodes + 1, np.int64)
    tok_base[1:] = np.cumsum(wl.node_len.astype(np.int64))
    total = int(tok_base[-1])
    for c in range(len(e["chunk_q_ptr"]) - 1):
        qs = e["chunk_q"][e["chunk_q_ptr"][c]:e["chunk_q_ptr"][c + 1]].astype(np.int64)
        masks = e["chunk_q_mask"][e["chunk_q_ptr"][c]:e["chunk_q_ptr"][c + 1]]
        nodes = e["chunk_tok_node"][e["chunk_tok_ptr"][c]:e["chunk_tok_ptr"][c + 1]]
        ts = e["chunk_tok_t"][e["chunk_tok_ptr"][c]:e["chunk_tok_ptr"][c + 1]]
        gid = tok_base[nodes] + ts
        j = np.arange(len(gid))
        for q, m in zip(qs, masks):
            if m == np.uint64(0xFFFFFFFFFFFFFFFF):
                vis = np.ones(len(gid), bool)
            else:
                vis = ((np.uint64(m) >> j.astype(np.uint64)) & np.uint64(1)).astype(bool) if len(j) <= 64 else None
                assert vis is not None, "masked chunk longer than 64 tokens"
            codes.append(q * total + gid[vis])
    return np.sort(np.concatenate(codes)) if codes else np.zeros(0, np.int64)


def _visible_pairs(wl):
    tok_base = np.zeros(wl.n_nodes + 1, np.int64)
    tok_base[1:] = np.cumsum(wl.node_len.astype(np.int64))
    total = int(tok_base[-1])
    codes = []
    for q, path in enumerate(ot.query_paths(wl.parent, wl.query_node)):
        for n in path:
            codes.append(q * total + tok_base[n] + np.arange(int(wl.node_len[n]), dtype=np.int64))
    return np.sort(np.concatenate(codes))


_POLICIES = {"cost_model": {}, "none": {}, "uniform": {"fixed_chunk": 128}, "flatten": {},
             "flatten16": {"split_policy": "flatten", "fixed_chunk": 16},
             "flatten300": {"split_policy": "flatten", "fixed_chunk": 300}}


@pytest.mark.parametrize("policy", list(_POLICIES))
@pytest.mark.parametrize("wl", _workloads(), ids=lambda w: w.name)
def test_plan_covers_each_pair_exactly_once(lib, wl, policy):
    kw = {"split_policy": policy, **_POLICIES[policy]}
    e = _plan(lib, wl, **kw).export()
    got = _covered_pairs(wl, e)
    want = _visible_pairs(wl)
    assert got.shape == want.shape
    assert np.array_equal(got, want)            # same multiset: nothing missing, nothing twice
    # the merge list of each query names one partial row per chunk that contains it
    for q in range(wl.n_queries):
        rows = e["merge_row"][e["merge_ptr"][q]:e["merge_ptr"][q + 1]]
        assert len(rows) == len(set(rows.tolist()))
        n_chunks_with_q = sum(q in set(e["chunk_q"][e["chunk_q_ptr"][c]:e["chunk_q_ptr"][c + 1]].tolist())
                              for c in range(len(e["chunk_q_ptr"]) - 1))
        assert len(rows) == n_chunks_with_q


def _chunks(e):
    """Per chunk: (tokens as (node, t) pairs, queries, masks)."""
    out = []
    for c in range(len(e["chunk_q_ptr"]) - 1):
        a, b = e["chunk_tok_ptr"][c], e["chunk_tok_ptr"][c + 1]
        qa, qb = e["chunk_q_ptr"][c], e["chunk_q_ptr"][c + 1]
        out.append((list(zip(e["chunk_tok_node"][a:b].tolist(), e["chunk_tok_t"][a:b].tolist())),
                    e["chunk_q"][qa:qb].tolist(), [int(m) for m in e["chunk_q_mask"][qa:qb]]))
    return out


def test_deft_flatten_chunks_of_a_hand_laid_tree(lib):
    """DEFT-Flatten (DEFT, A.9) on a tree whose page layout is written out:
    root 40 tokens in pages 0, 1, 2 (rows 0-7 of page 2); child 1 (20 tokens)
    continues in page 2 at row 8 and ends in page 3; child 2 (20 tokens)
    starts a fresh page 4. Query 0 sits on child 1, query 1 on child 2.
    Depth-first, the root and child 1 are consecutive page rows and child 2
    is not, so with S_t = 64 the chunks are [root + child 1] (60 tokens,
    masked: query 1 sees only the root's 40) and [child 2]; with S_t = 32 the
    root's first 32 tokens form a chunk of their own (one node: no mask),
    then [root tokens 32-39 + child 1] (28 tokens, query 1 sees 8) and
    [child 2]."""
    all_ones = 2**64 - 1
    tree = lib.tree_build([40, 20, 20], [-1, 0, 0], [0, 3, 5, 7], [0, 1, 2, 2, 3, 4, 5], first_offset=[0, 8, 0],
                          page_size=16, num_pages=6)
    def plan(st):
        return _chunks(lib.plan_create(tree, [1, 2], 8, 2, 128, "bf16", num_sms=152, split_policy="flatten",
                                       fixed_chunk=st).export())
    root = [(0, t) for t in range(40)]
    c1 = [(1, t) for t in range(20)]
    c2 = [(2, t) for t in range(20)]
    assert plan(64) == [(root + c1, [0, 1], [(1 << 60) - 1, (1 << 40) - 1]), (c2, [1], [all_ones])]
    assert plan(32) == [(root[:32], [0, 1], [all_ones, all_ones]),
                        (root[32:] + c1, [0, 1], [(1 << 28) - 1, (1 << 8) - 1]),
                        (c2, [1], [all_ones])]


def _same_export(a, b):
    return a.keys() == b.keys() and all(np.array_equal(a[k], b[k]) for k in a)


# (the flattened control of document QA on 148 SMs is a case the flattened
# chunking wins under the measured tables)
@pytest.mark.parametrize("make,sms", [(lambda: synth.tree_of_thought("gqa"), 152), (synth.document_qa, 152),
                                      (synth.few_shot, 152), (synth.speculative, 152),
                                      (lambda: synth.random_tree(1007), 152),
                                      (lambda: synth.flat_control(synth.document_qa()), 148)],
                         ids=["tot_gqa", "document_qa", "few_shot", "speculative", "random", "document_qa_flat"])
def test_cost_model_scores_flatten_candidates(lib, make, sms):
    """The cost-model policy also scores DEFT-Flatten chunkings of 1024 and
    2048 tokens and keeps one only when its predicted makespan is at least
    3 % below the node partition's; switched off, the node partition stays.
    The rule is checked against plans built separately (whichever way the
    measured cost tables decide it for this workload), and the plan kept is
    the separately built one, array for array."""
    wl = make()
    node_plan = _plan(lib, wl, flatten_candidates=False, num_sms=sms)
    node = node_plan.stats()
    assert node["split_policy"] == 0
    flat_plans = {st: _plan(lib, wl, split_policy="flatten", fixed_chunk=st, num_sms=sms) for st in (1024, 2048)}
    flat = {st: p.stats()["predicted_makespan_us"] for st, p in flat_plans.items()}
    chosen_plan = _plan(lib, wl, num_sms=sms)
    chosen = chosen_plan.stats()
    best_st = min(flat, key=lambda st: (flat[st], st))
    if flat[best_st] < 0.97 * node["predicted_makespan_us"]:
        assert chosen["split_policy"] == 3 and chosen["fixed_chunk"] == best_st
        assert chosen["predicted_makespan_us"] == flat[best_st]
        assert _same_export(chosen_plan.export(), flat_plans[best_st].export())
    else:
        assert chosen["split_policy"] == 0
        assert chosen["predicted_makespan_us"] == node["predicted_makespan_us"]
        assert _same_export(chosen_plan.export(), node_plan.export())


def test_flatten_wins_somewhere(lib):
    """The flattened winner is reachable (so the test above can check it):
    under the measured tables some no-sharing control flattens on some SM
    count (the 148-SM document-QA control is the case the test above uses)."""
    wins = []
    for make in (lambda: synth.flat_control(synth.document_qa()), lambda: synth.flat_control(synth.speculative())):
        wl = make()
        for sms in (148, 64, 8):
            wins.append(_plan(lib, wl, num_sms=sms).stats()["split_policy"] == 3)
    assert any(wins)


def test_speculative_drafts_are_packed_with_masks(lib):
    wl = synth.speculative()
    e = _plan(lib, wl).export()
    n_chunks = len(e["chunk_q_ptr"]) - 1
    masked = [c for c in range(n_chunks)
              if np.any(e["chunk_q_mask"][e["chunk_q_ptr"][c]:e["chunk_q_ptr"][c + 1]] != np.uint64(2**64 - 1))]
    assert len(masked) == 8                     # one 64-token draft chunk per tree
    for c in masked:
        assert e["chunk_tok_ptr"][c + 1] - e["chunk_tok_ptr"][c] == 64
        assert e["chunk_q_ptr"][c + 1] - e["chunk_q_ptr"][c] == 64
        assert e["chunk_kind"][c] == 1          # 64 queries x 4 = 256 rows: tensor cores


def test_kernel_choice_by_rows(lib):
    wl = synth.document_qa()
    e = _plan(lib, wl).export()
    for c in range(len(e["chunk_q_ptr"]) - 1):
        nq = e["chunk_q_ptr"][c + 1] - e["chunk_q_ptr"][c]
        assert e["chunk_kind"][c] == (1 if nq * 4 >= 16 else 0)
    e1 = _plan(lib, synth.tiny_two_level()).export()
    assert not np.any(e1["chunk_kind"])         # fp32 never runs on tensor cores


def test_planner_never_worse_than_fixed_splits(lib):
    for wl in (synth.document_qa(), synth.few_shot(), synth.tree_of_thought("gqa"), synth.speculative()):
        best = _plan(lib, wl).stats()["predicted_makespan_us"]
        others = [_plan(lib, wl, split_policy="none").stats()["predicted_makespan_us"]]
        for ch in (256, 1024, 4096):
            others.append(_plan(lib, wl, split_policy="uniform", fixed_chunk=ch).stats()["predicted_makespan_us"])
        assert best <= min(others) * (1 + 1e-9)


def test_cost_table_interpolation(lib):
    rows = [1, 4, 16, 256]
    toks = [64, 1024, 16384]
    us = np.array([[1, 2, 20], [1.5, 3, 30], [2, 4, 40], [4, 8, 80]], np.float32)
    lib.cost_set_table(1, rows, toks, us)
    try:
        assert abs(lib.cost_estimate(1, 16, 1024) - 4.0) < 1e-5
        assert abs(lib.cost_estimate(1, 4, 1024) - 3.0) < 1e-5
        mid = lib.cost_estimate(1, 8, 1024)       # halfway in log rows
        assert abs(mid - 3.5) < 1e-4
        assert abs(lib.cost_estimate(1, 1000, 16384) - 80) < 1e-4     # rows clamped to the grid
        assert abs(lib.cost_estimate(1, 256, 32768) - 160) < 1e-3     # linear in tokens past the grid
        assert abs(lib.cost_estimate(1, 1, 10) - 1.0) < 1e-5          # clamped below the grid
        lib.cost_set_table(2, rows, toks, us * 2)
        assert abs(lib.cost_estimate(2, 16, 1024) - 8.0) < 1e-5       # kinds are independent
        assert abs(lib.cost_estimate(1, 16, 1024) - 4.0) < 1e-5
        assert lib.cost_estimate(4, 16, 1024) == -1.0
        assert lib.cost_estimate(3, 16, 1024) > 0.0                   # the thin PAC's model
    finally:
        lib.cost_set_table(1, "builtin", None, None)
        lib.cost_set_table(2, "builtin", None, None)


# ------------------------------------------------------------ incremental plan (next decode step)

def _chunks_per_node(e, n_nodes):
    cnt = np.zeros(n_nodes, np.int64)
    for c in range(len(e["chunk_q_ptr"]) - 1):
        nodes = set(e["chunk_tok_node"][e["chunk_tok_ptr"][c]:e["chunk_tok_ptr"][c + 1]].tolist())
        if len(nodes) == 1:
            cnt[nodes.pop()] += 1
    return cnt


@pytest.mark.parametrize("wl", [synth.few_shot(), synth.document_qa()] +
                         [synth.random_tree(8600 + s, max_nodes=12, max_len=150, heads=(8, 2), d=128,
                                            dtype="bf16", n_queries=12) for s in range(6)],
                         ids=lambda w: w.name)
def test_plan_update_keeps_splits_and_covers(lib, wl):
    """The next step's plan (query nodes one token longer) covers every
    (query, token) pair of the grown tree exactly once and keeps each node's
    KV-axis split."""
    p = _plan(lib, wl)
    wl2 = synth.grow_query_nodes(wl, 1)
    p2 = lib.plan_update(p, _tree(lib, wl2))
    e, e2 = p.export(), p2.export()
    assert np.array_equal(_covered_pairs(wl2, e2), _visible_pairs(wl2))
    c1, c2 = _chunks_per_node(e, wl.n_nodes), _chunks_per_node(e2, wl.n_nodes)
    grown = np.zeros(wl.n_nodes, bool)
    grown[np.unique(wl.query_node)] = True
    # nodes that did not grow are cut exactly as before; grown ones keep their split
    # unless one more token needs a new tile boundary (never fewer chunks)
    assert np.array_equal(c1[~grown], c2[~grown])
    assert np.all(c2[grown] >= c1[grown])
    assert p2.stats()["n_chunks"] >= p.stats()["n_chunks"]


def test_plan_update_skips_the_partition_search(lib):
    wl = synth.tree_of_thought("gqa")
    p = _plan(lib, wl)
    p2 = lib.plan_update(p, _tree(lib, synth.grow_query_nodes(wl, 1)))
    assert p2.stats()["plan_us"] < p.stats()["plan_us"]
    assert abs(p2.stats()["cost_lower_bound_us"] - p.stats()["cost_lower_bound_us"]) < 1e-9


def test_plan_update_rejects_a_changed_shape(lib):
    wl = synth.random_tree(8603, max_nodes=12, max_len=150, heads=(8, 2), d=128, dtype="bf16", n_queries=12)
    p = _plan(lib, wl)
    t_small = lib.tree_build([5], [-1], [0, 1], [0], num_pages=1)
    with pytest.raises(lib.PstError) as e:
        lib.plan_update(p, t_small)
    assert e.value.code == -1
    # re-hang a queried node elsewhere: the paths change
    q0 = int(wl.query_node[0])
    parent = wl.parent.copy()
    parent[q0] = -1 if parent[q0] >= 0 else (0 if q0 != 0 else 1)
    t_moved = lib.tree_build(wl.node_len, parent, wl.page_ptr, wl.page_ids, wl.first_offset, wl.page_size,
                             wl.num_pages)
    with pytest.raises(lib.PstError) as e:
        lib.plan_update(p, t_moved)
    assert e.value.code == -1


# ------------------------------------------------------------ thin-chunk engine selection

def _thin_item_count(wl, e, thin):
    G = wl.n_q_heads // wl.n_kv_heads
    n = 0
    for c in range(len(e["chunk_q_ptr"]) - 1):
        if e["chunk_kind"][c] != 0:
            continue
        rows = int(e["chunk_q_ptr"][c + 1] - e["chunk_q_ptr"][c]) * G
        if thin:
            rb = 4 if rows <= 4 else 8
            n += -(-rows // rb) * (wl.n_kv_heads // 8)
        else:
            rt = 1 if rows <= 1 else 2 if rows <= 2 else 4 if rows <= 4 else 8
            n += -(-rows // rt) * wl.n_kv_heads
    return n


@pytest.mark.parametrize("case", ["bf16_d128_hkv8", "cuda_core_engine", "d64", "f32", "hkv2"])
def test_thin_engine_selection_and_items(lib, case):
    """Thin chunks take the tcgen05 thin PAC (items of 8 kv heads, row blocks of
    4 or 8) for bf16, d = 128 and Hkv a multiple of 8, else the CUDA-core PAC
    (one item per kv head and row tile)."""
    heads, d, dtype, opts = (32, 8), 128, "bf16", {}
    if case == "cuda_core_engine":
        opts = dict(thin_engine="cuda_core")
    elif case == "d64":
        d = 64
    elif case == "f32":
        dtype = "f32"
    elif case == "hkv2":
        heads = (8, 2)
    wl = synth.random_tree(8620, max_nodes=14, max_len=200, heads=heads, d=d, dtype=dtype, n_queries=10)
    p = _plan(lib, wl, **opts)
    e = p.export()
    thin = case == "bf16_d128_hkv8"
    assert p.stats()["n_cc_items"] == _thin_item_count(wl, e, thin)
    assert np.array_equal(_covered_pairs(wl, e), _visible_pairs(wl))


def test_thin_chunks_start_on_page_row_boxes(lib):
    """The thin PAC's tiles are 16-row page boxes: a thin chunk that does not
    start its node starts on a multiple of 16 in page space."""
    for s in range(6):
        wl = synth.random_tree(8630 + s, max_nodes=14, max_len=400, heads=(32, 8), d=128, dtype="bf16",
                               n_queries=10)
        e = _plan(lib, wl, split_policy="uniform", fixed_chunk=64).export()
        for c in range(len(e["chunk_q_ptr"]) - 1):
            if e["chunk_kind"][c] != 0:
                continue
            n0 = int(e["chunk_tok_node"][e["chunk_tok_ptr"][c]])
            t0 = int(e["chunk_tok_t"][e["chunk_tok_ptr"][c]])
            if t0 > 0:
                assert (int(wl.first_offset[n0]) + t0) % 16 == 0


def test_grow_query_nodes_input():
    """The grown-tree generator keeps every existing row and adds k new tokens
    to each node a query sits on, in free rows."""
    wl = synth.random_tree(8605, max_nodes=12, max_len=150, heads=(8, 2), d=128, dtype="bf16", n_queries=12)
    w2 = synth.grow_query_nodes(wl, 3)
    q_nodes = np.unique(wl.query_node)
    want = wl.node_len.astype(np.int64).copy()
    want[q_nodes] += 3
    assert np.array_equal(w2.node_len, want)
    r1, r2 = wl.row_lids(), w2.row_lids()
    assert np.array_equal(r2[:r1.size][r1 >= 0], r1[r1 >= 0])
    assert (r2 >= 0).sum() == (r1 >= 0).sum() + 3 * q_nodes.size
    assert len(np.unique(r2[r2 >= 0])) == (r2 >= 0).sum()


# ------------------------------------------------------------ plan update across a changed tree shape

@pytest.mark.parametrize("seed", [3, 11])
def test_plan_update_tree_after_accept_and_prune(lib, seed):
    """Speculative decoding, next step: in each tree one draft path is
    accepted (kept as a chain under the prompt), the rest pruned, and a new
    64-node draft tree with new queries hangs off the last accepted draft. The
    updated plan covers every (query, token) pair of the new tree exactly once,
    its index equals the oracle's, the prompts keep their KV-axis split and the
    new drafts are packed with bit causal masks."""
    wl = synth.speculative(batch=3, prompt=2000)
    p = _plan(lib, wl)
    wl2, prev_node = synth.speculative_next_step(wl, seed)
    p2 = lib.plan_update_tree(p, _tree(lib, wl2), wl2.query_node, prev_node)
    e, e2 = p.export(), p2.export()
    assert np.array_equal(_covered_pairs(wl2, e2), _visible_pairs(wl2))
    # the index (query -> path, node -> queries) is the oracle's
    paths = ot.query_paths(wl2.parent, wl2.query_node)
    for q, path in enumerate(paths):
        assert e2["qpath_node"][e2["qpath_ptr"][q]:e2["qpath_ptr"][q + 1]].tolist() == path
    nq = ot.node_queries(wl2.parent, wl2.query_node, wl2.n_nodes)
    for n in range(wl2.n_nodes):
        assert e2["nodeq"][e2["nodeq_ptr"][n]:e2["nodeq_ptr"][n + 1]].tolist() == nq[n]
    # kept prompts: split as before
    c1, c2 = _chunks_per_node(e, wl.n_nodes), _chunks_per_node(e2, wl2.n_nodes)
    for n in range(wl2.n_nodes):
        if prev_node[n] >= 0 and wl2.parent[n] < 0:
            assert c2[n] == c1[prev_node[n]], (n, c2[n], c1[prev_node[n]])
    # the new drafts are packed: some chunk of the new plan carries masks
    masks = e2["chunk_q_mask"]
    assert np.any(masks != np.uint64(0xFFFFFFFFFFFFFFFF))
    assert p2.stats()["plan_us"] < p.stats()["plan_us"] * 4


def test_plan_update_tree_rejects_a_bad_node_map(lib):
    wl = synth.speculative(batch=2, prompt=500)
    p = _plan(lib, wl)
    wl2, prev_node = synth.speculative_next_step(wl, 5)
    t2 = _tree(lib, wl2)
    bad = prev_node.copy()
    bad[0] = wl.n_nodes          # no such node in the previous tree
    with pytest.raises(lib.PstError):
        lib.plan_update_tree(p, t2, wl2.query_node, bad)
    with pytest.raises(ValueError):
        lib.plan_update_tree(p, t2, wl2.query_node, prev_node[:-1])
