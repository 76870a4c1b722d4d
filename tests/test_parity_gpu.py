"""GPU parity: libpst's CUDA path against the fp64 oracle, element by element.

Tolerances (fp32 output, bf16 or fp32 inputs): every |O - O_ref| <= 2e-3,
per (query, head) row max|O - O_ref| / max(max|O_ref|, 1e-6) <= 1e-2, and
|LSE - LSE_ref| <= 1e-3 (natural log)."""
import numpy as np
import pytest

import synth
from oracle import attention as oa

pytestmark = pytest.mark.gpu

ABS_TOL, REL_TOL, LSE_TOL = 2e-3, 1e-2, 1e-3


def run_gpu(lib, wl, pools=None, Q=None, **opts):
    import torch
    from prefix_shared_tree_gb300.torch_api import TreeDecodeAttention, to_device
    K, V = wl.kv_pools() if pools is None else pools
    Q = wl.q() if Q is None else Q
    att = TreeDecodeAttention.from_workload(wl, **opts)
    Qd, Kd, Vd = to_device(Q, wl.dtype), to_device(K, wl.dtype), to_device(V, wl.dtype)
    O, L = att(Qd, Kd, Vd)
    torch.cuda.synchronize()
    assert att.check_status() == 0
    O2, L2 = att(Qd, Kd, Vd)
    torch.cuda.synchronize()
    assert torch.equal(O, O2) and torch.equal(L, L2), "repeated calls differ"
    return O.cpu().numpy(), L.cpu().numpy(), (K, V, Q), att


_ORACLE_CACHE = {}


def full_size(name):
    """A full-size workload with its pools, queries and oracle outputs (all
    queries), computed once per test session."""
    if name not in _ORACLE_CACHE:
        wl = {"document_qa": synth.document_qa, "speculative": synth.speculative,
              "few_shot": synth.few_shot}.get(name) or (lambda: synth.tree_of_thought(name.split("_")[-1]))
        wl = wl()
        K, V = wl.kv_pools()
        Q = wl.q()
        _ORACLE_CACHE.clear()   # one full-size workload in host memory at a time
        _ORACLE_CACHE[name] = (wl, K, V, Q, oa.decode_attention(wl, K, V, Q))
    return _ORACLE_CACHE[name]


def assert_matches(wl, O, L, K, V, Q, queries=None, ref=None):
    qs = list(range(wl.n_queries)) if queries is None else list(queries)
    Oref, Lref = oa.decode_attention(wl, K, V, Q, qs) if ref is None else ref
    for q in qs:
        o = O[q].astype(np.float64)
        r = Oref[q]
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(L[q]))
        err = np.abs(o - r)
        assert err.max() <= ABS_TOL, f"query {q}: max abs {err.max():.3e}"
        rel = err.max(axis=1) / np.maximum(np.abs(r).max(axis=1), 1e-6)
        assert rel.max() <= REL_TOL, f"query {q}: row rel {rel.max():.3e}"
        le = np.abs(L[q].astype(np.float64) - Lref[q])
        assert le.max() <= LSE_TOL, f"query {q}: lse {le.max():.3e}"


def test_tiny_two_level_fp32(lib):
    wl = synth.tiny_two_level()
    O, L, (K, V, Q), _ = run_gpu(lib, wl)
    assert_matches(wl, O, L, K, V, Q)


RANDOM_CASES = []
for s in range(48):
    heads = [(4, 2), (8, 1), (32, 8), (4, 4), (2, 1), (16, 16)][s % 6]
    d = (64, 128)[(s // 6) % 2]
    dtype = ("bf16", "bf16", "f32")[(s // 12) % 3]
    RANDOM_CASES.append((s, heads, d, dtype))


@pytest.mark.parametrize("seed,heads,d,dtype", RANDOM_CASES)
def test_random_trees(lib, seed, heads, d, dtype):
    wl = synth.random_tree(7000 + seed, max_nodes=14, max_len=150, heads=heads, d=d, dtype=dtype,
                           n_queries=None)
    O, L, (K, V, Q), _ = run_gpu(lib, wl)
    assert_matches(wl, O, L, K, V, Q)


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("opts", [dict(tc_min_rows=1), dict(split_policy="uniform", fixed_chunk=64),
                                  dict(split_policy="none"), dict(pack_masks=False),
                                  dict(tc_min_rows=1, tc_engine="mma_sync"), dict(thin_engine="cuda_core"),
                                  dict(tc_min_rows=17, split_policy="uniform", fixed_chunk=128),
                                  dict(split_policy="flatten"), dict(split_policy="flatten", fixed_chunk=200)],
                         ids=["all_tensor_core", "uniform64", "no_split", "no_masks", "mma_sync", "cuda_core_thin",
                              "thin_uniform128", "flatten64", "flatten200"])
def test_random_trees_plan_variants(lib, seed, opts):
    wl = synth.random_tree(8000 + seed, max_nodes=12, max_len=300, heads=(8, 2), d=128, dtype="bf16",
                           n_queries=24)
    O, L, (K, V, Q), _ = run_gpu(lib, wl, **opts)
    assert_matches(wl, O, L, K, V, Q)


THIN_CASES = [(8500 + s, h, 400, 6 + s) for s, h in
              enumerate([(16, 1), (8, 1), (32, 2), (4, 1), (16, 2), (2, 2), (1, 1), (6, 2)])]
THIN_CASES += [(8607, (4, 1), 40, 10), (8607, (8, 2), 40, 10), (8694, (4, 1), 40, 10)]   # packed masked chunks


@pytest.mark.parametrize("seed,heads,max_len,n_queries", THIN_CASES)
def test_thin_pac_up_to_16_rows(lib, seed, heads, max_len, n_queries):
    """Thin chunks of 1 to 16 rows (tc_min_rows=17) on the tcgen05 thin PAC:
    GQA groups of 1-16, single-token and ragged nodes, packed masked chunks."""
    wl = synth.random_tree(seed, max_nodes=14, max_len=max_len, heads=heads, d=128, dtype="bf16",
                           n_queries=n_queries)
    O, L, (K, V, Q), att = run_gpu(lib, wl, tc_min_rows=17)
    assert att.plan.stats()["n_cc_items"] > 0
    assert_matches(wl, O, L, K, V, Q)


@pytest.mark.parametrize("name", ["speculative", "tree_of_thought_gqa"])
def test_thin_pac_many_row_blocks(lib, name):
    """Every chunk on the thin PAC (tc_min_rows above any row count): chunks
    of up to 1024 rows in blocks of 16, DEFT's masked draft chunks; every
    query compared with the oracle."""
    wl, K, V, Q, ref = full_size(name)
    O, L, _, att = run_gpu(lib, wl, pools=(K, V), Q=Q, tc_min_rows=1 << 20)
    assert att.plan.stats()["n_tc_items"] == 0
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    assert_matches(wl, O, L, K, V, Q, ref=ref)


@pytest.mark.parametrize("name", ["few_shot", "random_a", "random_b"])
def test_plan_update_next_step(lib, name):
    """Two decode steps: the plan of step 2 (every query node one token longer,
    new pages appended to the pool) comes from pst_plan_update on step 1's plan."""
    import torch
    from prefix_shared_tree_gb300.torch_api import TreeDecodeAttention, to_device
    wl = synth.few_shot() if name == "few_shot" else synth.random_tree(
        8600 + (name == "random_b"), max_nodes=12, max_len=150, heads=(8, 2), d=128, dtype="bf16", n_queries=12)
    att = TreeDecodeAttention.from_workload(wl)
    K, V = wl.kv_pools()
    Q = wl.q()
    O, L = att(to_device(Q, wl.dtype), to_device(K, wl.dtype), to_device(V, wl.dtype))
    torch.cuda.synchronize()
    assert_matches(wl, O.cpu().numpy(), L.cpu().numpy(), K, V, Q, queries=range(min(wl.n_queries, 8)))
    wl2 = synth.grow_query_nodes(wl, 1)
    att.update_tree(wl2.node_len, wl2.parent, wl2.page_ptr, wl2.page_ids, wl2.first_offset, wl2.num_pages)
    K2, V2 = wl2.kv_pools()
    Q2 = wl2.q()
    O2, L2 = att(to_device(Q2, wl2.dtype), to_device(K2, wl2.dtype), to_device(V2, wl2.dtype))
    torch.cuda.synchronize()
    assert att.check_status() == 0
    assert_matches(wl2, O2.cpu().numpy(), L2.cpu().numpy(), K2, V2, Q2)


@pytest.mark.parametrize("seed", [3, 11])
def test_plan_update_tree_speculative_two_steps(lib, seed):
    """Two speculative decoding steps: after step 1 one draft path per tree is
    accepted, the other drafts are pruned and a new draft tree (new queries)
    grows; step 2's plan comes from pst_plan_update_tree on step 1's plan."""
    import torch
    from prefix_shared_tree_gb300.torch_api import TreeDecodeAttention, to_device
    wl = synth.speculative(batch=4, prompt=3000)
    att = TreeDecodeAttention.from_workload(wl)
    K, V = wl.kv_pools()
    Q = wl.q()
    O, L = att(to_device(Q, wl.dtype), to_device(K, wl.dtype), to_device(V, wl.dtype))
    torch.cuda.synchronize()
    assert_matches(wl, O.cpu().numpy(), L.cpu().numpy(), K, V, Q, queries=range(0, wl.n_queries, 9))
    wl2, prev_node = synth.speculative_next_step(wl, seed)
    att.update_shape(wl2.node_len, wl2.parent, wl2.page_ptr, wl2.page_ids, wl2.first_offset, wl2.num_pages,
                     wl2.query_node, prev_node)
    K2, V2 = wl2.kv_pools()
    Q2 = wl2.q()
    O2, L2 = att(to_device(Q2, wl2.dtype), to_device(K2, wl2.dtype), to_device(V2, wl2.dtype))
    torch.cuda.synchronize()
    assert att.check_status() == 0
    assert_matches(wl2, O2.cpu().numpy(), L2.cpu().numpy(), K2, V2, Q2)


@pytest.mark.parametrize("name", ["few_shot", "speculative", "tiny"])
def test_cuda_graph_replay_equals_direct_call(lib, name):
    """A decode step captured as a CUDA graph (forked launch groups, join,
    POR) and replayed gives the direct call's outputs bit for bit, also after
    new queries are copied into the captured input tensor."""
    import torch
    from prefix_shared_tree_gb300.torch_api import TreeDecodeAttention, to_device
    wl = {"few_shot": synth.few_shot, "speculative": lambda: synth.speculative(batch=3, prompt=2500),
          "tiny": synth.tiny_two_level}[name]()
    att = TreeDecodeAttention.from_workload(wl)
    K, V = wl.kv_pools()
    Q = wl.q()
    Qd, Kd, Vd = to_device(Q, wl.dtype), to_device(K, wl.dtype), to_device(V, wl.dtype)
    O_ref, L_ref = att(Qd, Kd, Vd)
    O = torch.full_like(O_ref, float("nan"))
    L = torch.full_like(L_ref, float("nan"))
    g = att.capture(Qd, Kd, Vd, O, L)
    for _ in range(2):
        O.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(O, O_ref) and torch.equal(L, L_ref)
    # new queries through the same graph
    Q2 = np.roll(Q, 1, axis=0)
    Qd.copy_(to_device(Q2, wl.dtype))
    g.replay()
    torch.cuda.synchronize()
    assert att.check_status() == 0
    assert_matches(wl, O.cpu().numpy(), L.cpu().numpy(), K, V, Q2, queries=range(0, wl.n_queries, 5))


@pytest.mark.parametrize("case", ["few_shot", "random_bf16_all_groups", "random_fp32_cuda_core", "mma_sync"])
def test_launch_modes_give_identical_outputs(lib, case):
    """The PAC launch groups chained on one stream (each launch after the
    first with a programmatic dependency on the one before: the default) and
    on forked side streams joined before POR give the same outputs bit for
    bit; the side-stream outputs also match the oracle."""
    if case == "few_shot":
        wl, opts = synth.few_shot(), {}
    elif case == "random_bf16_all_groups":
        # five PAC launches: tensor-core groups with P rounded once and exact,
        # above and below 128 rows per block, and the thin PAC
        wl = synth.random_tree(5189, max_nodes=16, max_len=1500, heads=(32, 8), d=128, dtype="bf16", n_queries=48)
        opts = {"p_bf16_min_tokens": 256}
    elif case == "random_fp32_cuda_core":
        wl = synth.random_tree(5151, max_nodes=12, max_len=200, heads=(8, 2), d=64, dtype="f32", n_queries=24)
        opts = {}
    else:
        wl = synth.random_tree(5152, max_nodes=12, max_len=200, heads=(16, 4), d=128, dtype="bf16", n_queries=24)
        opts = {"tc_engine": "mma_sync", "tc_min_rows": 1}
    O1, L1, (K, V, Q), att1 = run_gpu(lib, wl, **opts)
    O2, L2, _, att2 = run_gpu(lib, wl, pools=(K, V), Q=Q, side_streams=True, **opts)
    assert att1.plan.stats()["n_launches"] == att2.plan.stats()["n_launches"]
    assert np.array_equal(O1.view(np.uint32), O2.view(np.uint32))
    assert np.array_equal(L1.view(np.uint32), L2.view(np.uint32))
    qs = range(0, wl.n_queries, 7) if case == "few_shot" else None
    assert_matches(wl, O2, L2, K, V, Q, queries=qs)


def test_non_finite_junk_in_unused_page_rows(lib):
    """Rows of a page that no node covers may hold NaN; they never reach O."""
    for seed in range(6):
        wl = synth.random_tree(9100 + seed, max_nodes=10, max_len=90, heads=(8, 2), d=128, dtype="bf16",
                               n_queries=20)
        K, V = wl.kv_pools()
        unused = (wl.row_lids() < 0).reshape(wl.num_pages, wl.page_size)
        K[np.broadcast_to(unused[:, None, :, None], K.shape)] = 0x7FC0
        V[np.broadcast_to(unused[:, None, :, None], V.shape)] = 0x7FC0
        for opts in ({}, {"tc_min_rows": 1}):
            O, L, _, _ = run_gpu(lib, wl, pools=(K, V), **opts)
            assert_matches(wl, O, L, K, V, wl.q())


def test_few_shot_full(lib):
    wl, K, V, Q, ref = full_size("few_shot")
    O, L, _, att = run_gpu(lib, wl, pools=(K, V), Q=Q)
    assert_matches(wl, O, L, K, V, Q, ref=ref)
    st = att.plan.stats()
    assert st["n_tc_items"] > 0 and st["n_cc_items"] > 0


_FLATTEN = {"split_policy": "flatten"}


@pytest.mark.parametrize("name,opts", [
    ("document_qa", {}), ("speculative", {}), ("speculative", _FLATTEN),
    ("speculative", dict(_FLATTEN, fixed_chunk=1024)), ("tree_of_thought_gqa", {}),
    ("tree_of_thought_gqa", dict(_FLATTEN, fixed_chunk=256)), ("tree_of_thought_mqa", {}),
    ("tree_of_thought_mha", {})],
    ids=["document_qa", "speculative", "speculative-flatten64", "speculative-flatten1024", "tree_of_thought_gqa",
         "tree_of_thought_gqa-flatten256", "tree_of_thought_mqa", "tree_of_thought_mha"])
def test_full_size_every_query(lib, name, opts):
    """The full-size workloads with the default plan (and DEFT-Flatten
    chunking for the trees of many small nodes), every query and head
    compared with the oracle."""
    wl, K, V, Q, ref = full_size(name)
    O, L, _, att = run_gpu(lib, wl, pools=(K, V), Q=Q, **opts)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(L))
    assert_matches(wl, O, L, K, V, Q, ref=ref)


def test_flat_control_matches_shared(lib):
    """The no-sharing flat control (copied pages) computes the same outputs."""
    wl = synth.few_shot()
    O, L, (K, V, Q), _ = run_gpu(lib, wl)
    fl = synth.flat_control(wl)
    Of, Lf, (Kf, Vf, Qf), att = run_gpu(lib, fl)
    assert np.array_equal(Qf, Q)
    assert np.abs(Of - O).max() <= 2 * ABS_TOL and np.abs(Lf - L).max() <= 2 * LSE_TOL
    assert_matches(fl, Of, Lf, Kf, Vf, Qf, queries=[0, 31, 63])


def _boosted_prefix(prefix, n_req, boost_from):
    """A document-QA tree whose root tokens from `boost_from` on carry a large
    key component that only the even-numbered queries see: their running max
    jumps by ~33 (log2 units) in the middle of the root chunk while the odd
    queries' does not, so the lazy O rescale runs on some rows of a warp and
    not on the others."""
    wl = synth.document_qa(prefix=prefix, n_req=n_req)
    K, V = wl.kv_pools()
    Q = wl.q()
    lids = wl.row_lids().reshape(wl.num_pages, wl.page_size)
    boosted = np.isin(lids, wl.lid[wl.lid_ptr[0] + boost_from:wl.lid_ptr[1]])
    bf16_16 = 0x4180                       # 16.0 in bf16
    k0 = K[..., 0]
    k0[np.broadcast_to(boosted[:, None, :], k0.shape)] = bf16_16
    Q[0::2, :, 0] = bf16_16                # score += 16 * 16 / sqrt(128) on boosted tokens
    return wl, K, V, Q


@pytest.mark.parametrize("prefix,n_req,boost,opts", [
    (2048, 64, 1024, {"split_policy": "none"}),   # 256 rows in two halves, P rounded once
    (2048, 16, 1024, {"split_policy": "none"}),   # 64 rows, alternate tiles per softmax group
    (768, 64, 384, {"split_policy": "none"}),     # short chunk: P split into hi + lo
    (2048, 64, 1024, {}),
])
def test_lazy_rescale_on_some_rows(lib, prefix, n_req, boost, opts):
    wl, K, V, Q = _boosted_prefix(prefix, n_req, boost)
    O, L, _, att = run_gpu(lib, wl, pools=(K, V), Q=Q, **opts)
    assert att.plan.stats()["n_tc_items"] > 0
    assert_matches(wl, O, L, K, V, Q, queries=range(0, n_req, 3))


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("p_bf16_min_tokens", [0, 1], ids=["default_precision", "p_rounded_once"])
def test_random_trees_many_rows(lib, seed, d, p_bf16_min_tokens):
    """Up to 96 queries x G=4 per node: row blocks of 256 (both softmax row
    halves) and of fewer than 128 rows side by side, both P precisions."""
    wl = synth.random_tree(9500 + seed, max_nodes=8, max_len=400, heads=(8, 2), d=d, dtype="bf16",
                           n_queries=96)
    O, L, (K, V, Q), att = run_gpu(lib, wl, tc_min_rows=16, p_bf16_min_tokens=p_bf16_min_tokens)
    assert att.plan.stats()["n_tc_items"] > 0
    assert_matches(wl, O, L, K, V, Q)


def _peaked_prefix(prefix, n_req):
    """A document-QA tree in which every query has one dominant token in the
    shared prefix: query q puts a large value A in channel q of all its heads,
    and its token t_q carries B_q in that channel of every kv head, so its
    score on t_q rises by A B_q / sqrt(d) (8.0 to 10.6 nats): that one token
    takes from a few percent up to 98 % of a row's softmax mass (most rows
    above 30 %). The dominant tokens sit past the first tile of the prefix and
    their V rows are +-3. A model of P rounded once to bf16 (with the running
    max lagging the true one) misses the oracle by up to ~8e-3 here."""
    wl = synth.document_qa(prefix=prefix, n_req=n_req)
    K, V = wl.kv_pools()
    Q = wl.q()
    lids = wl.row_lids().reshape(wl.num_pages, wl.page_size)
    root = wl.lid[wl.lid_ptr[0]:wl.lid_ptr[1]]
    bf16 = {8.0: 0x4100, 9.0: 0x4110, 10.0: 0x4120, 11.0: 0x4130, 12.0: 0x4140, 3.0: 0x4040, -3.0: 0xC040}
    for q in range(n_req):
        t = 160 + (q * 613) % (prefix - 160)
        page, row = np.argwhere(lids == root[t])[0]
        c = q % wl.d
        K[page, :, row, c] = bf16[(9.0, 10.0, 11.0, 12.0)[q % 4]]
        V[page, :, row, :] = np.where(np.arange(wl.d) % 2 == q % 2, bf16[3.0], bf16[-3.0])
        Q[q, :, c] = bf16[10.0]
    return wl, K, V, Q


@pytest.mark.parametrize("n_req", [64, 16], ids=["rows256", "rows64"])
@pytest.mark.parametrize("opts", [{}, {"p_bf16_min_tokens": 1}, {"split_policy": "none"}],
                         ids=["default", "p_rounded_once_everywhere", "no_split"])
def test_peaked_attention_on_long_node(lib, n_req, opts):
    """Softmax mass concentrated on one token of a 2048-token node: the
    tensor-core PAC instance that rounds P to bf16 must add the lo products on
    the tiles where one weight dominates."""
    wl, K, V, Q = _peaked_prefix(2048, n_req)
    O, L, _, att = run_gpu(lib, wl, pools=(K, V), Q=Q, **opts)
    assert att.plan.stats()["n_tc_items"] > 0
    assert_matches(wl, O, L, K, V, Q)
