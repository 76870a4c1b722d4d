"""pst_decode_attn_noalloc: the entry point for callers that cannot allocate
device memory where they run attention (its scratch is a fixed array inside
the library). Its outputs must equal pst_decode_attn's on the same inputs: the
same kernels run the same plan on the same data, and every kernel's result
depends only on its own item (never on which block ran it or when), so the
two paths agree bit for bit. Two calls are checked, with a different plan
(more partial rows) run through the shared array between them, so that the
second call starts from unrelated contents. The array's status word is read
with pst_noalloc_check_status. Both launch orders are checked (launch groups
chained on one stream, and one after the other). This file sorts last so that a run stopping at
its first failure has run everything else."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

ABS_TOL, LSE_TOL = 2e-3, 1e-3


def _setup(wl, **opts):
    import torch
    from prefix_shared_tree_gb300.torch_api import TreeDecodeAttention, to_device
    att = TreeDecodeAttention.from_workload(wl, **opts)
    K, V = wl.kv_pools()
    return att, to_device(wl.q(), wl.dtype), to_device(K, wl.dtype), to_device(V, wl.dtype)


def _other_plan():
    """Unrelated data for the shared array: the few-shot tree cut into
    256-token chunks (more partial rows than any plan checked here, and a
    scratch that still fits the array)."""
    return _setup(synth.few_shot(), split_policy="uniform", fixed_chunk=256)


@pytest.mark.parametrize("make", [synth.few_shot, lambda: synth.random_tree(4242, max_nodes=12, max_len=200,
                                                                              heads=(8, 2), d=128, n_queries=30),
                                  synth.tiny_two_level],
                         ids=["few_shot", "random_bf16", "tiny_fp32"])
@pytest.mark.parametrize("side_streams", [False, True], ids=["chained", "serial"])
def test_noalloc_matches_workspace_path(lib, make, side_streams):
    """side_streams: the workspace path forks its launch groups onto side
    streams and the no-allocation path runs them one after the other; else
    both chain them on the caller's stream."""
    import torch
    wl = make()
    att, Q, K, V = _setup(wl, side_streams=side_streams)
    assert att.plan.workspace_bytes <= lib.NOALLOC_WORKSPACE_BYTES
    O_ref, L_ref = att(Q, K, V)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream().cuda_stream
    other, oQ, oK, oV = _other_plan()
    assert other.plan.stats()["n_partial_rows"] > att.plan.stats()["n_partial_rows"]
    oO = torch.empty((other.n_queries, other.n_q_heads, other.d), dtype=torch.float32, device=Q.device)
    oL = torch.empty((other.n_queries, other.n_q_heads), dtype=torch.float32, device=Q.device)
    for call in range(2):
        if call == 1:
            lib.decode_attn_noalloc(other.plan, oQ.data_ptr(), oK.data_ptr(), oV.data_ptr(), oO.data_ptr(),
                                    oL.data_ptr(), st)
        O = torch.full_like(O_ref, float("nan"))
        L = torch.full_like(L_ref, float("nan"))
        lib.decode_attn_noalloc(att.plan, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), L.data_ptr(), st)
        torch.cuda.synchronize()
        assert lib.noalloc_check_status(st) == 0
        assert torch.equal(O, O_ref) and torch.equal(L, L_ref), f"call {call} differs from the workspace path"


def test_noalloc_reports_a_wait_that_ran_out(lib):
    """A bounded wait that runs out inside a no-allocation call (the test-only
    plan option debug_stall) shows in the array's status word; the next call
    is clean."""
    import torch
    wl = synth.document_qa(prefix=1024, n_req=64)
    stalled, Q, K, V = _setup(wl, debug_stall=True)
    normal, _, _, _ = _setup(wl)
    st = torch.cuda.current_stream().cuda_stream
    O = torch.empty((wl.n_queries, wl.n_q_heads, wl.d), dtype=torch.float32, device=Q.device)
    L = torch.empty((wl.n_queries, wl.n_q_heads), dtype=torch.float32, device=Q.device)
    lib.decode_attn_noalloc(stalled.plan, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), L.data_ptr(), st)
    torch.cuda.synchronize()
    assert lib.noalloc_check_status(st) & 1
    assert lib.noalloc_check_status(st) == 0
    O_ref, L_ref = normal(Q, K, V)
    lib.decode_attn_noalloc(normal.plan, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), L.data_ptr(), st)
    torch.cuda.synchronize()
    assert lib.noalloc_check_status(st) == 0
    assert torch.equal(O, O_ref) and torch.equal(L, L_ref)


def test_noalloc_after_another_plan(lib):
    """A call with plan B after plan A: B's metadata replaces A's in the array."""
    import torch
    a = _setup(synth.few_shot())
    b = _setup(synth.random_tree(4343, max_nodes=9, max_len=120, heads=(8, 2), d=128, n_queries=12))
    st = torch.cuda.current_stream().cuda_stream
    refs = [x[0](x[1], x[2], x[3]) for x in (a, b)]
    for (att, Q, K, V), (O_ref, L_ref) in zip((a, b), refs):
        O = torch.empty_like(O_ref)
        L = torch.empty_like(L_ref)
        lib.decode_attn_noalloc(att.plan, Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), L.data_ptr(), st)
        torch.cuda.synchronize()
        assert np.abs(O.cpu().numpy() - O_ref.cpu().numpy()).max() <= ABS_TOL
        assert np.abs(L.cpu().numpy() - L_ref.cpu().numpy()).max() <= LSE_TOL


def test_noalloc_rejects_oversized_plan(lib):
    """A plan whose scratch exceeds the built-in array is refused before any GPU work."""
    wl = synth.tree_of_thought("mha")
    t = lib.tree_build(wl.node_len, wl.parent, wl.page_ptr, wl.page_ids, wl.first_offset, wl.page_size,
                       wl.num_pages)
    p = lib.plan_create(t, wl.query_node, wl.n_q_heads, wl.n_kv_heads, wl.d, wl.dtype, num_sms=152,
                        split_policy="uniform", fixed_chunk=64)
    assert p.workspace_bytes > lib.NOALLOC_WORKSPACE_BYTES
    with pytest.raises(lib.PstError) as e:
        lib.decode_attn_noalloc(p, 16, 16, 16, 16, 16, 0)
    assert e.value.code == -5 and "built-in scratch" in str(e.value)
