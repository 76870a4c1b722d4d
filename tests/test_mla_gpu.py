"""GPU parity of the MLA path: pst_mla_reconstruct (per-head K/V rebuilt from
a latent cache on the tensor cores) against oracle/mla.py, then the decode
pipeline on the rebuilt pools against the oracle's attention on its own.

The rebuilt values are bf16: the kernel rounds an fp32 tensor-core sum, the
oracle the exact fp64 sum. Where they differ, the kernel's value must be the
bf16 rounding of some value within the fp32 sum's error bound of the exact
one (d_c * 2^-23 * sum |w c|: twice the bound for fp32 accumulation of d_c
exact products in any order), i.e. lie between the roundings of
exact - bound and exact + bound; such elements are rare (near a rounding
boundary, or small values of sums that cancel)."""
import numpy as np
import pytest

import synth
from oracle import attention as oa
from oracle import mla

pytestmark = pytest.mark.gpu

ABS_TOL, REL_TOL, LSE_TOL = 2e-3, 1e-2, 1e-3
SENTINEL = 0x7FC1   # a NaN pattern: pages outside the tree must keep it


def _run(lib, wl, d_c):
    import torch
    from prefix_shared_tree_gb300.torch_api import TreeDecodeAttention, to_device
    C, Wk, Wv = wl.mla_inputs(d_c)
    att = TreeDecodeAttention.from_workload(wl)
    Cd, Wkd, Wvd = (to_device(x, "bf16") for x in (C, Wk, Wv))
    shape = (wl.num_pages, wl.n_kv_heads, wl.page_size, wl.d)
    Kd = torch.full(shape, 0, dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    Vd = torch.full(shape, 0, dtype=torch.int16, device="cuda").fill_(SENTINEL).view(torch.bfloat16)
    att.mla_reconstruct(Cd, Wkd, Wvd, Kd, Vd)
    Q = wl.q()
    O, L = att(to_device(Q, "bf16"), Kd, Vd)
    torch.cuda.synchronize()
    assert att.check_status() == 0
    Kg = Kd.view(torch.int16).cpu().numpy().view(np.uint16)
    Vg = Vd.view(torch.int16).cpu().numpy().view(np.uint16)
    return (C, Wk, Wv), (Kg, Vg), Q, O.cpu().numpy(), L.cpu().numpy()


def _check_pools(wl, inputs, got):
    C, Wk, Wv = inputs
    Kg, Vg = got
    exact = mla.reconstruct_exact(wl, C, Wk, Wv)
    pages = set(exact)
    d_c = C.shape[-1]
    absw = [np.abs(oa.bf16_to_f64(W)) for W in (Wk, Wv)]
    flips = 0
    for page in range(wl.num_pages):
        if page not in pages:
            assert np.all(Kg[page] == SENTINEL) and np.all(Vg[page] == SENTINEL), f"page {page} written"
            continue
        absc = np.abs(oa.bf16_to_f64(C[page]))
        for which, (g, x) in enumerate(((Kg[page], exact[page][0]), (Vg[page], exact[page][1]))):
            want = mla.f64_to_bf16(x)
            diff = g != want
            if not diff.any():
                continue
            gv = oa.bf16_to_f64(g[diff])
            mag = np.einsum("hec,rc->hre", absw[which], absc)[diff]
            bound = d_c * 2.0 ** -23 * mag
            lo = oa.bf16_to_f64(mla.f64_to_bf16(x[diff] - bound))
            hi = oa.bf16_to_f64(mla.f64_to_bf16(x[diff] + bound))
            assert np.all((gv >= lo) & (gv <= hi)), f"page {page}: a value no fp32 sum of the products rounds to"
            flips += int(diff.sum())
    return flips


@pytest.mark.parametrize("seed,d_c,heads,d", [(1, 128, (4, 2), 128), (2, 256, (8, 8), 128), (3, 512, (8, 4), 128),
                                              (4, 384, (4, 4), 64), (5, 512, (16, 16), 64), (6, 256, (2, 1), 128)])
def test_mla_rebuild_and_decode_match_the_oracle(lib, seed, d_c, heads, d):
    wl = synth.random_tree(7100 + seed, max_nodes=12, max_len=200, heads=heads, d=d, dtype="bf16", n_queries=20)
    inputs, got, Q, O, L = _run(lib, wl, d_c)
    flips = _check_pools(wl, inputs, got)
    # every flip is already proven legal above; this only bounds their number
    # (fp32 sums of a few hundred products are off by ~1e-5 relative, the bf16
    # half unit is 2^-9, so roughly one element in a few thousand flips)
    n_el = len(np.unique(wl.page_ids)) * wl.n_kv_heads * wl.page_size * wl.d * 2
    assert flips <= 2e-3 * n_el
    # attention on the rebuilt pools against the oracle's attention on its own
    Oref, Lref = mla.decode_attention_mla(wl, *inputs, Q)
    err = np.abs(O.astype(np.float64) - Oref)
    assert np.all(np.isfinite(O)) and err.max() <= ABS_TOL
    rel = err.max(axis=2) / np.maximum(np.abs(Oref).max(axis=2), 1e-6)
    assert rel.max() <= REL_TOL
    assert np.abs(L.astype(np.float64) - Lref).max() <= LSE_TOL


def test_mla_document_qa_shape_every_query(lib):
    """A document-QA tree (4096-token shared prefix, 32 requests) with MHA
    after the rebuild: 16 heads of 128, latent of 512."""
    wl = synth.document_qa(prefix=4096, n_req=32, heads=(16, 16))
    inputs, got, Q, O, L = _run(lib, wl, 512)
    _check_pools(wl, inputs, got)
    Oref, Lref = mla.decode_attention_mla(wl, *inputs, Q)
    err = np.abs(O.astype(np.float64) - Oref)
    assert err.max() <= ABS_TOL
    rel = err.max(axis=2) / np.maximum(np.abs(Oref).max(axis=2), 1e-6)
    assert rel.max() <= REL_TOL
    assert np.abs(L.astype(np.float64) - Lref).max() <= LSE_TOL
