"""Pins of the MLA oracle (oracle/mla.py) to facts outside itself: bf16
rounding against an integer round-half-even on fp32 bit patterns and worked
ties; the reconstruction against selection matrices, whose products are
slices of the latent exactly; and the reduction to the plain decode oracle.
A planted mistake (the up-projection read transposed) fails a pin."""
import numpy as np
import pytest

import synth
from oracle import attention as oa
from oracle import mla


def _bf16_rne_of_f32(x32: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 bits with the integer form of round half to
    even on the low 16 bits of the pattern (finite inputs)."""
    u = np.asarray(x32, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)).astype(np.uint16)


def test_bf16_rounding_worked_ties():
    one = 1.0
    cases = {one: 0x3F80, one + 2.0**-8: 0x3F80,           # tie, even (down)
             one + 3 * 2.0**-8: 0x3F82,                     # tie, even (up)
             one + 2.0**-8 + 2.0**-30: 0x3F81,              # just above the tie
             -(one + 2.0**-8 + 2.0**-30): 0xBF81,
             -(one + 3 * 2.0**-8): 0xBF82}
    for x, want in cases.items():
        assert int(mla.f64_to_bf16(np.array([x]))[0]) == want, x
    assert int(mla.f64_to_bf16(np.array([0.0]))[0]) == 0


def test_bf16_rounding_matches_integer_rne_on_fp32_values():
    x = (synth.rng.normal(synth.rng.stream_key(7, 1), 0, 200000) * 10.0).astype(np.float32)
    x[::7] *= np.float32(1e-20)
    x[::11] *= np.float32(1e20)
    assert np.array_equal(mla.f64_to_bf16(x.astype(np.float64)), _bf16_rne_of_f32(x))


def test_bf16_rounding_of_values_between_fp32_neighbours():
    # x = f + a quarter of an fp32 ulp: no double rounding through fp32
    f = np.float32(1.0) + np.float32(2.0**-8)          # an exact bf16 tie as fp32
    x = float(f) + 2.0**-26                            # slightly above the tie
    assert int(mla.f64_to_bf16(np.array([x]))[0]) == 0x3F81
    x = float(f) - 2.0**-26                            # slightly below the tie
    assert int(mla.f64_to_bf16(np.array([x]))[0]) == 0x3F80


def _selection(H, d, d_c, shift, value_bits=0x3F80):
    """W[h][e][c] = value at c == (h * shift + e) % d_c, else 0 (bf16 bits)."""
    W = np.zeros((H, d, d_c), np.uint16)
    for h in range(H):
        for e in range(d):
            W[h, e, (h * shift + e) % d_c] = value_bits
    return W


@pytest.mark.parametrize("d_c", [128, 256])
def test_reconstruction_by_selection_is_a_slice_of_the_latent(d_c):
    wl = synth.random_tree(41, max_nodes=8, max_len=50, heads=(4, 4), d=128, n_queries=5)
    C, _, _ = wl.mla_inputs(d_c)
    H, d = wl.n_kv_heads, wl.d
    Wk = _selection(H, d, d_c, shift=37)
    Wv = _selection(H, d, d_c, shift=5, value_bits=0x4000)     # 2.0
    K, V = mla.reconstruct(wl, C, Wk, Wv)
    used = np.unique(wl.page_ids)
    Cf = oa.bf16_to_f64(C)
    for page in range(wl.num_pages):
        for h in range(H):
            idx_k = (h * 37 + np.arange(d)) % d_c
            idx_v = (h * 5 + np.arange(d)) % d_c
            if page in used:
                assert np.array_equal(K[page, h], C[page][:, idx_k])
                assert np.array_equal(oa.bf16_to_f64(V[page, h]), 2.0 * Cf[page][:, idx_v])
            else:
                assert not K[page].any() and not V[page].any()     # untouched


def test_planted_transpose_fails_the_selection_pin():
    wl = synth.random_tree(42, max_nodes=6, max_len=40, heads=(2, 2), d=128, n_queries=4)
    C, _, _ = wl.mla_inputs(128)
    Wk = _selection(2, 128, 128, shift=3)

    def wrong_exact(tr, C_pool, W_uk, W_uv):   # reads W[h] as [d_c][d]
        out = {}
        for page in mla.tree_pages(tr):
            c = oa.bf16_to_f64(C_pool[page])
            out[int(page)] = (np.einsum("hce,rc->hre", oa.bf16_to_f64(W_uk), c),) * 2
        return out

    good = mla.reconstruct_exact(wl, C, Wk, Wk)
    bad = wrong_exact(wl, C, Wk, Wk)
    p = int(mla.tree_pages(wl)[0])
    sel = np.stack([oa.bf16_to_f64(C[p])[:, (h * 3 + np.arange(128)) % 128] for h in range(2)])
    assert np.array_equal(good[p][0], sel)
    assert not np.array_equal(bad[p][0], sel)


def test_mla_attention_reduces_to_plain_decode():
    """With selection up-projections the rebuilt pools are known exactly, so
    MLA decode equals the plain decode oracle on those pools."""
    wl = synth.random_tree(43, max_nodes=8, max_len=60, heads=(4, 2), d=128, n_queries=6)
    C, _, _ = wl.mla_inputs(256)
    Wk = _selection(2, 128, 256, shift=64)
    Wv = _selection(2, 128, 256, shift=11)
    Q = wl.q()
    O, L = mla.decode_attention_mla(wl, C, Wk, Wv, Q)
    K = np.zeros((wl.num_pages, 2, 16, 128), np.uint16)
    V = np.zeros_like(K)
    for page in np.unique(wl.page_ids):
        for h in range(2):
            K[page, h] = C[page][:, (h * 64 + np.arange(128)) % 256]
            V[page, h] = C[page][:, (h * 11 + np.arange(128)) % 256]
    O2, L2 = oa.decode_attention(wl, K, V, Q)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
