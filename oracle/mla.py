"""Oracle, multi-head latent attention: per-head K/V rebuilt from a latent
cache, then the same decode attention.

TEST INFRASTRUCTURE (see the package docstring).

Source
  * CoDec, "supplementary details" (the kernel module paragraph on MLA
    models): the per-head KV blocks are first reconstructed from the latent
    representation, then the same prefix-aware attention and reduction run.

Readings where the page leaves a step open
  * Token j's latent c_j has d_c channels; kv head h reconstructs
    k_{h,j} = W_UK[h] c_j and v_{h,j} = W_UV[h] c_j with up-projections of
    d x d_c (W[h][e] is the weight row of output channel e). No decoupled
    positional key part: the page names only the reconstruction.
  * The reconstructed blocks are stored in the pools' element type (bf16),
    rounded once to nearest-even from the exact (here fp64) product, and the
    attention then reads them like any other pool.
  * Only the pages the tree's nodes use are reconstructed; every row of such
    a page is (rows no node covers are never read by the attention).

All arithmetic is fp64; the only rounding is the final one to bf16.
"""
from __future__ import annotations

import numpy as np

from . import attention as _att


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 bit patterns, nearest-even, in one step:
    the bf16 grid point nearest to x (the even one on a tie), found from the
    two neighbours that bracket x, so no intermediate fp32 rounding occurs.
    Finite inputs within the bf16 range only."""
    x = np.asarray(x, dtype=np.float64)
    # truncation toward zero to a bf16 value: fp32 truncation of the fp64
    # value can round, so step the fp32 bits down when it overshot |x|
    f = x.astype(np.float32)
    overshoot = np.abs(f.astype(np.float64)) > np.abs(x)
    fb = f.view(np.uint32).copy()
    fb[overshoot] -= np.uint32(1)          # the fp32 just below |x| in magnitude
    lo = fb & np.uint32(0xFFFF0000)        # bf16 at or below |x| in magnitude
    hi = lo + np.uint32(0x10000)           # the next bf16 up in magnitude
    lo_v = lo.view(np.float32).astype(np.float64)
    hi_v = hi.view(np.float32).astype(np.float64)
    d_lo = np.abs(x - lo_v)
    d_hi = np.abs(hi_v - x)
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (((lo >> np.uint32(16)) & np.uint32(1)) == 1))
    out = np.where(take_hi, hi, lo) >> np.uint32(16)
    return np.where(x == 0, np.uint32(0), out).astype(np.uint16)


def tree_pages(tr) -> np.ndarray:
    """Every page some node of the tree uses, once, ascending."""
    return np.unique(np.asarray(tr.page_ids, dtype=np.int64))


def reconstruct_exact(tr, C_pool, W_uk, W_uv):
    """Exact (fp64) per-head K and V of the tree's pages:
    dict page -> (K [Hkv][page_size][d], V likewise), from the latent pool
    C_pool [num_pages][page_size][d_c] and W [Hkv][d][d_c] (bf16 bits)."""
    Wk = _att.bf16_to_f64(W_uk)
    Wv = _att.bf16_to_f64(W_uv)
    out = {}
    for page in tree_pages(tr):
        c = _att.bf16_to_f64(C_pool[page])                   # [page_size][d_c]
        # k[h][r][e] = sum_c W[h][e][c] * c[r][c]
        k = np.einsum("hec,rc->hre", Wk, c)
        v = np.einsum("hec,rc->hre", Wv, c)
        out[int(page)] = (k, v)
    return out


def reconstruct(tr, C_pool, W_uk, W_uv, K_pool=None, V_pool=None):
    """The rebuilt pools (bf16 bits, [num_pages][Hkv][page_size][d]): the
    tree's pages hold bf16(W C); other pages keep K_pool / V_pool's contents
    (zeros when not given)."""
    Hkv, d, _ = np.shape(W_uk)
    num_pages, page_size, _ = np.shape(C_pool)
    K = np.zeros((num_pages, Hkv, page_size, d), np.uint16) if K_pool is None else np.array(K_pool, np.uint16)
    V = np.zeros_like(K) if V_pool is None else np.array(V_pool, np.uint16)
    for page, (k, v) in reconstruct_exact(tr, C_pool, W_uk, W_uv).items():
        K[page] = f64_to_bf16(k)
        V[page] = f64_to_bf16(v)
    return K, V


def decode_attention_mla(tr, C_pool, W_uk, W_uv, Q, queries=None):
    """Tree decode attention on the reconstructed pools (the same oracle as
    for stored K/V)."""
    K, V = reconstruct(tr, C_pool, W_uk, W_uv)
    return _att.decode_attention(tr, K, V, Q, queries)
