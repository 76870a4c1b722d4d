// Device helpers shared by the PAC and POR kernels: mbarriers with bounded
// waits, TMA tile loads, the 128-byte swizzle of staged K/V tiles, and the
// TMA producer loop that streams a chunk's pages into a shared-memory ring.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pst_internal.h"

namespace pst {
namespace dev {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// A wait gives up after this many SM cycles (about two seconds), sets the
// status word and lets the caller leave the kernel.
constexpr long long kWaitCycles = 4000000000LL;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > kWaitCycles) {
            atomicOr(status, kStatusWaitTimeout);
            return false;
        }
    }
}

// 3-D tiled TMA load (dims: channel, row-in-page, page*Hkv + head) into shared
// memory, completing on the mbarrier `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Byte offset of 16-byte chunk `c` (0..7) of row `row` inside a 128-byte-wide
// slab staged with the TMA 128B swizzle (slab base 1024-byte aligned).
__device__ __forceinline__ uint32_t swz(int row, int c) {
    return static_cast<uint32_t>(row * 128 + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Chunk geometry in page space: the chunk covers positions
// [pos_begin, pos_end); tiles of kTileTokens start at multiples of the tile.
struct ChunkGeo {
    int pos_begin, pos_end, tile0, n_tiles;
};

__device__ __forceinline__ ChunkGeo chunk_geo(const DevChunk& c) {
    ChunkGeo g;
    g.pos_begin = c.pos_begin;
    g.pos_end = c.pos_begin + c.n_tok;
    g.tile0 = (c.pos_begin / kTileTokens) * kTileTokens;
    g.n_tiles = (g.pos_end - g.tile0 + kTileTokens - 1) / kTileTokens;
    return g;
}

// TMA producer (one elected thread): streams every tile of the chunk through
// a ring of `STAGES` stages. Stage s holds K then V, each NSLAB slabs of
// kTileTokens rows x 128 bytes. Boxes entirely outside the chunk are skipped.
template <int NSLAB, int STAGES, int ELEMS_PER_SLAB>
__device__ void produce_chunk(const DevPlan& P, const DevChunk& C, int head, uint32_t ring,
                              uint32_t bar_full, uint32_t bar_empty, const CUtensorMap* tk,
                              const CUtensorMap* tv) {
    constexpr uint32_t kSlabBytes = kTileTokens * 128;
    constexpr uint32_t kHalf = NSLAB * kSlabBytes;  // K (or V) part of a stage
    const ChunkGeo g = chunk_geo(C);
    const int ps = P.page_size;
    const int n_list = (g.pos_end - 1) / ps + 1;  // page list entries the chunk reaches
    for (int i = 0; i < g.n_tiles; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES) {
            if (!mbar_wait(bar_empty + 8 * s, ((i / STAGES) - 1) & 1, P.status)) return;
        }
        const int tpos = g.tile0 + i * kTileTokens;
        uint32_t nbox = 0;
#pragma unroll
        for (int b = 0; b < kTileTokens / kBoxRows; ++b) {
            const int pos = tpos + b * kBoxRows;
            if (pos + kBoxRows > g.pos_begin && pos < g.pos_end) ++nbox;
        }
        const uint32_t full = bar_full + 8 * s;
        mbar_arrive_expect_tx(full, nbox * NSLAB * kBoxRows * 128u * 2u);
        const uint32_t kbase = ring + s * 2 * kHalf;
        const uint32_t vbase = kbase + kHalf;
#pragma unroll
        for (int b = 0; b < kTileTokens / kBoxRows; ++b) {
            const int pos = tpos + b * kBoxRows;
            if (!(pos + kBoxRows > g.pos_begin && pos < g.pos_end)) continue;
            const int li = pos / ps;
            int page = 0;
            if (li < n_list) page = P.pages[C.page_base + li];
            const int slab_z = page * P.n_kv_heads + head;
            const int row0 = pos % ps;
#pragma unroll
            for (int sl = 0; sl < NSLAB; ++sl) {
                const uint32_t off = sl * kSlabBytes + b * kBoxRows * 128;
                tma_load_3d(kbase + off, tk, sl * ELEMS_PER_SLAB, row0, slab_z, full);
                tma_load_3d(vbase + off, tv, sl * ELEMS_PER_SLAB, row0, slab_z, full);
            }
        }
    }
}

// TMA producer for one operand (K when `vee` is false, V when true) with its
// own full/empty barriers, so K stages can be refilled as soon as Q K^T has
// read them while V stages wait for P V. Stage s holds K at
// ring + s*stage_bytes and V right after it (NSLAB slabs each).
template <int NSLAB, int STAGES, int ELEMS_PER_SLAB>
__device__ void produce_operand(const DevPlan& P, const DevChunk& C, int head, uint32_t ring, uint32_t stage_bytes,
                                uint32_t bar_full, uint32_t bar_empty, const CUtensorMap* map, bool vee) {
    constexpr uint32_t kSlabBytes = kTileTokens * 128;
    constexpr uint32_t kHalf = NSLAB * kSlabBytes;
    const ChunkGeo g = chunk_geo(C);
    const int ps = P.page_size;
    const int n_list = (g.pos_end - 1) / ps + 1;
    for (int i = 0; i < g.n_tiles; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES) {
            if (!mbar_wait(bar_empty + 8 * s, ((i / STAGES) - 1) & 1, P.status)) return;
        }
        const int tpos = g.tile0 + i * kTileTokens;
        uint32_t nbox = 0;
#pragma unroll
        for (int b = 0; b < kTileTokens / kBoxRows; ++b) {
            const int pos = tpos + b * kBoxRows;
            if (pos + kBoxRows > g.pos_begin && pos < g.pos_end) ++nbox;
        }
        const uint32_t full = bar_full + 8 * s;
        mbar_arrive_expect_tx(full, nbox * NSLAB * kBoxRows * 128u);
        const uint32_t dst0 = ring + s * stage_bytes + (vee ? kHalf : 0);
#pragma unroll
        for (int b = 0; b < kTileTokens / kBoxRows; ++b) {
            const int pos = tpos + b * kBoxRows;
            if (!(pos + kBoxRows > g.pos_begin && pos < g.pos_end)) continue;
            const int li = pos / ps;
            int page = 0;
            if (li < n_list) page = P.pages[C.page_base + li];
            const int slab_z = page * P.n_kv_heads + head;
            const int row0 = pos % ps;
#pragma unroll
            for (int sl = 0; sl < NSLAB; ++sl)
                tma_load_3d(dst0 + sl * kSlabBytes + b * kBoxRows * 128, map, sl * ELEMS_PER_SLAB, row0, slab_z, full);
        }
    }
}

}  // namespace dev
}  // namespace pst
