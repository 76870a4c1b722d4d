// Device helpers shared by the PAC and POR kernels: mbarriers with bounded
// waits, TMA tile loads, the 128-byte swizzle of staged K/V tiles, and the
// TMA producer loop that streams a chunk's pages into a shared-memory ring.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <utility>

#include "pst_internal.h"

namespace pst {

// One-time set-up per device of a kernel's launch (its shared-memory limit,
// the register-count check, the SM count or resident blocks): the runtime
// keeps function attributes per device, so each device runs the set-up once,
// under a lock, and keeps two values from it.
constexpr int kMaxCachedDevices = 64;
struct DeviceOnce {
    std::mutex mu;
    int v0[kMaxCachedDevices] = {}, v1[kMaxCachedDevices] = {};   // v0 == 0: not set up yet
};
template <typename F>
inline cudaError_t per_device(DeviceOnce& c, int* v0, int* v1, F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxCachedDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(c.mu);
    if (!c.v0[dev]) {
        int a = 0, b = 0;
        e = setup(dev, &a, &b);
        if (e != cudaSuccess) return e;
        c.v0[dev] = a > 0 ? a : 1;
        c.v1[dev] = b;
    }
    if (v0) *v0 = c.v0[dev];
    if (v1) *v1 = c.v1[dev];
    return cudaSuccess;
}

// Kernel launch with an optional programmatic dependency on the kernel
// before it on `st` (programmatic dependent launch, sm_90 and later). With
// `pdl` the kernel may start as soon as every block of that kernel has
// executed griddepcontrol.launch_dependents (each PAC kernel does so first
// thing), instead of when it has finished: the PAC launch groups of one call
// then share the SMs in launch order on a single stream. A later launch
// without the attribute still waits for every kernel before it to finish,
// and griddepcontrol.wait waits for all of them too.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                 bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The kernels of one decode call in launch order: on one stream (`chain`)
// every kernel after the first gets the programmatic dependency above; on
// per-group streams none does.
struct LaunchSeq {
    cudaStream_t st;
    bool chain;
    int n = 0;
    LaunchSeq(cudaStream_t s, bool c) : st(s), chain(c) {}
    bool next_pdl() {
        const bool r = chain && n > 0;
        ++n;
        return r;
    }
};

namespace dev {

// Let the next kernel on the stream start once every block of this one has
// started (no-op when it was not launched with the attribute).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until every kernel this one depends on has finished and its writes
// are visible (returns at once for a launch without the attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// As mbar_try_wait, but the hardware may suspend the thread (without taking
// issue slots from the warps that do work) until the phase completes or about
// `ns` nanoseconds have passed.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// A wait gives up after this many SM cycles (about two seconds), sets the
// status word and lets the caller leave the kernel.
constexpr long long kWaitCycles = 4000000000LL;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* status,
                                          long long limit = kWaitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait_suspend(bar, parity, limit < kWaitCycles ? 1000u : 100000u)) return true;
        if (clock64() - t0 > limit) {
            atomicOr(status, kStatusWaitTimeout);
            return false;
        }
    }
}

// Before a block leaves after a wait gave up, a TMA producer waits (bounded)
// until the loads it issued into a ring's last stages have landed, so that no
// bulk copy still writes into the block's shared memory when it exits: ring
// tile g (global count, `issued` tiles so far) completes phase (g / ST) & 1
// of full barrier g % ST, and for the last ST tiles issued that phase is the
// barrier's latest.
template <int ST>
__device__ __forceinline__ void drain_ring(uint32_t bar_full, int issued, int32_t* status) {
    for (int g = issued > ST ? issued - ST : 0; g < issued; ++g) mbar_wait(bar_full + 8 * (g % ST), (g / ST) & 1, status);
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

// 5-D tiled TMA load (64 channels, page row, head, slab, page) into shared
// memory: the pools' second view, whose slab stride (128 bytes) lets one box
// carry both 64-channel halves of a row.
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            int c4, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
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

// max(a, b, c) in one instruction (sm_100 family)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Chunk geometry in page space: the chunk covers positions
// [pos_begin, pos_end); tiles of TT tokens start at multiples of TT.
struct ChunkGeo {
    int pos_begin, pos_end, tile0, n_tiles;
};

template <int TT = kTileTokens>
__device__ __forceinline__ ChunkGeo chunk_geo(const DevChunk& c) {
    ChunkGeo g;
    g.pos_begin = c.pos_begin;
    g.pos_end = c.pos_begin + c.n_tok;
    g.tile0 = (c.pos_begin / TT) * TT;
    g.n_tiles = (g.pos_end - g.tile0 + TT - 1) / TT;
    return g;
}

// TMA producer (one elected thread): streams every tile of the chunk through
// a ring of `STAGES` stages. Stage s holds K then V, each NSLAB slabs of
// kTileTokens rows x 128 bytes. Boxes entirely outside the chunk are skipped.
// `tbase` tiles went through the ring before this chunk (stage and phase
// continue from there).
template <int NSLAB, int STAGES, int ELEMS_PER_SLAB>
__device__ bool produce_chunk(const DevPlan& P, const DevChunk& C, int head, uint32_t ring,
                              uint32_t bar_full, uint32_t bar_empty, const CUtensorMap* tk,
                              const CUtensorMap* tv, int tbase = 0) {
    constexpr uint32_t kSlabBytes = kTileTokens * 128;
    constexpr uint32_t kHalf = NSLAB * kSlabBytes;  // K (or V) part of a stage
    const ChunkGeo g = chunk_geo(C);
    const int ps = P.page_size;
    const int n_list = (g.pos_end - 1) / ps + 1;  // page list entries the chunk reaches
    for (int i = 0; i < g.n_tiles; ++i) {
        const int I = tbase + i;
        const int s = I % STAGES;
        if (I >= STAGES) {
            if (!mbar_wait(bar_empty + 8 * s, ((I / STAGES) - 1) & 1, P.status)) {
                drain_ring<STAGES>(bar_full, I, P.status);
                return false;
            }
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
    return true;
}

// The end of a producer's work: its last loads have landed before it leaves
// (when its consumers stopped early they would not wait for them).
template <int ST>
__device__ __forceinline__ void producer_done(uint32_t bar_full, int issued, int32_t* status) {
    drain_ring<ST>(bar_full, issued, status);
}

// TMA producer for one operand (K or V) with its own full/empty barriers:
// tiles of TT tokens go round a ring of STAGES stages; stage s starts at
// ring + s * NSLAB * TT * 128 and holds NSLAB slabs of TT rows x 128 bytes.
// Boxes entirely outside the chunk are skipped.
// With NPART > 1, producer `part` of NPART issues the boxes b with
// b % NPART == part and announces their bytes (bar_full then expects NPART
// arrivals): the TMA unit takes a few hundred cycles per instruction from one
// thread, so several issuing threads fill a stage sooner.
template <int NSLAB, int TT, int STAGES, int NPART = 1>
__device__ bool produce_tiles(const DevPlan& P, const DevChunk& C, int head, uint32_t ring, uint32_t bar_full,
                              uint32_t bar_empty, const CUtensorMap* map, int part = 0) {
    constexpr uint32_t kSlabBytes = TT * 128;
    constexpr uint32_t kStageBytes = NSLAB * kSlabBytes;
    const ChunkGeo g = chunk_geo<TT>(C);
    const int ps = P.page_size;
    const int n_list = (g.pos_end - 1) / ps + 1;
    for (int i = 0; i < g.n_tiles; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES) {
            if (!mbar_wait(bar_empty + 8 * s, ((i / STAGES) - 1) & 1, P.status)) {
                drain_ring<STAGES>(bar_full, i, P.status);
                return false;
            }
        }
        const int tpos = g.tile0 + i * TT;
        int page[TT / kBoxRows];
        uint32_t nbox = 0;
#pragma unroll
        for (int b = 0; b < TT / kBoxRows; ++b) {
            const int pos = tpos + b * kBoxRows;
            const bool in = pos + kBoxRows > g.pos_begin && pos < g.pos_end && b % NPART == part;
            const int li = pos / ps;
            page[b] = (in && li < n_list) ? P.pages[C.page_base + li] : 0;
            nbox += in ? 1u : 0u;
        }
        const uint32_t full = bar_full + 8 * s;
        mbar_arrive_expect_tx(full, nbox * NSLAB * kBoxRows * 128u);
        const uint32_t dst0 = ring + s * kStageBytes;
#pragma unroll
        for (int b = 0; b < TT / kBoxRows; ++b) {
            const int pos = tpos + b * kBoxRows;
            if (!(pos + kBoxRows > g.pos_begin && pos < g.pos_end) || b % NPART != part) continue;
            const int slab_z = page[b] * P.n_kv_heads + head;
            const int row0 = pos % ps;
#pragma unroll
            for (int sl = 0; sl < NSLAB; ++sl)
                tma_load_3d(dst0 + sl * kSlabBytes + b * kBoxRows * 128, map, sl * 64, row0, slab_z, full);
        }
    }
    producer_done<STAGES>(bar_full, g.n_tiles, P.status);
    return true;
}

// TMA producer for one operand with d = 128 in page boxes: each 16-row box of
// a tile is one 5-D load of both 64-channel slabs (4 KB, [slab][row]), so a
// tile of TT tokens is TT / 16 boxes at ring + s * TT * 256 + box * 4096.
// Boxes entirely outside the chunk are skipped.
template <int TT, int STAGES>
__device__ bool produce_pages(const DevPlan& P, const DevChunk& C, int head, uint32_t ring, uint32_t bar_full,
                              uint32_t bar_empty, const CUtensorMap* map5) {
    constexpr uint32_t kBox = 2 * kBoxRows * 128;
    constexpr uint32_t kStageBytes = TT * 256;
    const ChunkGeo g = chunk_geo<TT>(C);
    const int ps = P.page_size;
    const int n_list = (g.pos_end - 1) / ps + 1;
    for (int i = 0; i < g.n_tiles; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES) {
            if (!mbar_wait(bar_empty + 8 * s, ((i / STAGES) - 1) & 1, P.status)) {
                drain_ring<STAGES>(bar_full, i, P.status);
                return false;
            }
        }
        const int tpos = g.tile0 + i * TT;
        int page[TT / kBoxRows];
        uint32_t nbox = 0;
#pragma unroll
        for (int b = 0; b < TT / kBoxRows; ++b) {
            const int pos = tpos + b * kBoxRows;
            const bool in = pos + kBoxRows > g.pos_begin && pos < g.pos_end;
            const int li = pos / ps;
            page[b] = (in && li < n_list) ? P.pages[C.page_base + li] : 0;
            nbox += in ? 1u : 0u;
        }
        const uint32_t full = bar_full + 8 * s;
        mbar_arrive_expect_tx(full, nbox * kBox);
        const uint32_t dst0 = ring + s * kStageBytes;
#pragma unroll
        for (int b = 0; b < TT / kBoxRows; ++b) {
            const int pos = tpos + b * kBoxRows;
            if (!(pos + kBoxRows > g.pos_begin && pos < g.pos_end)) continue;
            tma_load_5d(dst0 + b * kBox, map5, 0, pos % ps, head, 0, page[b], full);
        }
    }
    producer_done<STAGES>(bar_full, g.n_tiles, P.status);
    return true;
}

using u64 = unsigned long long;

// Two floats in one 64-bit register pair, for Blackwell's packed f32x2 ALU ops.
__device__ __forceinline__ u64 pk2(float a, float b) {
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk2(u64 r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
    u64 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
    u64 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ u64 add2(u64 a, u64 b) {
    u64 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

}  // namespace dev
}  // namespace pst
