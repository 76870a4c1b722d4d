// Tensor-core partial attention computation (PAC) for chunks whose
// aggregated query rows (queries x GQA group) form a dense tile (>= 16 rows).
//
// CoDec, "intra-block primitives": K/V of a node chunk is loaded into shared
// memory once and reused by every aggregated query row; the rows are the
// queries that share the node, gathered into shared memory at block start
// (CoDec, "KV cache management": query aggregation, no query tensor is
// prepared in global memory). DEFT's bit causal mask supplies per-row
// visibility inside packed draft-token chunks.
//
// Layout of the work: one thread block per (chunk, kv head, block of 128 rows).
// A producer warp streams 64-token tiles (four 16-row pages per slab,
// 128B-swizzled) with TMA into a 4-stage ring; 8 compute warps each own 16
// rows and run S = Q K^T and O += P V with bf16 mma.sync (fp32 accumulate),
// the online softmax between them in registers (log2 domain, 1/sqrt(d)
// folded into the exponent). In tiles at the chunk edges the V fragments of
// out-of-range rows are cleared in registers, so stale or non-finite page
// rows never meet a zero probability.
#include "dev_common.cuh"

namespace pst {
namespace dev {

constexpr int kTcWarps = 8;
constexpr int kTcStages = 4;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// (a, b) -> bf16 pairs hi = rn(a, b) and lo = rn(a - hi_a, b - hi_b)
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16(a, b);
    const float ha = __uint_as_float(hi << 16), hb = __uint_as_float(hi & 0xffff0000u);
    lo = pack_bf16(a - ha, b - hb);
}

template <int D>
__global__ void __launch_bounds__((kTcWarps + 1) * 32, 1)
pac_tc_kernel(DevPlan P, const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
              const __nv_bfloat16* __restrict__ Q, int item_off) {
    constexpr int NSLAB = D / 64;                       // 128-byte slabs per row
    constexpr uint32_t kSlabBytes = kTileTokens * 128;  // one slab of a 64-token tile
    constexpr uint32_t kHalf = NSLAB * kSlabBytes;
    constexpr uint32_t kStage = 2 * kHalf;
    constexpr uint32_t kQSlab = kTcRowsPerBlock * 128;
    constexpr int KSTEPS = D / 16;

    extern __shared__ uint8_t smem_raw[];
    pdl_launch_dependents();   // the next launch group may take the SMs this grid leaves
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring = smem_u32(base);
    uint8_t* qs = base + kTcStages * kStage;
    const uint32_t qs_u32 = smem_u32(qs);
    uint64_t* bars = reinterpret_cast<uint64_t*>(qs + NSLAB * kQSlab);
    const uint32_t bar_full = smem_u32(bars), bar_empty = smem_u32(bars + kTcStages);

    const DevItem it = P.items[item_off + blockIdx.x];
    const DevChunk C = P.chunks[it.chunk];
    const int head = it.kv_head, rb = it.row_block;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kTcWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == kTcWarps) {
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            if (produce_chunk<NSLAB, kTcStages, 64>(P, C, head, ring, bar_full, bar_empty, &tk, &tv))
                producer_done<kTcStages>(bar_full, chunk_geo(C).n_tiles, P.status);
        }
        return;
    }

    const int G = P.group, Hq = P.n_q_heads;
    const int rows_total = C.n_q * G;
    const int row0 = rb * kTcRowsPerBlock;
    const int rows_here = min(kTcRowsPerBlock, rows_total - row0);

    // ---- gather the block's query rows into shared memory (swizzled like K)
    for (int idx = threadIdx.x; idx < kTcRowsPerBlock * NSLAB * 8; idx += kTcWarps * 32) {
        const int r = idx / (NSLAB * 8), ch = idx % (NSLAB * 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < rows_here) {
            const int row = row0 + r;
            const int qi = row / G, gh = row % G;
            const int qid = P.chunk_q[C.q_base + qi];
            const uint8_t* src = reinterpret_cast<const uint8_t*>(Q + ((int64_t)qid * Hq + head * G + gh) * D);
            v = *reinterpret_cast<const uint4*>(src + ch * 16);
        }
        *reinterpret_cast<uint4*>(qs + (ch / 8) * kQSlab + swz(r, ch % 8)) = v;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kTcWarps * 32) : "memory");

    const bool active = warp * 16 < rows_here;
    const int g = lane / 4, c4 = lane % 4;
    const int rA = warp * 16 + g, rB = rA + 8;  // this thread's two rows
    uint64_t maskA = ~0ull, maskB = ~0ull;
    if (C.mask_base >= 0) {
        if (rA < rows_here) maskA = P.masks[C.mask_base + (row0 + rA) / G];
        if (rB < rows_here) maskB = P.masks[C.mask_base + (row0 + rB) / G];
    }

    uint32_t qa[KSTEPS][4];
    if (active) {
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            const int r = warp * 16 + (lane % 16);
            const int ch = 2 * kk + lane / 16;
            ldsm_x4(qs_u32 + (ch / 8) * kQSlab + swz(r, ch % 8), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
        }
    }

    float oacc[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    const float sl = P.scale_log2;

    const ChunkGeo geo = chunk_geo(C);
    bool ok = true;
    for (int i = 0; i < geo.n_tiles; ++i) {
        const int s = i % kTcStages;
        if (!mbar_wait(bar_full + 8 * s, (i / kTcStages) & 1, P.status)) { ok = false; break; }
        const uint32_t kb = ring + s * kStage;
        const uint32_t vb = kb + kHalf;
        const int tpos = geo.tile0 + i * kTileTokens;
        const bool edge = tpos < geo.pos_begin || tpos + kTileTokens > geo.pos_end;
        if (active) {
            float sacc[8][4];
#pragma unroll
            for (int j = 0; j < 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
                for (int jp = 0; jp < 4; ++jp) {
                    const int idx = lane / 8;
                    const int tok = 16 * jp + (lane % 8) + 8 * (idx / 2);
                    const int ch = 2 * kk + (idx % 2);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + (ch / 8) * kSlabBytes + swz(tok, ch % 8), b0, b1, b2, b3);
                    mma_bf16(sacc[2 * jp], qa[kk], b0, b1);
                    mma_bf16(sacc[2 * jp + 1], qa[kk], b2, b3);
                }
            }
            // mask and row maxima (raw scores; the scale is positive)
            float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = 8 * j + 2 * c4 + e;
                    const int pos = tpos + col;
                    const int t = pos - geo.pos_begin;
                    const bool inr = pos >= geo.pos_begin && pos < geo.pos_end;
                    const bool vA = inr && (t >= 64 || ((maskA >> (t & 63)) & 1ull));
                    const bool vB = inr && (t >= 64 || ((maskB >> (t & 63)) & 1ull));
                    sacc[j][e] = vA ? sacc[j][e] * sl : -INFINITY;
                    sacc[j][2 + e] = vB ? sacc[j][2 + e] * sl : -INFINITY;
                    mxA = fmaxf(mxA, sacc[j][e]);
                    mxB = fmaxf(mxB, sacc[j][2 + e]);
                }
            }
            mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
            mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
            mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
            mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
            const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
            const float uA = nA == -INFINITY ? 0.f : nA, uB = nB == -INFINITY ? 0.f : nB;
            const float aA = fast_exp2(mA - uA), aB = fast_exp2(mB - uB);
            mA = nA;
            mB = nB;
            float sumA = 0.f, sumB = 0.f;
            // P enters the PV product as bf16 hi + lo parts (p = hi + lo to about
            // 2^-16 relative), so rounding P to bf16 costs no accuracy.
            uint32_t pa[4][4], pl[4][4];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float p0 = fast_exp2(sacc[j][0] - uA), p1 = fast_exp2(sacc[j][1] - uA);
                const float p2 = fast_exp2(sacc[j][2] - uB), p3 = fast_exp2(sacc[j][3] - uB);
                sumA += p0 + p1;
                sumB += p2 + p3;
                const int kk = j / 2, hi = j % 2;
                split_bf16(p0, p1, pa[kk][hi * 2 + 0], pl[kk][hi * 2 + 0]);
                split_bf16(p2, p3, pa[kk][hi * 2 + 1], pl[kk][hi * 2 + 1]);
            }
            lA = lA * aA + sumA;
            lB = lB * aB + sumB;
#pragma unroll
            for (int j = 0; j < D / 8; ++j) {
                oacc[j][0] *= aA;
                oacc[j][1] *= aA;
                oacc[j][2] *= aB;
                oacc[j][3] *= aB;
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                // At the chunk edges, V rows outside the chunk may hold stale or
                // non-finite data: clear their halves of the B fragments (this
                // thread holds tokens 16kk+2c, +1 in b0/b2 and 16kk+8+2c, +1 in b1/b3).
                uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
                if (edge) {
                    const int p0 = tpos + 16 * kk + 2 * c4;
                    auto in = [&](int p) { return p >= geo.pos_begin && p < geo.pos_end; };
                    mlo = (in(p0) ? 0x0000ffffu : 0u) | (in(p0 + 1) ? 0xffff0000u : 0u);
                    mhi = (in(p0 + 8) ? 0x0000ffffu : 0u) | (in(p0 + 9) ? 0xffff0000u : 0u);
                }
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    const int idx = lane / 8;
                    const int tok = 16 * kk + (lane % 8) + 8 * (idx % 2);
                    const int ch = 2 * dp + idx / 2;
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vb + (ch / 8) * kSlabBytes + swz(tok, ch % 8), b0, b1, b2, b3);
                    b0 &= mlo;
                    b1 &= mhi;
                    b2 &= mlo;
                    b3 &= mhi;
                    mma_bf16(oacc[2 * dp], pa[kk], b0, b1);
                    mma_bf16(oacc[2 * dp + 1], pa[kk], b2, b3);
                    mma_bf16(oacc[2 * dp], pl[kk], b0, b1);
                    mma_bf16(oacc[2 * dp + 1], pl[kk], b2, b3);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
    if (!ok || !active) return;

    // ---- normalise and write this block's partial outputs
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = half ? rB : rA;
        if (r >= rows_here) continue;
        const float l = half ? lB : lA, m = half ? mB : mA;
        const int row = row0 + r;
        const int qi = row / G, gh = row % G;
        const int64_t prow = (int64_t)C.part_base + (int64_t)qi * Hq + head * G + gh;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float* dst = P.part_o + prow * D;
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            float2 v = make_float2(oacc[j][2 * half] * inv, oacc[j][2 * half + 1] * inv);
            *reinterpret_cast<float2*>(dst + 8 * j + 2 * c4) = v;
        }
        if (c4 == 0) P.part_lse[prow] = l > 0.f ? m + __log2f(l) : -INFINITY;
    }
}

template <int D>
size_t tc_smem_bytes() {
    constexpr int NSLAB = D / 64;
    return 1024 + kTcStages * 2 * NSLAB * kTileTokens * 128 + NSLAB * kTcRowsPerBlock * 128 + 2 * kTcStages * 8;
}

template <int D>
cudaError_t launch_tc_t(const DevPlan& P, const CUtensorMap* tk, const CUtensorMap* tv, const void* Q,
                        int n_items, int item_off, cudaStream_t st, bool pdl) {
    const size_t smem = tc_smem_bytes<D>();
    static DeviceOnce once;   // per device
    cudaError_t e = per_device(once, nullptr, nullptr, [&](int, int* a, int*) {
        *a = 1;
        return cudaFuncSetAttribute(pac_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (e != cudaSuccess) return e;
    return launch_kernel(pac_tc_kernel<D>, dim3(n_items), dim3((kTcWarps + 1) * 32), smem, st, pdl, P, *tk, *tv,
                         static_cast<const __nv_bfloat16*>(Q), item_off);
}

}  // namespace dev

cudaError_t launch_pac_tc(const DevPlan& P, const void* tk, const void* tv, const void* Q, int n_items,
                          int item_off, cudaStream_t st, bool pdl) {
    const CUtensorMap* k = static_cast<const CUtensorMap*>(tk);
    const CUtensorMap* v = static_cast<const CUtensorMap*>(tv);
    if (P.d == 128) return dev::launch_tc_t<128>(P, k, v, Q, n_items, item_off, st, pdl);
    return dev::launch_tc_t<64>(P, k, v, Q, n_items, item_off, st, pdl);
}

}  // namespace pst
