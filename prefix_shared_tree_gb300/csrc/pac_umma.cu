// Tensor-core partial attention computation (PAC) on the 5th-generation
// tensor cores (tcgen05 + tensor memory) for chunks whose aggregated query
// rows (queries x GQA group) form a dense tile.
//
// CoDec, "intra-block primitives": the node chunk's K/V tiles are loaded into
// shared memory once and shared by all the node's aggregated query rows,
// which are gathered into shared memory when the block starts (CoDec, "KV
// cache management"); the PAC emits a partial output with its softmax
// statistics for the POR merge. DEFT's bit causal mask gives per-row
// visibility inside packed draft-token chunks.
//
// One thread block per (chunk, kv head, block of 128 rows), warp-specialised:
//   warp 0      TMA producer: 64-token K/V tiles (16-row page boxes, 128B
//               swizzle) into a 4-stage ring;
//   warp 1      allocates tensor memory and issues the MMAs from one thread:
//               S_j = Q K_j^T (M=128, N=64, fp32 in tensor memory, double
//               buffered) and O += P_j V_j (M=128, N=d) with V read MN-major;
//   warps 2-5   softmax, one thread per row (= tensor-memory lane): read S_j,
//               mask, online max/sum in the log2 domain, write P_j to shared
//               memory as bf16 hi + lo parts (so rounding P costs no
//               accuracy). The running max is only moved (and O rescaled in
//               tensor memory) when it grows by more than 2^8, which keeps
//               every exponent <= 8 and the result exact in fp32.
// The MMA warp issues S_{j+1} before PV_j, so the softmax of one tile
// overlaps the tensor-core work of the previous one.
#include "dev_common.cuh"
#include "umma.cuh"

namespace pst {
namespace dev {

constexpr int kUWarps = 6;       // producer, MMA, 4 softmax warps
constexpr int kUStages = 4;
constexpr int kUThreads = kUWarps * 32;
constexpr float kLazyRescale = 8.f;

template <int D>
struct UmmaLayout {
    static constexpr int NSLAB = D / 64;
    static constexpr uint32_t kSlab = kTileTokens * 128;          // one 64-row slab
    static constexpr uint32_t kHalf = NSLAB * kSlab;              // K or V of a stage
    static constexpr uint32_t kStage = 2 * kHalf;
    static constexpr uint32_t kQSlab = kTcRowsPerBlock * 128;
    static constexpr uint32_t kRing = kUStages * kStage;
    static constexpr uint32_t kQ = kRing;                         // Q: NSLAB x 128 rows x 128 B
    static constexpr uint32_t kPhi = kQ + NSLAB * kQSlab;         // P hi: 128 rows x 64 tokens bf16
    static constexpr uint32_t kPlo = kPhi + kTcRowsPerBlock * 128;
    static constexpr uint32_t kBars = kPlo + kTcRowsPerBlock * 128;
    // barriers: kv_full[ST], kv_empty[ST], q_ready, s_full[2], p_full, o_done, mma_done, tmem slot
    static constexpr uint32_t kBytes = kBars + 8 * (2 * kUStages + 6) + 16;
    static constexpr uint32_t kTmemCols = 256;                    // S0 | S1 | O (<= 128 columns)
    static constexpr uint32_t kColS = 0, kColO = 128;
};

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int D>
__global__ void __launch_bounds__(kUThreads, 1)
pac_umma_kernel(DevPlan P, const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                const __nv_bfloat16* __restrict__ Q, int item_off) {
    using L = UmmaLayout<D>;
    constexpr int NSLAB = L::NSLAB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(base);
    const uint32_t ring = sbase, sQ = sbase + L::kQ, sPhi = sbase + L::kPhi, sPlo = sbase + L::kPlo;
    const uint32_t bars = sbase + L::kBars;
    const uint32_t kv_full = bars, kv_empty = bars + 8 * kUStages;
    const uint32_t q_ready = bars + 16 * kUStages;
    const uint32_t s_full = q_ready + 8;            // 2 barriers
    const uint32_t p_full = s_full + 16, o_done = p_full + 8, mma_done = o_done + 8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kBars + 8 * (2 * kUStages + 6));

    const DevItem it = P.items[item_off + blockIdx.x];
    const DevChunk C = P.chunks[it.chunk];
    const int head = it.kv_head, rb = it.row_block;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kUStages; ++s) {
            mbar_init(kv_full + 8 * s, 1);
            mbar_init(kv_empty + 8 * s, 1);
        }
        mbar_init(q_ready, 128);
        mbar_init(s_full, 1);
        mbar_init(s_full + 8, 1);
        mbar_init(p_full, 128);
        mbar_init(o_done, 1);
        mbar_init(mma_done, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        umma::tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const ChunkGeo geo = chunk_geo(C);
    const int n = geo.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            produce_chunk<NSLAB, kUStages, 64>(P, C, head, ring, kv_full, kv_empty, &tk, &tv);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = umma::idesc_bf16_f32(128, kTileTokens, 0, 0);
            constexpr uint32_t idO = umma::idesc_bf16_f32(128, D, 0, 1);
            bool ok = mbar_wait(q_ready, 0, P.status);
            umma::fence_after_sync();
            auto issue_pv = [&](int jj) {
                const uint32_t vb = ring + (jj % kUStages) * L::kStage + L::kHalf;
#pragma unroll
                for (int kk = 0; kk < kTileTokens / 16; ++kk) {
                    const uint64_t dv = umma::smem_desc_sw128(vb + kk * 2048, L::kSlab, 1024);
                    const uint64_t dh = umma::smem_desc_sw128(sPhi + kk * 32, 16, 1024);
                    const uint64_t dl = umma::smem_desc_sw128(sPlo + kk * 32, 16, 1024);
                    umma::mma_bf16_ss(tmem + L::kColO, dh, dv, idO, (jj > 0 || kk > 0) ? 1u : 0u);
                    umma::mma_bf16_ss(tmem + L::kColO, dl, dv, idO, 1u);
                }
                umma::commit(o_done);
                umma::commit(kv_empty + 8 * (jj % kUStages));
            };
            for (int j = 0; j < n && ok; ++j) {
                const int s = j % kUStages;
                if (!mbar_wait(kv_full + 8 * s, (j / kUStages) & 1, P.status)) { ok = false; break; }
                const uint32_t kb = ring + s * L::kStage;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t dq = umma::smem_desc_sw128(sQ + (kk / 4) * L::kQSlab + (kk % 4) * 32, 16, 1024);
                    const uint64_t dk = umma::smem_desc_sw128(kb + (kk / 4) * L::kSlab + (kk % 4) * 32, 16, 1024);
                    umma::mma_bf16_ss(tmem + L::kColS + (j & 1) * kTileTokens, dq, dk, idS, kk > 0 ? 1u : 0u);
                }
                umma::commit(s_full + 8 * (j & 1));
                if (j >= 1) {
                    if (!mbar_wait(p_full, (j - 1) & 1, P.status)) { ok = false; break; }
                    umma::fence_after_sync();
                    issue_pv(j - 1);
                }
            }
            if (ok && n >= 1) {
                if (mbar_wait(p_full, (n - 1) & 1, P.status)) {
                    umma::fence_after_sync();
                    issue_pv(n - 1);
                }
            }
            // every MMA issued above has finished before tensor memory is released
            umma::commit(mma_done);
            mbar_wait(mma_done, 0, P.status);
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int r = 32 * (warp % 4) + lane;       // row = tensor-memory lane
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp % 4)) << 16);
        const int G = P.group, Hq = P.n_q_heads;
        const int rows_total = C.n_q * G;
        const int row0 = rb * kTcRowsPerBlock;
        const int rows_here = min(kTcRowsPerBlock, rows_total - row0);
        const bool row_ok = r < rows_here;
        int qi = 0, gh = 0;
        uint64_t mask = ~0ull;
        {
            uint8_t* qdst = base + L::kQ;
            if (row_ok) {
                qi = (row0 + r) / G;
                gh = (row0 + r) % G;
                const int qid = P.chunk_q[C.q_base + qi];
                const uint8_t* src = reinterpret_cast<const uint8_t*>(Q + ((int64_t)qid * Hq + head * G + gh) * D);
                if (C.mask_base >= 0) mask = P.masks[C.mask_base + qi];
#pragma unroll
                for (int ch = 0; ch < NSLAB * 8; ++ch)
                    *reinterpret_cast<uint4*>(qdst + (ch / 8) * L::kQSlab + swz(r, ch % 8)) =
                        *reinterpret_cast<const uint4*>(src + ch * 16);
            } else {
#pragma unroll
                for (int ch = 0; ch < NSLAB * 8; ++ch)
                    *reinterpret_cast<uint4*>(qdst + (ch / 8) * L::kQSlab + swz(r, ch % 8)) = make_uint4(0, 0, 0, 0);
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(q_ready);

        const float sl = P.scale_log2;
        const bool masked_chunk = C.mask_base >= 0;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            if (!mbar_wait(s_full + 8 * (j & 1), (j >> 1) & 1, P.status)) { ok = false; break; }
            umma::fence_after_sync();
            float x[kTileTokens];
            {
                float v[32];
                umma::ld32(lane_addr + L::kColS + (j & 1) * kTileTokens, v);
                umma::wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] = v[c];
                umma::ld32(lane_addr + L::kColS + (j & 1) * kTileTokens + 32, v);
                umma::wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) x[32 + c] = v[c];
            }
            const int tpos = geo.tile0 + j * kTileTokens;
            const bool edge = tpos < geo.pos_begin || tpos + kTileTokens > geo.pos_end;
            float mx = -INFINITY;
            if (edge || masked_chunk) {
#pragma unroll
                for (int c = 0; c < kTileTokens; ++c) {
                    const int pos = tpos + c;
                    const int t = pos - geo.pos_begin;
                    const bool vis = pos >= geo.pos_begin && pos < geo.pos_end && (t >= 64 || ((mask >> (t & 63)) & 1ull));
                    x[c] = vis ? x[c] * sl : -INFINITY;
                    mx = fmaxf(mx, x[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < kTileTokens; ++c) {
                    x[c] *= sl;
                    mx = fmaxf(mx, x[c]);
                }
            }
            // PV_{j-1} must have finished: it reads the P buffer and writes O
            if (j >= 1) {
                if (!mbar_wait(o_done, (j - 1) & 1, P.status)) { ok = false; break; }
                umma::fence_after_sync();
            }
            const bool grow = (m_ref == -INFINITY) ? (mx != -INFINITY) : (mx > m_ref + kLazyRescale);
            bool rescaled = false;
            if (grow) {
                const float alpha = fast_exp2(m_ref - mx);   // 0 when nothing was accumulated
                if (j >= 1 && m_ref != -INFINITY) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        umma::ld32(lane_addr + L::kColO + 32 * c, o);
                        umma::wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        umma::st32(lane_addr + L::kColO + 32 * c, o);
                    }
                    rescaled = true;
                }
                l *= alpha;
                m_ref = mx;
            }
            const float mu = m_ref == -INFINITY ? 0.f : m_ref;
            uint8_t* phi = base + L::kPhi;
            uint8_t* plo = base + L::kPlo;
            float sum = 0.f;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint32_t h[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a = fast_exp2(x[8 * ch + 2 * k] - mu);
                    const float b = fast_exp2(x[8 * ch + 2 * k + 1] - mu);
                    sum += a + b;
                    h[k] = bf16x2_bits(a, b);
                    lo[k] = bf16x2_bits(a - __uint_as_float(h[k] << 16), b - __uint_as_float(h[k] & 0xffff0000u));
                }
                *reinterpret_cast<uint4*>(phi + swz(r, ch)) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4*>(plo + swz(r, ch)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            l += sum;
            if (edge) {
                // V rows outside the chunk may hold stale or non-finite values:
                // zero them before PV_j multiplies them by P = 0.
                const int s = j % kUStages;
                if (!mbar_wait(kv_full + 8 * s, (j / kUStages) & 1, P.status)) { ok = false; break; }
                if (r < kTileTokens * NSLAB) {
                    const int t = r % kTileTokens, sl_i = r / kTileTokens;
                    const int pos = tpos + t;
                    if (pos < geo.pos_begin || pos >= geo.pos_end) {
                        uint8_t* vrow = base + s * L::kStage + L::kHalf + sl_i * L::kSlab + t * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + 16 * c) = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            if (rescaled) umma::wait_st();
            fence_proxy_async_smem();
            umma::fence_before_sync();
            mbar_arrive(p_full);
        }
        // ---- epilogue: O / l to the partial-output rows
        if (ok && n >= 1 && mbar_wait(o_done, (n - 1) & 1, P.status)) {
            umma::fence_after_sync();
            const int64_t prow = (int64_t)C.part_base + (int64_t)qi * Hq + head * G + gh;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            float* dst = P.part_o + prow * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                umma::ld32(lane_addr + L::kColO + 32 * c, o);
                umma::wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(dst + 32 * c + i) =
                            make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
                }
            }
            if (row_ok) P.part_lse[prow] = l > 0.f ? m_ref + __log2f(l) : -INFINITY;
        }
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int D>
cudaError_t launch_umma_t(const DevPlan& P, const CUtensorMap* tk, const CUtensorMap* tv, const void* Q, int n_items,
                          int item_off, cudaStream_t st) {
    const size_t smem = 1024 + UmmaLayout<D>::kBytes;
    static bool attr_set = false;  // once per process (single device per process)
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(pac_umma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    pac_umma_kernel<D><<<n_items, kUThreads, smem, st>>>(P, *tk, *tv, static_cast<const __nv_bfloat16*>(Q), item_off);
    return cudaGetLastError();
}

}  // namespace dev

cudaError_t launch_pac_umma(const DevPlan& P, const void* tk, const void* tv, const void* Q, int n_items, int item_off,
                            cudaStream_t st) {
    const CUtensorMap* k = static_cast<const CUtensorMap*>(tk);
    const CUtensorMap* v = static_cast<const CUtensorMap*>(tv);
    if (P.d == 128) return dev::launch_umma_t<128>(P, k, v, Q, n_items, item_off, st);
    return dev::launch_umma_t<64>(P, k, v, Q, n_items, item_off, st);
}

}  // namespace pst
