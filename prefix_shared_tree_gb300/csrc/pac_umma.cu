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
// One thread block per (chunk, kv head, block of up to 256 rows), warp-
// specialised (11 warps):
//   warps 0, 10 TMA producers of K and of V: 64-token tiles (16-row page
//               boxes, 128B swizzle) into 3-stage rings; a K stage is
//               refilled as soon as Q K^T has read it, a V stage after P V;
//   warp 1      allocates all 512 tensor-memory columns and issues every MMA
//               from one thread: S = Q K^T (M=128, N=64) and O += P V
//               (M=128, N=d; P from shared memory, V MN-major);
//   warps 2-9   two softmax warpgroups, one thread per row (tensor-memory
//               lane). With more than 128 rows each group owns one 128-row
//               half and both consume every tile; with at most 128 rows the
//               groups take alternate tiles into separate O accumulators
//               and merge them at the end (split-KV inside the block). Either
//               way two softmax warps share each scheduler.
// Softmax works in the log2 domain with 1/sqrt(d) folded into one FMA; the
// running max only moves (and O is rescaled in tensor memory) when it grows
// by more than 2^8, so the result is exact in fp32. P goes to shared memory
// as bf16 hi + lo parts (p = hi + lo to ~2^-16), which keeps the PV product
// as accurate as an fp32 one. (Measured on GB300: with P kept in tensor
// memory instead, the PV MMAs reading it ran at about half rate while the
// softmax warps loaded S and stored P; from shared memory they run at full rate.)
#include "dev_common.cuh"
#include "umma.cuh"

namespace pst {
namespace dev {

constexpr int kUWarps = 11;      // K producer, MMA, 2 x 4 softmax warps, V producer
constexpr int kUStages = 3;
constexpr int kUThreads = kUWarps * 32;
constexpr float kLazyRescale = 8.f;

template <int D>
struct UmmaLayout {
    static constexpr int NSLAB = D / 64;
    static constexpr uint32_t kSlab = kTileTokens * 128;          // one 64-row slab
    static constexpr uint32_t kHalf = NSLAB * kSlab;              // K or V of a stage
    static constexpr uint32_t kStage = 2 * kHalf;
    static constexpr uint32_t kQSlab = 128 * 128;                 // 128 rows x 128 B
    static constexpr uint32_t kRing = kUStages * kStage;
    static constexpr uint32_t kQ = kRing;                         // Q: 2 halves x NSLAB slabs
    static constexpr uint32_t kP = kQ + 2 * NSLAB * kQSlab;       // P[w][hi|lo]: 128 rows x 64 tokens bf16
    static constexpr uint32_t kPBuf = 128 * 128;
    static constexpr uint32_t kXchg = kP + 4 * kPBuf;             // 128 x (m, l) for the split-KV merge
    static constexpr uint32_t kBars = kXchg + 128 * 8;
    // k_full[ST], k_empty[ST], v_full[ST], v_empty[ST], q_ready, s_full[2][2], p_full[2][2],
    // o_done[2], mma_done, tmem slot
    static constexpr int kNumBars = 4 * kUStages + 12;
    static constexpr uint32_t kBytes = kBars + 8 * kNumBars + 16;
    static_assert(kBytes + 1024 <= 232448, "shared memory");
    static constexpr uint32_t kTmemCols = 512;
    // tensor-memory columns: S[w][b] at 128w + 64b, O[w] at 256 + D*w
    __device__ static constexpr uint32_t colS(int w, int b) { return 128 * w + 64 * b; }
    __device__ static constexpr uint32_t colO(int w) { return 256 + D * w; }
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
    const uint32_t ring = sbase, sQ = sbase + L::kQ, sP = sbase + L::kP;
    const uint32_t bars = sbase + L::kBars;
    // K and V stages have separate barriers: a K stage is refilled once Q K^T
    // has read it, a V stage once P V has.
    const uint32_t k_full = bars, k_empty = bars + 8 * kUStages;
    const uint32_t v_full = bars + 16 * kUStages, v_empty = bars + 24 * kUStages;
    const uint32_t q_ready = bars + 32 * kUStages;
    // One p_full per S buffer: a group can then never complete two phases of
    // the same barrier before the MMA warp has waited for the first.
    const uint32_t s_full = q_ready + 8;      // [w][b] at s_full + 8*(2w+b)
    const uint32_t p_full = s_full + 32;      // [w][b] at p_full + 8*(2w+b)
    const uint32_t o_done = p_full + 32;      // [w]
    const uint32_t mma_done = o_done + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kBars + 8 * L::kNumBars);
    float2* xchg = reinterpret_cast<float2*>(base + L::kXchg);

    const DevItem it = P.items[item_off + blockIdx.x];
    const DevChunk C = P.chunks[it.chunk];
    const int head = it.kv_head, rb = it.row_block;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int G = P.group, Hq = P.n_q_heads;
    const int rows_total = C.n_q * G;
    const int row0 = rb * C.r_tile;                 // C.r_tile: 256 or 128 rows per block
    const int rows_here = min(C.r_tile, rows_total - row0);
    const bool split_rows = rows_here > 128;   // mode A: groups own row halves; else alternate tiles

    if (threadIdx.x == 0) {
        for (int s = 0; s < kUStages; ++s) {
            mbar_init(k_full + 8 * s, 1);
            mbar_init(k_empty + 8 * s, 1);
            mbar_init(v_full + 8 * s, 1);
            mbar_init(v_empty + 8 * s, 1);
        }
        mbar_init(q_ready, 256);
        for (int i = 0; i < 4; ++i) {
            mbar_init(s_full + 8 * i, 1);
            mbar_init(p_full + 8 * i, 128);
        }
        for (int w = 0; w < 2; ++w) mbar_init(o_done + 8 * w, 1);
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
    // steps of softmax group w: tiles it consumes, in order
    auto n_steps = [&](int w) { return split_rows ? n : (n - w + 1) / 2; };
    auto tile_of = [&](int w, int k) { return split_rows ? k : 2 * k + w; };

    if (warp == 0 || warp == kUWarps - 1) {
        // ------------------------------------------------------------ TMA producers
        // warp 0 streams K, the last warp streams V, each at its own pace (two
        // lanes of one warp would reconverge and tie the two streams together)
        if (lane == 0) {
            const bool vee = warp != 0;
            prefetch_tmap(vee ? &tv : &tk);
            produce_operand<NSLAB, kUStages, 64>(P, C, head, ring, L::kStage, vee ? v_full : k_full,
                                                 vee ? v_empty : k_empty, vee ? &tv : &tk, vee);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = umma::idesc_bf16_f32(128, kTileTokens, 0, 0);
            constexpr uint32_t idO = umma::idesc_bf16_f32(128, D, 0, 1);   // V is MN-major
            bool ok = mbar_wait(q_ready, 0, P.status);
            umma::fence_after_sync();
            // Descriptors are built once; an MMA only adds a compile-time byte
            // offset (>> 4) to the start-address field, which keeps the single
            // issuing thread far ahead of the tensor pipe. Shared-memory
            // addresses stay below 2^18, so the field never carries over.
            const uint64_t dq_base[2] = {umma::smem_desc_sw128(sQ, 16, 1024),
                                         umma::smem_desc_sw128(sQ + NSLAB * L::kQSlab, 16, 1024)};
            const uint64_t dk_base = umma::smem_desc_sw128(ring, 16, 1024);
            const uint64_t dv_base = umma::smem_desc_sw128(ring + L::kHalf, L::kSlab, 1024);
            const uint64_t dp_base = umma::smem_desc_sw128(sP, 16, 1024);
            auto issue_s = [&](int w, int k, int j) {
                const uint64_t dq = dq_base[split_rows ? w : 0];
                const uint64_t dk = dk_base + (uint64_t)(((j % kUStages) * L::kStage) >> 4);
                const uint32_t dst = tmem + L::colS(w, k & 1);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma::mma_bf16_ss(dst, dq + (((kk / 4) * L::kQSlab + (kk % 4) * 32) >> 4),
                                      dk + (((kk / 4) * L::kSlab + (kk % 4) * 32) >> 4), idS, kk > 0 ? 1u : 0u);
                umma::commit(s_full + 8 * (2 * w + (k & 1)));
            };
            // PV of step k of group w (tile j): O[w] += P_hi V + P_lo V
            auto issue_pv = [&](int w, int k, int j) -> bool {
                if (!mbar_wait(p_full + 8 * (2 * w + (k & 1)), (k >> 1) & 1, P.status)) return false;
                if (!mbar_wait(v_full + 8 * (j % kUStages), (j / kUStages) & 1, P.status)) return false;
                umma::fence_after_sync();
                const uint64_t dv = dv_base + (uint64_t)(((j % kUStages) * L::kStage) >> 4);
                const uint64_t dh = dp_base + (uint64_t)((2 * w * L::kPBuf) >> 4);
                const uint64_t dl = dh + (uint64_t)(L::kPBuf >> 4);
                const uint32_t dst = tmem + L::colO(w);
                const uint32_t acc0 = k > 0 ? 1u : 0u;
#pragma unroll
                for (int kk = 0; kk < kTileTokens / 16; ++kk) {
                    umma::mma_bf16_ss(dst, dh + ((kk * 32) >> 4), dv + ((kk * 2048) >> 4), idO, kk > 0 ? 1u : acc0);
                    umma::mma_bf16_ss(dst, dl + ((kk * 32) >> 4), dv + ((kk * 2048) >> 4), idO, 1u);
                }
                umma::commit(o_done + 8 * w);
                return true;
            };
            for (int j = 0; j < n && ok; ++j) {
                const int s = j % kUStages;
                if (!mbar_wait(k_full + 8 * s, (j / kUStages) & 1, P.status)) { ok = false; break; }
                if (split_rows) {
                    issue_s(0, j, j);
                    issue_s(1, j, j);
                } else {
                    issue_s(j & 1, j >> 1, j);
                }
                umma::commit(k_empty + 8 * s);     // K stage free once these S MMAs complete
                if (j >= 1) {
                    const bool good = split_rows ? (issue_pv(0, j - 1, j - 1) && issue_pv(1, j - 1, j - 1))
                                                 : issue_pv((j - 1) & 1, (j - 1) >> 1, j - 1);
                    if (!good) { ok = false; break; }
                    umma::commit(v_empty + 8 * ((j - 1) % kUStages));
                }
            }
            if (ok && n >= 1) {
                const int j = n - 1;
                bool good = split_rows ? (issue_pv(0, j, j) && issue_pv(1, j, j)) : issue_pv(j & 1, j >> 1, j);
                if (good) umma::commit(v_empty + 8 * (j % kUStages));
            }
            // every MMA issued above has finished before tensor memory is released
            umma::commit(mma_done);
            mbar_wait(mma_done, 0, P.status);
        }
    } else {
        // ------------------------------------------------------------ softmax warpgroups
        const int w = (warp - 2) / 4;                // group 0: warps 2-5, group 1: warps 6-9
        const int r = 32 * (warp % 4) + lane;        // tensor-memory lane = row within the half
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp % 4)) << 16);
        const int rloc = split_rows ? 128 * w + r : r;   // row within the block
        const bool row_ok = rloc < rows_here;
        int qi = 0, gh = 0;
        uint64_t mask = ~0ull;
        if (row_ok) {
            qi = (row0 + rloc) / G;
            gh = (row0 + rloc) % G;
            if (C.mask_base >= 0) mask = P.masks[C.mask_base + qi];
        }
        if (split_rows || w == 0) {
            uint8_t* qdst = base + L::kQ + (split_rows ? w : 0) * NSLAB * L::kQSlab;
            if (row_ok) {
                const int qid = P.chunk_q[C.q_base + qi];
                const uint8_t* src = reinterpret_cast<const uint8_t*>(Q + ((int64_t)qid * Hq + head * G + gh) * D);
#pragma unroll
                for (int ch = 0; ch < NSLAB * 8; ++ch)
                    *reinterpret_cast<uint4*>(qdst + (ch / 8) * L::kQSlab + swz(r, ch % 8)) =
                        *reinterpret_cast<const uint4*>(src + ch * 16);
            } else {
#pragma unroll
                for (int ch = 0; ch < NSLAB * 8; ++ch)
                    *reinterpret_cast<uint4*>(qdst + (ch / 8) * L::kQSlab + swz(r, ch % 8)) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
        }
        mbar_arrive(q_ready);

        const float sl = P.scale_log2;
        const bool masked_chunk = C.mask_base >= 0;
        const bool zero_v = split_rows ? (w == 0) : true;   // one group zeroes a tile's stray V rows
        float m_ref = -INFINITY, l = 0.f;                      // raw-score units for m_ref
        bool ok = true;
        const int nk = n_steps(w);
        for (int k = 0; k < nk; ++k) {
            const int j = tile_of(w, k);
            const int b = k & 1;
            if (!mbar_wait(s_full + 8 * (2 * w + b), (k >> 1) & 1, P.status)) { ok = false; break; }
            umma::fence_after_sync();
            float x[kTileTokens];
            {
                float v[32];
                umma::ld32(lane_addr + L::colS(w, b), v);
#pragma unroll
                for (int c = 0; c < 32; ++c) x[c] = v[c];
                umma::ld32(lane_addr + L::colS(w, b) + 32, v);
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
                    x[c] = vis ? x[c] : -INFINITY;
                    mx = fmaxf(mx, x[c]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < kTileTokens; ++c) mx = fmaxf(mx, x[c]);
            }
            const float mxs = mx * sl;   // scale > 0: max commutes with it
            const bool grow = (m_ref == -INFINITY) ? (mx != -INFINITY) : (mxs > m_ref + kLazyRescale);
            bool rescaled = false;
            if (grow) {
                const float alpha = fast_exp2(m_ref - mxs);   // 0 when nothing was accumulated
                if (k >= 1 && m_ref != -INFINITY) {
                    // O is about to be rescaled: the previous PV of this group must be
                    // done (waited for just below in any case).
                    if (!mbar_wait(o_done + 8 * w, (k - 1) & 1, P.status)) { ok = false; break; }
                    umma::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        umma::ld32(lane_addr + L::colO(w) + 32 * c, o);
                        umma::wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        umma::st32(lane_addr + L::colO(w) + 32 * c, o);
                    }
                    rescaled = true;
                }
                l *= alpha;
                m_ref = mxs;
            }
            const float nmu = m_ref == -INFINITY ? 0.f : -m_ref;
            uint32_t hi[32], lo[32];
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float a = fast_exp2(fmaf(x[2 * c], sl, nmu));
                const float bb = fast_exp2(fmaf(x[2 * c + 1], sl, nmu));
                sum += a + bb;
                const uint32_t h = bf16x2_bits(a, bb);
                hi[c] = h;
                lo[c] = bf16x2_bits(a - __uint_as_float(h << 16), bb - __uint_as_float(h & 0xffff0000u));
            }
            l += sum;
            // P's shared-memory buffer is reused every step: the previous PV of
            // this group must have read it. When S_k has completed, every PV
            // before step k-1 has too, so o_done is at most one phase behind and
            // the parity wait is exact.
            if (k >= 1 && !rescaled) {
                if (!mbar_wait(o_done + 8 * w, (k - 1) & 1, P.status)) { ok = false; break; }
            }
            {
                // row r of P (64 tokens = 128 bytes), K-major with the 128B swizzle
                uint8_t* ph = base + L::kP + 2 * w * L::kPBuf;
                uint8_t* pl = ph + L::kPBuf;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    *reinterpret_cast<uint4*>(ph + swz(r, ch)) =
                        make_uint4(hi[4 * ch], hi[4 * ch + 1], hi[4 * ch + 2], hi[4 * ch + 3]);
                    *reinterpret_cast<uint4*>(pl + swz(r, ch)) =
                        make_uint4(lo[4 * ch], lo[4 * ch + 1], lo[4 * ch + 2], lo[4 * ch + 3]);
                }
            }
            bool zeroed = false;
            if (edge && zero_v) {
                // V rows outside the chunk may hold stale or non-finite values:
                // zero them before the PV of this tile multiplies them by P = 0.
                const int s = j % kUStages;
                if (!mbar_wait(v_full + 8 * s, (j / kUStages) & 1, P.status)) { ok = false; break; }
                if (r < kTileTokens * NSLAB) {          // one 128-byte slab row per thread
                    const int t = r % kTileTokens, sl_i = r / kTileTokens;
                    const int pos = tpos + t;
                    if (pos < geo.pos_begin || pos >= geo.pos_end) {
                        uint8_t* vrow = base + s * L::kStage + L::kHalf + sl_i * L::kSlab + t * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + 16 * c) = make_uint4(0, 0, 0, 0);
                        zeroed = true;
                    }
                }
            }
            if (rescaled) umma::wait_st();
            (void)zeroed;
            fence_proxy_async_smem();   // P (and zeroed V rows) are read by the tensor core
            umma::fence_before_sync();
            mbar_arrive(p_full + 8 * (2 * w + b));
        }
        // ---- epilogue: wait for the MMA warp's final commit (every MMA done)
        bool have = ok && nk >= 1 && mbar_wait(mma_done, 0, P.status);
        if (have) umma::fence_after_sync();
        if (!split_rows) {
            // split-KV inside the block: group 1 hands (m, l) to group 0, which
            // reads both O accumulators (same lanes) and merges them
            if (w == 1) {
                xchg[r] = make_float2(have ? m_ref : -INFINITY, have ? l : 0.f);
                asm volatile("bar.arrive 1, 256;" ::: "memory");
            } else {
                asm volatile("bar.sync 1, 256;" ::: "memory");
            }
        }
        if (have && (split_rows || w == 0)) {
            float m1 = -INFINITY, l1 = 0.f;
            if (!split_rows) {
                const float2 ml = xchg[r];
                m1 = ml.x;
                l1 = ml.y;
            }
            const bool use1 = !split_rows && n >= 2;   // group 1's accumulator is complete (mma_done)
            const float M = fmaxf(m_ref, m1);
            const float Mu = M == -INFINITY ? 0.f : M;
            const float a0 = fast_exp2(m_ref - Mu), a1 = fast_exp2(m1 - Mu);
            const float Lt = l * a0 + l1 * a1;
            const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
            const int64_t prow = (int64_t)C.part_base + (int64_t)qi * Hq + head * G + gh;
            float* dst = P.part_o + prow * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                umma::ld32(lane_addr + L::colO(w) + 32 * c, o);
                umma::wait_ld();
                if (use1) {
                    float o1[32];
                    umma::ld32(lane_addr + L::colO(1) + 32 * c, o1);
                    umma::wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = o[i] * a0 + o1[i] * a1;
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= a0;
                }
                if (row_ok) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(dst + 32 * c + i) =
                            make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
                }
            }
            if (row_ok) P.part_lse[prow] = Lt > 0.f ? M + __log2f(Lt) : -INFINITY;
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
