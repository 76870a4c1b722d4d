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
// specialised (the producer/MMA warpgroup, then the softmax warpgroups):
//   warps 0, 3  TMA producers of K (alternate 16-row page boxes), warp 2 of
//               V (both 64-channel slabs of a page box in one load; d = 128):
//               128-token tiles, 128B swizzle, each operand in its own ring;
//               a K stage is refilled as soon as Q K^T has read it, a V stage
//               after P V;
//   warp 1      allocates all 512 tensor-memory columns and issues every MMA
//               from one thread: S = Q K^T (M=128, N=128, Q and K from shared
//               memory) and O += P V (M=128, N=d, P from tensor memory, V
//               MN-major from shared memory);
//   softmax warpgroups, one thread per tensor-memory lane: four above 128
//               rows (warps 4-19), two at most (warps 4-11). Above 128 rows
//               the MMA warp alternates between the two 128-row halves (P V
//               and S of half 0, then of half 1) and all four groups work on
//               each half as soon as its S is ready: group w takes S columns
//               [32w, 32w + 32), the row max (and, for the precision guard
//               below, the row sum so far) is combined from the groups'
//               values exchanged through shared memory, so a half's softmax
//               overlaps the other half's MMAs. With at most 128 rows the two
//               groups take alternate tiles into separate S buffers and O
//               accumulators and merge at the end (split-KV inside the block).
// The first warpgroup hands registers to the softmax warpgroups
// (setmaxnreg), which hold a whole 128-column row of S in registers.
// Tensor memory: S of half w in columns [128w, 128w+128), O of half w in
// [256 + d*w, 256 + d*w + d). The softmax overwrites S with P (bf16, two per
// column); the next S of that half is issued after the P V that reads it, and
// tcgen05 MMAs from one thread run in issue order.
// Softmax works in the log2 domain with 1/sqrt(d) folded into one FMA; the
// running max only moves (and O is rescaled in tensor memory) when it grows
// by more than 2^8, so the result is exact in fp32.
// Precision of P in P V. The EXACT instance (chunks of nodes shorter than the
// plan's p_bf16_min_tokens) splits every weight into a bf16 hi part and the
// bf16 remainder lo (p = hi + lo to ~2^-16) and multiplies V by both, which
// makes P V as accurate as an fp32 product. The other instance rounds each
// weight once to bf16 (relative error at most 2^-9) and keeps the row sum of
// the rounded weights, so O is an exact convex combination of V rows with
// slightly perturbed weights: a weight's error moves O by at most its share
// p (1 - p) of 2^-9 |v - O|, and the errors of many small weights, random in
// sign, average out. A weight that holds a large share of its row's sum so
// far (above kExactShare of it) is made exact instead: the running max moves
// to it (rescaling O), so it becomes 2^0 = 1 exactly. Scores a row may not
// see (tile edges, bit causal masks) are set to -inf in tensor memory before
// the row is loaded, which keeps masking out of the hot code.
#include "dev_common.cuh"
#include "umma.cuh"

namespace pst {
namespace dev {

// Warps: the producer/MMA warpgroup (K producer, MMA, V producer, K producer), then
// the softmax warpgroups: four above 128 rows (each takes 32 columns of a row
// half, so a half's softmax runs on four warps per scheduler), two at most.
// Registers per thread: at launch (the __launch_bounds__ cap), then after
// setmaxnreg in the producer/MMA warpgroup and in the softmax warpgroups; a
// split never exceeds the launch total.
template <bool SPLIT>
struct UWarps {
    static constexpr int kGroups = SPLIT ? 4 : 2;
    static constexpr int kWarps = 4 + 4 * kGroups;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kRegsLaunch = SPLIT ? 96 : 168;
    static constexpr int kRegsMma = SPLIT ? 160 : 104;       // producer/MMA warpgroup
    static constexpr int kRegsSoftmax = SPLIT ? 80 : 200;    // each softmax warpgroup
    static_assert(128 * kRegsMma + 128 * kGroups * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");
};
constexpr int kUT = kTcTileTokens;   // tokens per tile
constexpr int kKProducers = 2;       // threads issuing a K tile's TMA loads
constexpr float kLazyRescale = 8.f;
// A weight above this share of its row's softmax sum so far (itself included)
// is made exact (see the precision note above).
constexpr float kExactShare = 0.125f;

template <int D>
struct UmmaLayout {
    static constexpr int NSLAB = D / 64;
    static constexpr uint32_t kSlab = kUT * 128;                   // 128 token rows x 128 B
    static constexpr uint32_t kOp = NSLAB * kSlab;                 // one K or V tile
    static constexpr int KST = D == 128 ? 2 : 4;                   // K stages
    static constexpr int VST = D == 128 ? 2 : 4;                   // V stages
    // V tiles are stored by page box: [box][slab][16 rows] (with d = 64 this
    // is the K layout); a P V MMA takes one box (16 tokens)
    static constexpr uint32_t kVBox = NSLAB * kBoxRows * 128;
    static constexpr uint32_t kVSlab = kBoxRows * 128;             // slab stride inside a box
    static constexpr uint32_t kQSlab = 128 * 128;                  // 128 rows x 128 B
    static constexpr uint32_t kK = 0;
    static constexpr uint32_t kV = kK + KST * kOp;
    static constexpr uint32_t kQ = kV + VST * kOp;                 // 2 halves x NSLAB slabs
    static constexpr uint32_t kXchg = kQ + 2 * NSLAB * kQSlab;     // 128 x (m, l) for the split-KV merge
    static constexpr uint32_t kRed = kXchg + 128 * 8;              // [2][4][128] row maxima, then [2][4][128] sums
    static constexpr uint32_t kLRed = kRed + 2048 * 4;             // [2][4][128] row sums of the earlier tiles
    static constexpr uint32_t kBars = kLRed + 1024 * 4;
    // k_full[KST], k_empty[KST], v_full[VST], v_empty[VST], q_ready, s_full[2], p_full[2], mma_done,
    // xchg[2], lfin
    static constexpr int kNumBars = 2 * KST + 2 * VST + 10;
    static constexpr uint32_t kBytes = kBars + 8 * kNumBars + 16;
    static_assert(kBytes + 1024 <= 232448, "shared memory");
    static constexpr uint32_t kTmemCols = 512;
    __device__ static constexpr uint32_t colS(int w) { return 128 * w; }
    __device__ static constexpr uint32_t colO(int w) { return 256 + D * w; }
};

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// ---- softmax pieces (one thread = one tensor-memory lane = one row)

// NC columns of this lane from tensor memory into registers.
template <int NC>
__device__ __forceinline__ void ld_cols(uint32_t taddr, float (&x)[NC]) {
#pragma unroll
    for (int q = 0; q < NC / 32; ++q) {
        float v[32];
        umma::ld32(taddr + 32 * q, v);
#pragma unroll
        for (int c = 0; c < 32; ++c) x[32 * q + c] = v[c];
    }
    umma::wait_ld();
}

// Max of NC values: four independent chains of three-input maxima.
template <int NC>
__device__ __forceinline__ float row_max(const float (&x)[NC]) {
    float acc[4];
#pragma unroll
    for (int a = 0; a < 4; ++a) acc[a] = fmaxf(x[a], x[4 + a]);
#pragma unroll
    for (int c = 8; c < NC; c += 8) {
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a] = fmax3(acc[a], x[c + a], x[c + 4 + a]);
    }
    return fmaxf(fmax3(acc[0], acc[1], acc[2]), acc[3]);
}

// Scores this row may not see become -inf in tensor memory, 32 columns at a
// time, over the NC columns starting at col0 of the tile. [c_lo, c_hi) is the
// chunk's token range in tile columns; in a masked chunk, bit t of `mask` is
// chunk token t.
template <int NC>
__device__ __forceinline__ void mask_in_tmem(uint32_t s_addr, int col0, int c_lo, int c_hi, uint64_t mask,
                                             bool masked_chunk) {
#pragma unroll 1
    for (int c0 = col0; c0 < col0 + NC; c0 += 32) {
        if (!masked_chunk && c0 >= c_lo && c0 + 32 <= c_hi) continue;
        float v[32];
        umma::ld32(s_addr + c0, v);
        umma::wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int t = c0 + c - c_lo;   // token index in the chunk
            const bool vis = t >= 0 && c0 + c < c_hi && (t >= kMaskTokens || ((mask >> (t & 63)) & 1ull));
            v[c] = vis ? v[c] : -INFINITY;
        }
        umma::st32(s_addr + c0, v);
    }
    umma::wait_st();
}

// P = 2^(x*sl - m) for NC scores into tensor memory as bf16 pairs (P[2i],
// P[2i+1] in one column): at p_hi, and with EXACT the remainder p - hi at
// p_lo. Returns the row sum of the weights P V multiplies: the unrounded ones
// with EXACT (hi + lo), the rounded ones (hi) without.
template <int NC, bool EXACT>
__device__ __forceinline__ float softmax_p(const float (&x)[NC], float sl, float nmu, uint32_t p_hi, uint32_t p_lo) {
    const u64 sl2 = pk2(sl, sl), nmu2 = pk2(nmu, nmu);
    u64 sum2[4] = {0ull, 0ull, 0ull, 0ull};   // independent add chains
    if (!EXACT) {
#pragma unroll
        for (int q = 0; q < NC / 32; ++q) {
            uint32_t hi[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                float a, b;
                upk2(fma2(pk2(x[32 * q + 2 * c], x[32 * q + 2 * c + 1]), sl2, nmu2), a, b);
                a = fast_exp2(a);
                b = fast_exp2(b);
                hi[c] = bf16x2_bits(a, b);
                sum2[c & 3] = add2(sum2[c & 3], pk2(bf16lo(hi[c]), bf16hi(hi[c])));
            }
            umma::st16(p_hi + 16 * q, hi);
        }
    } else {
#pragma unroll
        for (int q = 0; q < NC / 16; ++q) {
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                float a, b;
                upk2(fma2(pk2(x[16 * q + 2 * c], x[16 * q + 2 * c + 1]), sl2, nmu2), a, b);
                a = fast_exp2(a);
                b = fast_exp2(b);
                sum2[c & 3] = add2(sum2[c & 3], pk2(a, b));
                hi[c] = bf16x2_bits(a, b);
                lo[c] = bf16x2_bits(a - __uint_as_float(hi[c] << 16), b - __uint_as_float(hi[c] & 0xffff0000u));
            }
            umma::st8(p_hi + 8 * q, hi);
            umma::st8(p_lo + 8 * q, lo);
        }
    }
    float s0, s1;
    upk2(add2(add2(sum2[0], sum2[1]), add2(sum2[2], sum2[3])), s0, s1);
    return s0 + s1;
}

// O columns [taddr, taddr + NC) of this row *= alpha (whole warp).
template <int NC>
__device__ __forceinline__ void scale_o(uint32_t taddr, float alpha) {
    static_assert(NC % 16 == 0, "O column block");
    if constexpr (NC % 32 == 0) {
#pragma unroll 1
        for (int c = 0; c < NC; c += 32) {
            float o[32];
            umma::ld32(taddr + c, o);
            umma::wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            umma::st32(taddr + c, o);
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < NC; c += 16) {
            uint32_t o[16];
            umma::ld16(taddr + c, o);
            umma::wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            umma::st16(taddr + c, o);
        }
    }
}

// V rows outside the chunk may hold stale or non-finite values: zero them
// (thread r owns token row r of tile j) before P V multiplies them by P = 0.
// False if the wait for the tile gave up.
template <typename L>
__device__ __forceinline__ bool zero_stray_v(const DevPlan& P, uint8_t* base, const ChunkGeo& geo, int tpos, int j, int r,
                                             uint32_t v_full) {
    const int s = j % L::VST;
    if (!mbar_wait(v_full + 8 * s, (j / L::VST) & 1, P.status)) return false;
    const int pos = tpos + r;
    if (pos < geo.pos_begin || pos >= geo.pos_end) {
#pragma unroll
        for (int sl_i = 0; sl_i < L::NSLAB; ++sl_i) {
            uint8_t* vrow = base + L::kV + s * L::kOp + (r / kBoxRows) * L::kVBox + sl_i * L::kVSlab + (r % kBoxRows) * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + 16 * c) = make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();   // zeroed V rows are read by the tensor core
    return true;
}

template <int D, bool EXACT, bool SPLIT>
__global__ void __launch_bounds__(UWarps<SPLIT>::kThreads, 1)
pac_umma_kernel(DevPlan P, const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                const __nv_bfloat16* __restrict__ Q, int item_off, const __grid_constant__ CUtensorMap tq, int q_tma) {
    using L = UmmaLayout<D>;
    constexpr int NSLAB = L::NSLAB;
    constexpr int KST = L::KST, VST = L::VST;
    extern __shared__ uint8_t smem_raw[];
    pdl_launch_dependents();   // the next launch group may take the SMs this grid leaves
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(base);
    const uint32_t sK = sbase + L::kK, sV = sbase + L::kV, sQ = sbase + L::kQ;
    const uint32_t bars = sbase + L::kBars;
    const uint32_t k_full = bars, k_empty = k_full + 8 * KST;
    const uint32_t v_full = k_empty + 8 * KST, v_empty = v_full + 8 * VST;
    const uint32_t q_ready = v_empty + 8 * VST;
    const uint32_t s_full = q_ready + 8;      // [w]
    const uint32_t p_full = s_full + 16;      // [w]
    const uint32_t mma_done = p_full + 16;
    const uint32_t xchg_bar = mma_done + 8;   // [half]: both groups' row maxima of a half are in
    const uint32_t lfin_bar = xchg_bar + 16;  // both groups' row sums are in
    const uint32_t q_full = lfin_bar + 8;     // the TMA copy of Q has landed
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
    // SPLIT instance: more than 128 rows in the block (both groups on both row
    // halves); otherwise the groups alternate tiles. The plan launches each
    // item with the instance its row count needs.
    constexpr bool split_rows = SPLIT;
    if ((rows_here > 128) != SPLIT) {
        if (threadIdx.x == 0) atomicOr(P.status, kStatusBadIndex);
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < KST; ++s) {
            mbar_init(k_full + 8 * s, kKProducers);
            mbar_init(k_empty + 8 * s, 1);
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(v_full + 8 * s, 1);
            mbar_init(v_empty + 8 * s, 1);
        }
        mbar_init(q_ready, 128 * UWarps<SPLIT>::kGroups);
        mbar_init(q_full, 1);
        for (int w = 0; w < 2; ++w) {
            mbar_init(s_full + 8 * w, 1);
            // above 128 rows every group works on each half
            mbar_init(p_full + 8 * w, split_rows ? 128 * UWarps<SPLIT>::kGroups : 128);
            mbar_init(xchg_bar + 8 * w, 128 * UWarps<SPLIT>::kGroups);
        }
        mbar_init(mma_done, 1);
        mbar_init(lfin_bar, 128 * UWarps<SPLIT>::kGroups);
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
    const ChunkGeo geo = chunk_geo<kUT>(C);
    // When the block's queries have consecutive ids (the chunk's query list
    // is ascending) and it has at least 128 rows, its Q rows (query-major,
    // then the G heads of this kv head) are one box per 128 rows and
    // 64-channel slab of the Q tensor map, copied by TMA instead of row by
    // row (q_tma: the map fits this plan)
    const int q_first = row0 / G, q_n = (rows_here + G - 1) / G;
    auto q_run = [&](int* qa) {   // read only by the threads that stage Q
        // a box holds 128 rows: blocks with fewer copy only their own rows
        if (!q_tma || rows_here < 128) return false;
        *qa = P.chunk_q[C.q_base + q_first];
        return P.chunk_q[C.q_base + q_first + q_n - 1] - *qa == q_n - 1;
    };
    const int n = geo.n_tiles;
    // steps of softmax group w: tiles it consumes, in order
    auto n_steps = [&](int w) { return split_rows ? n : (n - w + 1) / 2; };
    auto tile_of = [&](int w, int k) { return split_rows ? k : 2 * k + w; };

    if (warp < 4) {
        if (UWarps<SPLIT>::kRegsMma < UWarps<SPLIT>::kRegsLaunch)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(UWarps<SPLIT>::kRegsMma));
        else
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(UWarps<SPLIT>::kRegsMma));
    if (warp == 0 || warp == 2 || warp == 3) {
        // ------------------------------------------------------------ TMA producers
        // warps 0 and 3 stream K (alternate page boxes), warp 2 streams V, each
        // at its own pace (two lanes of one warp would reconverge and tie the
        // streams together)
        if (lane == 0) {
            if (warp != 2) {
                prefetch_tmap(&tk);
                produce_tiles<NSLAB, kUT, KST, kKProducers>(P, C, head, sK, k_full, k_empty, &tk, warp == 0 ? 0 : 1);
            } else {
                prefetch_tmap(&tv);
                if constexpr (D == 128)
                    produce_pages<kUT, VST>(P, C, head, sV, v_full, v_empty, &tv);   // 4 KB page boxes
                else
                    produce_tiles<NSLAB, kUT, VST>(P, C, head, sV, v_full, v_empty, &tv);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = umma::idesc_bf16_f32(128, kUT, 0, 0);
            constexpr uint32_t idO = umma::idesc_bf16_f32(128, D, 0, 1);   // V is MN-major
            // Q by TMA when the block's queries are consecutive (this thread
            // has nothing else to do before Q is in); the softmax threads
            // stage it row by row otherwise
            int qa = 0;
            const bool q_by_tma = q_run(&qa);
            if (q_by_tma) {
                prefetch_tmap(&tq);
                constexpr int kHalves = SPLIT ? 2 : 1;
                mbar_arrive_expect_tx(q_full, kHalves * NSLAB * L::kQSlab);
                for (int h = 0; h < kHalves; ++h)
                    for (int s = 0; s < NSLAB; ++s)
                        tma_load_3d(sQ + (h * NSLAB + s) * L::kQSlab, &tq, 64 * s, head * G, qa + h * (128 / G),
                                    q_full);
            }
            bool ok = mbar_wait(q_ready, 0, P.status);
            // (also waited for when the wait above gave up: no copy may still
            // be writing shared memory when the block leaves)
            if (q_by_tma) ok = mbar_wait(q_full, 0, P.status) && ok;
            // test only: mma_done gets its first arrival from this thread's
            // final commit below, so this bounded wait (about a millisecond)
            // runs out and the block leaves through its error path
            if (P.debug_stall) ok = mbar_wait(mma_done, 0, P.status, 2000000LL) && ok;
            umma::fence_after_sync();
            // Descriptors are built once; an MMA only adds a compile-time byte
            // offset (>> 4) to the start-address field. Shared-memory
            // addresses stay below 2^18, so the field never carries over.
            const uint64_t dq_base[2] = {umma::smem_desc_sw128(sQ, 16, 1024),
                                         umma::smem_desc_sw128(sQ + NSLAB * L::kQSlab, 16, 1024)};
            const uint64_t dk_base = umma::smem_desc_sw128(sK, 16, 1024);
            const uint64_t dv_base = umma::smem_desc_sw128(sV, L::kVSlab, 1024);
            // S of group w for tile j: Q half (mode A) x K tile j
            auto issue_s = [&](int w, int j) {
                const uint64_t dq = dq_base[split_rows ? w : 0];
                const uint64_t dk = dk_base + (uint64_t)(((j % KST) * L::kOp) >> 4);
                const uint32_t dst = tmem + L::colS(w);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma::mma_bf16_ss(dst, dq + (((kk / 4) * L::kQSlab + (kk % 4) * 32) >> 4),
                                      dk + (((kk / 4) * L::kSlab + (kk % 4) * 32) >> 4), idS, kk > 0 ? 1u : 0u);
                umma::commit(s_full + 8 * w);
            };
            // PV of group w for tile j (its step k): O[w] (+)= P V (+ P_lo V)
            auto issue_pv = [&](int w, int k, int j) -> bool {
                if (!mbar_wait(p_full + 8 * w, k & 1, P.status)) return false;
                umma::fence_after_sync();
                const uint64_t dv = dv_base + (uint64_t)(((j % VST) * L::kOp) >> 4);
                const uint32_t ph = tmem + L::colS(w);
                const uint32_t dst = tmem + L::colO(w);
                const uint32_t acc0 = k > 0 ? 1u : 0u;
#pragma unroll
                for (int kk = 0; kk < kUT / 16; ++kk)
                    umma::mma_bf16_ts(dst, ph + 8 * kk, dv + ((kk * L::kVBox) >> 4), idO, kk > 0 ? 1u : acc0);
                if (EXACT) {
#pragma unroll
                    for (int kk = 0; kk < kUT / 16; ++kk)
                        umma::mma_bf16_ts(dst, ph + 64 + 8 * kk, dv + ((kk * L::kVBox) >> 4), idO, 1u);
                }
                return true;
            };
            auto wait_v = [&](int j) { return mbar_wait(v_full + 8 * (j % VST), (j / VST) & 1, P.status); };
            if (split_rows) {
                // per tile j: PV_0(j-1), S_0(j), PV_1(j-1), S_1(j)
                for (int j = 0; j < n && ok; ++j) {
                    if (!mbar_wait(k_full + 8 * (j % KST), (j / KST) & 1, P.status)) { ok = false; break; }
                    if (j >= 1 && !wait_v(j - 1)) { ok = false; break; }
                    for (int w = 0; w < 2 && ok; ++w) {
                        if (j >= 1 && !issue_pv(w, j - 1, j - 1)) { ok = false; break; }
                        issue_s(w, j);
                    }
                    if (!ok) break;
                    umma::commit(k_empty + 8 * (j % KST));
                    if (j >= 1) umma::commit(v_empty + 8 * ((j - 1) % VST));
                }
                if (ok && n >= 1) {
                    const int j = n - 1;
                    ok = wait_v(j) && issue_pv(0, j, j) && issue_pv(1, j, j);
                    if (ok) umma::commit(v_empty + 8 * (j % VST));
                }
            } else {
                // tile j belongs to group j & 1 (its step j >> 1); per tile j:
                // PV of tile j-2 (same group), then S of tile j
                for (int j = 0; j < n && ok; ++j) {
                    const int w = j & 1;
                    if (!mbar_wait(k_full + 8 * (j % KST), (j / KST) & 1, P.status)) { ok = false; break; }
                    if (j >= 2) {
                        if (!(wait_v(j - 2) && issue_pv(w, (j >> 1) - 1, j - 2))) { ok = false; break; }
                        umma::commit(v_empty + 8 * ((j - 2) % VST));
                    }
                    issue_s(w, j);
                    umma::commit(k_empty + 8 * (j % KST));
                }
                for (int j = max(0, n - 2); j < n && ok; ++j) {
                    ok = wait_v(j) && issue_pv(j & 1, j >> 1, j);
                    if (ok) umma::commit(v_empty + 8 * (j % VST));
                }
            }
            // every MMA issued above has finished before tensor memory is read
            // by the epilogue or released
            umma::commit(mma_done);
            mbar_wait(mma_done, 0, P.status);
        }
    }
    } else {
        if (UWarps<SPLIT>::kRegsSoftmax > UWarps<SPLIT>::kRegsLaunch)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(UWarps<SPLIT>::kRegsSoftmax));
        else
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(UWarps<SPLIT>::kRegsSoftmax));
        // ------------------------------------------------------------ softmax warpgroups
        constexpr int NG = UWarps<SPLIT>::kGroups;
        const int w = (warp - 4) / 4;                // group w: warps 4 + 4w .. 7 + 4w
        const int r = 32 * (warp % 4) + lane;        // tensor-memory lane = row within the half
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp % 4)) << 16);
        // above 128 rows, groups 0 and 1 write out (and stage Q for) row halves 0 and 1
        const int rloc = split_rows ? 128 * (w & 1) + r : r;   // row within the block
        const bool row_ok = rloc < rows_here;
        int qi = 0, gh = 0;
        uint64_t mask = ~0ull;
        if (row_ok) {
            qi = (row0 + rloc) / G;
            gh = (row0 + rloc) % G;
            if (C.mask_base >= 0) mask = P.masks[C.mask_base + qi];
        }
        int qa_unused;
        if ((split_rows ? w < 2 : w == 0) && !q_run(&qa_unused)) {
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
        bool ok = true;
        // the row this thread writes out: its running max (log2 units) and sum
        float m_fin = -INFINITY, l_fin = 0.f;
        int nk;   // steps this thread took part in
        if constexpr (SPLIT) {
            // ---- more than 128 rows: every group works on both row halves of
            // every tile; group w owns S columns [kCols w, kCols (w + 1)) of
            // each half. The row max is the largest of the groups' maxima,
            // exchanged through shared memory; a half's softmax then runs on
            // all groups and overlaps the MMAs of the other half.
            constexpr int kCols = 128 / NG;
            nk = n;
            float* red = reinterpret_cast<float*>(base + L::kRed);   // [half][group][128]
            float* lred = reinterpret_cast<float*>(base + L::kLRed); // [half][group][128]
            float m_ref[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.f, 0.f};
            uint64_t mask_h[2] = {~0ull, ~0ull};
            if (masked_chunk) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    if (128 * h + r < rows_here) mask_h[h] = P.masks[C.mask_base + (row0 + 128 * h + r) / G];
            }
            const int col0 = kCols * w;
            for (int k = 0; k < n && ok; ++k) {
                const int tpos = geo.tile0 + k * kUT;
                const bool edge = tpos < geo.pos_begin || tpos + kUT > geo.pos_end;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    // tcgen05.ld/st are warp-collective: every decision that
                    // guards them is taken by the whole warp
                    if (!__all_sync(0xffffffffu, mbar_wait(s_full + 8 * h, k & 1, P.status))) { ok = false; break; }
                    umma::fence_after_sync();
                    const uint32_t s_addr = lane_addr + L::colS(h);
                    if (edge || masked_chunk) mask_in_tmem<kCols>(s_addr, col0, geo.pos_begin - tpos,
                                                                 geo.pos_end - tpos, mask_h[h], masked_chunk);
                    float x[kCols];
                    ld_cols<kCols>(s_addr + col0, x);
                    red[(NG * h + w) * 128 + r] = row_max(x);
                    if (!EXACT) lred[(NG * h + w) * 128 + r] = lsum[h];
                    mbar_arrive(xchg_bar + 8 * h);
                    if (!__all_sync(0xffffffffu, mbar_wait(xchg_bar + 8 * h, k & 1, P.status))) { ok = false; break; }
                    float mx = red[(NG * h) * 128 + r];
#pragma unroll
                    for (int g = 1; g < NG; ++g) mx = fmaxf(mx, red[(NG * h + g) * 128 + r]);
                    const float mxs = mx * sl;   // scale > 0: max commutes with it
                    bool grow = (m_ref[h] == -INFINITY) ? (mx != -INFINITY) : (mxs > m_ref[h] + kLazyRescale);
                    if (!EXACT && !grow && mx != -INFINITY && mxs > m_ref[h]) {
                        // the tile's largest weight, 2^(mxs - m_ref) <= 2^8, against
                        // the row's sum so far (every group adds the same values in
                        // the same order, so all take the same decision): if it is a
                        // large share, move the max to it so that it becomes 1 exactly
                        float lb = 0.f;
#pragma unroll
                        for (int g = 0; g < NG; ++g) lb += lred[(NG * h + g) * 128 + r];
                        const float wmax = fast_exp2(mxs - m_ref[h]);
                        grow = wmax > kExactShare * (lb + wmax);
                    }
                    float alpha = 1.f;
                    bool rescale = false;
                    if (grow) {
                        alpha = fast_exp2(m_ref[h] - mxs);   // 0 when nothing was accumulated
                        rescale = k >= 1 && m_ref[h] != -INFINITY;
                        lsum[h] *= alpha;
                        m_ref[h] = mxs;
                    }
                    // every group's S is in registers (exchange above): P may
                    // now go anywhere in the half's columns
                    lsum[h] += softmax_p<kCols, EXACT>(x, sl, m_ref[h] == -INFINITY ? 0.f : -m_ref[h],
                                                       s_addr + (kCols / 2) * w, s_addr + 64 + (kCols / 2) * w);
                    if (__any_sync(0xffffffffu, rescale))
                        scale_o<D / NG>(lane_addr + L::colO(h) + (D / NG) * w, rescale ? alpha : 1.f);
                    if (edge && w == 0 && h == 0) {
                        if (!__all_sync(0xffffffffu, zero_stray_v<L>(P, base, geo, tpos, k, r, v_full))) { ok = false; break; }
                    }
                    umma::wait_st();
                    umma::fence_before_sync();
                    mbar_arrive(p_full + 8 * h);
                }
            }
            // groups 0 and 1 write out halves 0 and 1 and need every group's
            // sums of their rows (the K ring is free only later)
            float* lx = red + 2 * NG * 128;   // [half][group][128]
            lx[w * 128 + r] = lsum[0];
            lx[(NG + w) * 128 + r] = lsum[1];
            mbar_arrive(lfin_bar);
            if (!__all_sync(0xffffffffu, mbar_wait(lfin_bar, 0, P.status))) ok = false;
            if (w < 2) {
                m_fin = m_ref[w];
                l_fin = 0.f;
#pragma unroll
                for (int g = 0; g < NG; ++g) l_fin += lx[(NG * w + g) * 128 + r];
            }
        } else {
            // ---- at most 128 rows: the groups take alternate tiles into their
            // own S buffer and O accumulator (split-KV inside the block)
            nk = n_steps(w);
            float m_ref = -INFINITY, l = 0.f;
            const uint32_t s_addr = lane_addr + L::colS(w);
            for (int k = 0; k < nk; ++k) {
                const int j = tile_of(w, k);
                if (!__all_sync(0xffffffffu, mbar_wait(s_full + 8 * w, k & 1, P.status))) { ok = false; break; }
                umma::fence_after_sync();
                const int tpos = geo.tile0 + j * kUT;
                const bool edge = tpos < geo.pos_begin || tpos + kUT > geo.pos_end;
                if (edge || masked_chunk) mask_in_tmem<kUT>(s_addr, 0, geo.pos_begin - tpos, geo.pos_end - tpos, mask,
                                                           masked_chunk);
                float x[kUT];
                ld_cols<kUT>(s_addr, x);
                const float mx = row_max(x);
                const float mxs = mx * sl;
                bool grow = (m_ref == -INFINITY) ? (mx != -INFINITY) : (mxs > m_ref + kLazyRescale);
                if (!EXACT && !grow && mx != -INFINITY && mxs > m_ref) {
                    // the tile's largest weight against the group's sum so far:
                    // if it is a large share, it becomes 1 exactly (see above)
                    const float wmax = fast_exp2(mxs - m_ref);
                    grow = wmax > kExactShare * (l + wmax);
                }
                float alpha = 1.f;
                bool rescale = false;
                if (grow) {
                    alpha = fast_exp2(m_ref - mxs);
                    rescale = k >= 1 && m_ref != -INFINITY;
                    l *= alpha;
                    m_ref = mxs;
                }
                l += softmax_p<kUT, EXACT>(x, sl, m_ref == -INFINITY ? 0.f : -m_ref, s_addr, s_addr + 64);
                if (__any_sync(0xffffffffu, rescale)) scale_o<D>(lane_addr + L::colO(w), rescale ? alpha : 1.f);
                if (edge) {
                    if (!__all_sync(0xffffffffu, zero_stray_v<L>(P, base, geo, tpos, j, r, v_full))) { ok = false; break; }
                }
                umma::wait_st();
                umma::fence_before_sync();
                mbar_arrive(p_full + 8 * w);
            }
            m_fin = m_ref;
            l_fin = l;
        }
        // ---- epilogue: wait for the MMA warp's final commit (every MMA done)
        const bool have = __all_sync(0xffffffffu, ok && nk >= 1 && mbar_wait(mma_done, 0, P.status));
        if (have) umma::fence_after_sync();
        float m1 = -INFINITY, l1 = 0.f;
        if (!split_rows) {
            // split-KV inside the block: group 1 hands (m, l) to group 0, which
            // reads both O accumulators (same lanes) and merges them
            if (w == 1) {
                xchg[r] = make_float2(have ? m_fin : -INFINITY, have ? l_fin : 0.f);
                asm volatile("bar.arrive 1, 256;" ::: "memory");
            } else {
                asm volatile("bar.sync 1, 256;" ::: "memory");
                const float2 ml = xchg[r];
                m1 = ml.x;
                l1 = ml.y;
            }
        }
        if (have && (split_rows ? w < 2 : w == 0)) {
            const bool use1 = !split_rows && n >= 2;   // group 1's accumulator is complete (mma_done)
            const float M = fmaxf(m_fin, m1);
            const float Mu = M == -INFINITY ? 0.f : M;
            const float a0 = fast_exp2(m_fin - Mu), a1 = fast_exp2(m1 - Mu);
            const float Lt = l_fin * a0 + l1 * a1;
            const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
            const int64_t prow = (int64_t)C.part_base + (int64_t)qi * Hq + head * G + gh;
            // The warp's 32 rows go through shared memory (the K/V rings are
            // free once every MMA has finished) so that each global store
            // writes whole 512-byte rows: row-major [32][D] floats, the 16-byte
            // units of row r permuted by r & 7 against bank conflicts.
            float* stage = reinterpret_cast<float*>(base + L::kK) + (size_t)(warp - 4) * 32 * D;
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
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const int u = 8 * c + i / 4;
                    *reinterpret_cast<float4*>(stage + lane * D + 4 * (u ^ (lane & 7))) =
                        make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv);
                }
            }
            __syncwarp();
            constexpr int kUnits = D / 4;            // float4 units per row
            constexpr int kRowsPerStep = 32 / kUnits;
            const int64_t my_prow = row_ok ? prow : -1;
#pragma unroll 4
            for (int rr = 0; rr < 32; rr += kRowsPerStep) {
                const int r2 = rr + lane / kUnits, u = lane % kUnits;
                const int64_t pr = __shfl_sync(0xffffffffu, my_prow, r2);
                if (pr >= 0)
                    *reinterpret_cast<float4*>(P.part_o + pr * D + 4 * u) =
                        *reinterpret_cast<const float4*>(stage + r2 * D + 4 * (u ^ (r2 & 7)));
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

template <int D, bool EXACT, bool SPLIT>
cudaError_t launch_umma_t(const DevPlan& P, const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tq,
                          const void* Q, int n_items, int item_off, cudaStream_t st, bool pdl) {
    const size_t smem = 1024 + UmmaLayout<D>::kBytes;
    static DeviceOnce once;   // per device
    cudaError_t e = per_device(once, nullptr, nullptr, [&](int, int* a, int*) {
        // setmaxnreg.inc waits for registers another warpgroup released: the
        // split is only valid for the launch register count it was sized for
        cudaFuncAttributes fa;
        cudaError_t r = cudaFuncGetAttributes(&fa, pac_umma_kernel<D, EXACT, SPLIT>);
        if (r != cudaSuccess) return r;
        if (fa.numRegs != UWarps<SPLIT>::kRegsLaunch) return cudaErrorInvalidConfiguration;
        r = cudaFuncSetAttribute(pac_umma_kernel<D, EXACT, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        *a = 1;
        return r;
    });
    if (e != cudaSuccess) return e;
    return launch_kernel(pac_umma_kernel<D, EXACT, SPLIT>, dim3(n_items), dim3(UWarps<SPLIT>::kThreads), smem, st, pdl,
                         P, *tk, *tv, static_cast<const __nv_bfloat16*>(Q), item_off, tq ? *tq : *tk, tq ? 1 : 0);
}

template <int D, bool EXACT>
cudaError_t launch_umma_m(const DevPlan& P, const CUtensorMap* tk, const CUtensorMap* tv, const CUtensorMap* tq,
                          const void* Q, int n_items, int item_off, bool split_rows, cudaStream_t st, bool pdl) {
    return split_rows ? launch_umma_t<D, EXACT, true>(P, tk, tv, tq, Q, n_items, item_off, st, pdl)
                      : launch_umma_t<D, EXACT, false>(P, tk, tv, tq, Q, n_items, item_off, st, pdl);
}

}  // namespace dev

// tq: the Q tensor map (boxes of 128 rows x 64 channels), or null to stage Q
// row by row
cudaError_t launch_pac_umma(const DevPlan& P, const void* tk, const void* tv, const void* tq, const void* Q,
                            int n_items, int item_off, bool exact_p, bool split_rows, cudaStream_t st, bool pdl) {
    const CUtensorMap* k = static_cast<const CUtensorMap*>(tk);
    const CUtensorMap* v = static_cast<const CUtensorMap*>(tv);
    const CUtensorMap* q = static_cast<const CUtensorMap*>(tq);
    if (P.d == 128)
        return exact_p ? dev::launch_umma_m<128, true>(P, k, v, q, Q, n_items, item_off, split_rows, st, pdl)
                       : dev::launch_umma_m<128, false>(P, k, v, q, Q, n_items, item_off, split_rows, st, pdl);
    return exact_p ? dev::launch_umma_m<64, true>(P, k, v, q, Q, n_items, item_off, split_rows, st, pdl)
                   : dev::launch_umma_m<64, false>(P, k, v, q, Q, n_items, item_off, split_rows, st, pdl);
}

}  // namespace pst
