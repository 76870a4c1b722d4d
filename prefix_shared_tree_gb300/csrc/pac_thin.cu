// Tensor-core partial attention computation (PAC) for thin chunks: fewer
// aggregated query rows (queries x GQA group) per kv head than the
// tensor-core PAC's threshold; bf16, d = 128, Hkv a multiple of 8.
//
// CoDec, "intra-block primitives": each K/V tile of the chunk is loaded into
// shared memory once for all of the chunk's query rows and the PAC emits a
// partial output with its softmax statistics for the POR merge. CoDec, "KV
// cache management": node-local stabilisation with a running max and sum.
// DEFT's bit causal mask gives per-row visibility inside packed chunks.
//
// Layout of the work. A thin chunk has too few rows to fill the 128-row M
// side of a tcgen05 MMA, so the roles are swapped: the M side holds keys, and
// a block takes 8 kv heads at once, so one 16-token page row-box of all 8
// heads fills it (lane 16 h + t = token t of head h). One TMA instruction then
// moves a whole 32 KB K (or V) tile: the per-instruction cost of the TMA unit,
// not the bytes, limits paged loads of single-head 2 KB boxes on GB300. Per
// tile of 16 tokens x 8 heads:
//     S^T   = K Q^T        M = 128 (head, token), N = 8 R (head, row), K = d;
//                          only the blocks with matching heads are used
//     O^T_h += V_h^T P_h^T  per head h: M = d, N = 16 (R rows used), K = the
//                          head's 16 tokens (V read MN-major, P^T from shared memory)
// R = 4 or 8 rows per head. Each head's 16 tokens sit in one half-warp, so a
// row's tile maximum is a 16-lane shuffle reduction. P^T goes to shared memory
// in bf16 as hi + lo parts (p = hi + lo to ~2^-16), rows r and R + r of one
// 16-row operand, so one N = 16 MMA per head reads the V tile once and keeps
// both parts in separate O^T columns (summed at the end): P V is as accurate
// as an fp32 product. Two softmax warpgroups take alternate tiles of an item
// (even and odd tile index, so the result does not depend on which block ran
// the item), each into its own O^T accumulator (split-KV inside the block),
// and merge at the end of the item; S^T of global tile g goes to buffer g & 1.
// A group's running max only moves (and its O^T is rescaled in tensor memory,
// after a vote of its four warps) when it grows by more than 2^8.
//
// Persistent blocks, one per SM, take items (largest first) from a work queue:
//   warp 0      claims an item, stages its Q rows in shared memory, then
//               streams the chunk's K tiles with TMA; warp 2 streams its V
//               tiles into a second ring at its own pace;
//   warp 1      allocates tensor memory and issues the S^T MMAs (one
//               thread); warp 3 issues the P V MMAs (one thread);
//   warps 4-7, 8-11  two softmax warpgroups (even and odd tiles of an item),
//               one thread per tensor-memory lane, and the epilogue.
#include <algorithm>

#include "dev_common.cuh"
#include "umma.cuh"

namespace pst {
namespace dev {

constexpr int kThinTT = kBoxRows;                // tokens per tile (one page row-box)
constexpr int kThinThreads = 384;
constexpr float kThinLazy = 8.f;

template <int R>
struct ThinLayout {
    static constexpr int D = 128;
    static constexpr int NS = kThinHeads * R;                // S^T columns = staged Q rows
    static constexpr int NSLAB = D / 64;
    static constexpr uint32_t kSlab = 128 * 128;             // 128 (head, token) rows x 128 B
    static constexpr uint32_t kOp = NSLAB * kSlab;           // one K or V tile (32 KB)
    static constexpr int KST = 3, VST = R == 4 ? 3 : 2;
    static constexpr uint32_t kQSlab = NS * 128;             // NS rows x 128 B
    static constexpr uint32_t kQBuf = NSLAB * kQSlab;
    static constexpr uint32_t kPSlab = 16 * 128;             // P^T: 16 rows (hi r, lo R + r) x 64 lanes
    static constexpr uint32_t kPBuf = 2 * kPSlab;            // 16 rows x 128 lanes
    static constexpr uint32_t kK = 0;
    static constexpr uint32_t kV = kK + KST * kOp;
    static constexpr uint32_t kQ = kV + VST * kOp;           // 2 slots (item parity)
    static constexpr uint32_t kP = kQ + 2 * kQBuf;           // [group]
    static constexpr uint32_t kVote = kP + 2 * kPBuf;        // [group][vote parity][head]: grew flag, R alphas
    static constexpr uint32_t kSum = kVote + 2 * 2 * kThinHeads * (R + 1) * 4;   // [item parity][group][2][head][R]
    static constexpr uint32_t kSlot = kSum + 2 * 2 * 2 * kThinHeads * R * 4;  // ThinSlot x 2 (item parity)
    static constexpr uint32_t kBars = kSlot + 2 * 64;
    // k_full[KST], k_empty[KST], v_full[VST], v_empty[VST], item_full[2], item_empty[2], q_empty[2],
    // s_full[2], p_full[2], vote_bar[2], s_free[2], pv_done[2], o_full, fin, fin_pv, lsum_bar, epi_bar
    static constexpr int kNumBars = 2 * KST + 2 * VST + 16 + 5;
    static constexpr uint32_t kTslot = kBars + 8 * kNumBars;
    static constexpr uint32_t kBytes = kTslot + 16;
    static_assert(kBytes + 1024 <= 232448, "shared memory");
    static_assert(kQ % 1024 == 0 && kP % 1024 == 0 && kQSlab % 1024 == 0, "SW128 operand alignment");
    static constexpr uint32_t kTmemCols = 512;
    // S^T of global tile g in buffer g & 1; O^T of group w, head h: hi part of
    // row r at colO(w) + 16 h + r, lo part at colO(w) + 16 h + R + r
    __device__ static constexpr uint32_t colS(int b) { return NS * b; }
    __device__ static constexpr uint32_t colO(int w) { return 2 * NS + 16 * kThinHeads * w; }
    static_assert(2 * NS + 2 * 16 * kThinHeads <= kTmemCols, "tensor memory columns");
};

// R per-lane values reduced over the 16 lanes of a half-warp (max or sum):
// each butterfly stage with more than one live value sends half of them to
// the partner lane and keeps the other half; afterwards lane l of the half
// holds the result for value index (l & 15) >> (4 - log2 R), in a[0].
template <int OFF, int NV, bool MAX>
struct HRed {
    template <int R>
    __device__ __forceinline__ static void run(float (&a)[R], int lane) {
        if constexpr (OFF >= 1) {
            if constexpr (NV > 1) {
                constexpr int H = NV / 2;
                const bool up = (lane & OFF) != 0;
#pragma unroll
                for (int i = 0; i < H; ++i) {
                    const float send = up ? a[i] : a[i + H];
                    const float keep = up ? a[i + H] : a[i];
                    const float got = __shfl_xor_sync(0xffffffffu, send, OFF);
                    a[i] = MAX ? fmaxf(keep, got) : keep + got;
                }
                HRed<OFF / 2, H, MAX>::run(a, lane);
            } else {
                const float got = __shfl_xor_sync(0xffffffffu, a[0], OFF);
                a[0] = MAX ? fmaxf(a[0], got) : a[0] + got;
                HRed<OFF / 2, 1, MAX>::run(a, lane);
            }
        }
    }
};

// An item as the producer hands it to the MMA threads and the softmax warps
// (index -1: no more items).
struct alignas(16) ThinSlot {
    DevChunk C;
    DevItem it;
    int32_t idx;
    int32_t pad[5];
};
static_assert(sizeof(ThinSlot) == 64, "ThinSlot layout");

// TMA producer (one thread) of one operand: every 16-token tile of the chunk
// for the block's 8 heads into a ring of ST stages (one 32 KB box per tile:
// both 64-channel slabs x 8 heads x 16 rows, landing as [slab][head][row]).
// Tile i is global tile g = gbase + i of this block. K and V have their own
// producers: V stages free late (after the softmax and P V) and must not hold
// back the next K tiles. False if a wait gave up.
template <int ST>
__device__ bool thin_produce(const DevPlan& P, const DevChunk& C, int head0, uint32_t ring, uint32_t full,
                             uint32_t empty, const CUtensorMap* map, int gbase) {
    constexpr uint32_t kOp = 2 * 128 * 128;
    const ChunkGeo geo = chunk_geo<kThinTT>(C);
    const int ps = P.page_size;
    for (int i = 0; i < geo.n_tiles; ++i) {
        const int g = gbase + i;
        const int tpos = geo.tile0 + i * kThinTT;
        const int page = P.pages[C.page_base + tpos / ps];
        const int s = g % ST;
        if (g >= ST && !mbar_wait(empty + 8 * s, ((g / ST) - 1) & 1, P.status)) {
            drain_ring<ST>(full, g, P.status);
            return false;
        }
        mbar_arrive_expect_tx(full + 8 * s, kOp);
        tma_load_5d(ring + s * kOp, map, 0, tpos % ps, head0, 0, page, full + 8 * s);
    }
    return true;
}

// tcgen05.ld of 2R columns (32 lanes x 32 bit) without the wait.
template <int R>
__device__ __forceinline__ void ld_2r(uint32_t taddr, uint32_t (&v)[2 * R]) {
    if constexpr (R == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                     : "r"(taddr)
                     : "memory");
    } else {
        umma::ld16(taddr, v);
    }
}

template <int R>
__global__ void __launch_bounds__(kThinThreads, 1)
pac_thin_kernel(DevPlan P, const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                const __nv_bfloat16* __restrict__ Q, int item_off, int n_items, int counter) {
    using L = ThinLayout<R>;
    constexpr int NS = L::NS, D = L::D, KST = L::KST, VST = L::VST, HB = kThinHeads;
    constexpr int kSh = R == 4 ? 2 : 1;   // half-warp lane l holds row (l & 15) >> kSh after a reduction
    static_assert(R == 4 || R == 8, "rows per head");
    extern __shared__ uint8_t smem_raw[];
    pdl_launch_dependents();   // the next launch group may take the SMs this grid leaves
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(base);
    const uint32_t bars = sbase + L::kBars;
    const uint32_t k_full = bars, k_empty = k_full + 8 * KST;
    const uint32_t v_full = k_empty + 8 * KST, v_empty = v_full + 8 * VST;
    const uint32_t item_full = v_empty + 8 * VST, item_empty = item_full + 16, q_empty = item_empty + 16;
    const uint32_t s_full = q_empty + 16;     // [S^T buffer]
    const uint32_t p_full = s_full + 16;      // [group]
    const uint32_t vote_bar = p_full + 16;    // [group]: every head's growth flag is in
    const uint32_t s_free = vote_bar + 16;    // [S^T buffer]: its softmax has loaded it
    const uint32_t pv_done = s_free + 16;     // [group]: the group's P V products issued so far have finished
    const uint32_t o_full = pv_done + 16, fin = o_full + 8, fin_pv = fin + 8;
    const uint32_t lsum_bar = fin_pv + 8;     // both groups' row sums and maxima are in
    const uint32_t epi_bar = lsum_bar + 8;    // both groups have read both accumulators
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kTslot);
    ThinSlot* slots = reinterpret_cast<ThinSlot*>(base + L::kSlot);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int G = P.group, Hq = P.n_q_heads;

    if (threadIdx.x == 0) {
        for (int s = 0; s < KST; ++s) {
            mbar_init(k_full + 8 * s, 1);
            mbar_init(k_empty + 8 * s, 1);
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(v_full + 8 * s, 1);
            mbar_init(v_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(item_full + 8 * b, 32);       // every lane of the producer warp (its Q stores)
            mbar_init(item_empty + 8 * b, 3 + 8);   // the V producer, the two MMA threads, the eight softmax warps
            mbar_init(q_empty + 8 * b, 1);
            mbar_init(s_full + 8 * b, 1);
            mbar_init(p_full + 8 * b, 128);
            mbar_init(vote_bar + 8 * b, 128);
            mbar_init(s_free + 8 * b, 128);
            mbar_init(pv_done + 8 * b, 1);
        }
        mbar_init(fin_pv, 1);
        mbar_init(o_full, 1);
        mbar_init(fin, 1);
        mbar_init(lsum_bar, 256);
        mbar_init(epi_bar, 256);
        fence_barrier_init();
    }
    // P^T rows 2R..15 stay zero (the P V MMAs read 16 rows)
    for (uint32_t i = threadIdx.x; i < 2 * L::kPBuf / 16; i += kThinThreads)
        *reinterpret_cast<uint4*>(base + L::kP + 16 * i) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 1) {
        umma::tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ items, Q and TMA
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
        }
        int gbase = 0;
        for (int q = 0;; ++q) {
            const int slot = q & 1;
            if (q >= 2) {
                // the slot's index was read and the MMAs reading its Q are done
                bool w = true;
                if (lane == 0)
                    w = mbar_wait(item_empty + 8 * slot, ((q >> 1) - 1) & 1, P.status) &&
                        mbar_wait(q_empty + 8 * slot, ((q >> 1) - 1) & 1, P.status);
                if (!__shfl_sync(0xffffffffu, w, 0)) break;
            }
            // claimed only now: with few items, claiming ahead leaves blocks idle
            int idx = 0;
            if (lane == 0) idx = atomicAdd(P.counters + counter, 1);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            DevChunk C{};
            DevItem it{};
            if (idx < n_items) {
                it = P.items[item_off + idx];
                C = P.chunks[it.chunk];
                const int rows_total = C.n_q * G;
                const int row0 = it.row_block * R;
                const int rows_here = min(R, rows_total - row0);
                int qid[R];
#pragma unroll
                for (int r = 0; r < R; ++r) qid[r] = r < rows_here ? P.chunk_q[C.q_base + (row0 + r) / G] : 0;
                // Q row n = (head h, row r), K-major with the 128B swizzle: row n of
                // slab d / 64 at n * 128. All loads of a batch are issued before
                // its shared-memory stores.
                uint8_t* qdst = base + L::kQ + slot * L::kQBuf;
                constexpr int kUnits = NS * 16 / 32, kBatch = 8;
#pragma unroll
                for (int i0 = 0; i0 < kUnits; i0 += kBatch) {
                    uint4 v[kBatch];
#pragma unroll
                    for (int i = 0; i < kBatch; ++i) {
                        const int u = lane + 32 * (i0 + i), n = u / 16, ch = u % 16;
                        const int h = n / R, r = n % R;
                        v[i] = make_uint4(0, 0, 0, 0);
                        if (r < rows_here) {
                            const int row = row0 + r;
                            int qr = qid[0];   // qid[r] without a local-memory index
#pragma unroll
                            for (int rr = 1; rr < R; ++rr) qr = rr == r ? qid[rr] : qr;
                            v[i] = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(
                                Q + ((int64_t)qr * Hq + (it.kv_head + h) * G + row % G) * D) + ch * 16));
                        }
                    }
#pragma unroll
                    for (int i = 0; i < kBatch; ++i) {
                        const int u = lane + 32 * (i0 + i), n = u / 16, ch = u % 16;
                        *reinterpret_cast<uint4*>(qdst + (ch / 8) * L::kQSlab + swz(n, ch % 8)) = v[i];
                    }
                }
                fence_proxy_async_smem();
            }
            if (lane == 0) {
                slots[slot].C = C;
                slots[slot].it = it;
                slots[slot].idx = idx < n_items ? idx : -1;
            }
            __syncwarp();
            mbar_arrive(item_full + 8 * slot);
            if (idx >= n_items) break;
            const int head0 = it.kv_head;
            bool ok = true;
            if (lane == 0) ok = thin_produce<KST>(P, C, head0, sbase + L::kK, k_full, k_empty, &tk, gbase);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                gbase = -1;   // drained already
                break;
            }
            gbase += chunk_geo<kThinTT>(C).n_tiles;
        }
        // the last K loads have landed before the producer leaves
        if (lane == 0 && gbase >= 0) drain_ring<KST>(k_full, gbase, P.status);
    } else if (warp == 2) {
        // ------------------------------------------------------------ V producer
        if (lane == 0) {
            prefetch_tmap(&tv);
            int gbase = 0;
            for (int q = 0;; ++q) {
                const int slot = q & 1;
                if (!mbar_wait(item_full + 8 * slot, (q >> 1) & 1, P.status)) break;
                const int idx = slots[slot].idx;
                const DevChunk C = slots[slot].C;
                const int head0 = slots[slot].it.kv_head;
                mbar_arrive(item_empty + 8 * slot);
                if (idx < 0) break;
                if (!thin_produce<VST>(P, C, head0, sbase + L::kV, v_full, v_empty, &tv, gbase)) {
                    gbase = -1;   // drained already
                    break;
                }
                gbase += chunk_geo<kThinTT>(C).n_tiles;
            }
            if (gbase >= 0) drain_ring<VST>(v_full, gbase, P.status);
        }
        __syncwarp();
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------------------ MMA issuers
        // Two threads issue the tensor-core work side by side: warp 1 the S^T
        // MMAs of every tile, warp 3 the P V MMAs (issuing a tcgen05 MMA costs
        // its thread tens of cycles, so one thread for both streams serialises
        // them). Each orders its own MMAs; the softmax warps get the cross
        // orderings from barriers: S^T buffer g & 1 is refilled once its
        // softmax has loaded it (s_free), and a group waits for its previous
        // P V (pv_done) before it rescales O^T or rewrites its P^T.
        if (lane == 0) {
            constexpr uint32_t idS = umma::idesc_bf16_f32(128, NS, 0, 0);   // K and Q both K-major
            constexpr uint32_t idO = umma::idesc_bf16_f32(128, 16, 1, 0);   // V^T MN-major, P^T K-major
            // Descriptors are built once; an MMA only adds a compile-time byte
            // offset (>> 4) to the start-address field, which never carries
            // over (shared-memory addresses stay below 2^18).
            const uint64_t dk0 = umma::smem_desc_sw128(sbase + L::kK, 16, 1024);
            const uint64_t dv0 = umma::smem_desc_sw128(sbase + L::kV, L::kSlab, 1024);
            const uint64_t dq0 = umma::smem_desc_sw128(sbase + L::kQ, 16, 1024);
            const uint64_t dp0 = umma::smem_desc_sw128(sbase + L::kP, 16, 1024);
            const bool s_side = warp == 1;
            int gbase = 0;
            int n_p[2] = {0, 0};   // P V side: p_full phases consumed per group
            bool ok = true;
            for (int q = 0; ok; ++q) {
                const int slot = q & 1;
                if (!mbar_wait(item_full + 8 * slot, (q >> 1) & 1, P.status)) break;
                const int idx = slots[slot].idx;
                const DevChunk C = slots[slot].C;
                mbar_arrive(item_empty + 8 * slot);
                if (idx < 0) break;
                const int n = chunk_geo<kThinTT>(C).n_tiles;
                if (s_side) {
                    const uint64_t dq = dq0 + (uint64_t)((slot * L::kQBuf) >> 4);
                    for (int j = 0; j < n; ++j) {
                        const int g = gbase + j;
                        // buffer g & 1 last held S^T of tile g - 2: loaded by its softmax
                        if (g >= 2 && !mbar_wait(s_free + 8 * (g & 1), ((g >> 1) - 1) & 1, P.status)) {
                            ok = false;
                            break;
                        }
                        if (!mbar_wait(k_full + 8 * (g % KST), (g / KST) & 1, P.status)) { ok = false; break; }
                        umma::fence_after_sync();
                        const uint64_t dk = dk0 + (uint64_t)(((g % KST) * L::kOp) >> 4);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            umma::mma_bf16_ss(tmem + L::colS(g & 1), dk + (((kk / 4) * L::kSlab + (kk % 4) * 32) >> 4),
                                              dq + (((kk / 4) * L::kQSlab + (kk % 4) * 32) >> 4), idS,
                                              kk > 0 ? 1u : 0u);
                        umma::commit(s_full + 8 * (g & 1));
                        umma::commit(k_empty + 8 * (g % KST));
                        if (j == n - 1) umma::commit(q_empty + 8 * slot);
                    }
                } else {
                    // O^T_h of group w (+)= V_h^T [P_hi; P_lo]_h^T for tile g, every
                    // head h; a group's first tile of the item starts its accumulator
                    for (int j = 0; j < n; ++j) {
                        const int g = gbase + j, w = j & 1;
                        if (!mbar_wait(p_full + 8 * w, n_p[w]++ & 1, P.status)) { ok = false; break; }
                        if (!mbar_wait(v_full + 8 * (g % VST), (g / VST) & 1, P.status)) { ok = false; break; }
                        umma::fence_after_sync();
                        const uint64_t dv = dv0 + (uint64_t)(((g % VST) * L::kOp) >> 4);
                        const uint64_t dp = dp0 + (uint64_t)((w * L::kPBuf) >> 4);   // group w's P^T
#pragma unroll
                        for (int h = 0; h < HB; ++h)
                            umma::mma_bf16_ss(tmem + L::colO(w) + 16 * h, dv + ((h * 2048) >> 4),
                                              dp + (((h / 4) * L::kPSlab + (h % 4) * 32) >> 4), idO,
                                              j < 2 ? 0u : 1u);
                        umma::commit(v_empty + 8 * (g % VST));
                        umma::commit(pv_done + 8 * w);
                    }
                    if (ok) umma::commit(o_full);
                }
                gbase += n;
            }
            // every MMA this thread issued has finished before tensor memory is released
            const uint32_t done = s_side ? fin : fin_pv;
            umma::commit(done);
            mbar_wait(done, 0, P.status);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax and epilogue
        const int w = (warp - 4) / 4;             // group: tiles j of an item with j & 1 == w
        const int wq = warp % 4;                  // lane quarter of tensor memory
        const int ell = 32 * wq + lane;           // lane: (head h, token t) in S^T, channel in O^T
        const int h = ell / 16, t = ell % 16;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * wq) << 16);
        float* vote = reinterpret_cast<float*>(base + L::kVote) + w * 2 * HB * (R + 1);   // [vote parity][head][1 + R]
        const float sl = P.scale_log2;
        int gbase = 0, n_done = 0, n_vote = 0, n_tiles_w = 0;   // n_tiles_w: this group's tiles so far (all items)
        bool ok = true;
        for (int q = 0; ok; ++q) {
            const int slot = q & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(item_full + 8 * slot, (q >> 1) & 1, P.status))) break;
            const int idx = slots[slot].idx;
            const DevItem it = slots[slot].it;
            const DevChunk C = slots[slot].C;
            __syncwarp();
            if (lane == 0) mbar_arrive(item_empty + 8 * slot);
            if (idx < 0) break;
            const int rows_total = C.n_q * G;
            const int row0 = it.row_block * R;
            const int rows_here = min(R, rows_total - row0);
            const ChunkGeo geo = chunk_geo<kThinTT>(C);
            const int n = geo.n_tiles;
            const bool masked = C.mask_base >= 0;
            uint64_t mask[R];
#pragma unroll
            for (int r = 0; r < R; ++r)
                mask[r] = (masked && r < rows_here) ? P.masks[C.mask_base + (row0 + r) / G] : ~0ull;
            // running max (log2 units) and this lane's share of the row sums, for head h
            float m_ref[R], lp[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                m_ref[r] = -INFINITY;
                lp[r] = 0.f;
            }
            for (int j = w; j < n; j += 2) {
                const int g = gbase + j;
                const int k_w = n_tiles_w++;   // this group's tiles before this one (all items)
                if (!__all_sync(0xffffffffu, mbar_wait(s_full + 8 * (g & 1), (g >> 1) & 1, P.status))) {
                    ok = false;
                    break;
                }
                umma::fence_after_sync();
                uint32_t sr[2 * R];   // this warp's two heads
                ld_2r<R>(lane_addr + L::colS(g & 1) + 2 * wq * R, sr);
                umma::wait_ld();
                umma::fence_before_sync();
                mbar_arrive(s_free + 8 * (g & 1));   // the S^T MMA thread may refill the buffer
                // The group's previous P V (tile j - 2, issued by the other MMA
                // thread) has finished before its O^T is rescaled or its P^T
                // rewritten; for tiles j < 2 the previous item's P V products
                // finished before its epilogue.
                bool pv_waited = j < 2;
                auto wait_prev_pv = [&]() -> bool {
                    if (pv_waited) return true;
                    pv_waited = true;
                    if (!__all_sync(0xffffffffu, mbar_wait(pv_done + 8 * w, (k_w - 1) & 1, P.status))) return false;
                    umma::fence_after_sync();   // order later tensor-memory accesses after those MMAs
                    return true;
                };
                const int tpos = geo.tile0 + j * kThinTT;
                const int pos = tpos + t;
                const bool in = pos >= geo.pos_begin && pos < geo.pos_end;
                const int tc = pos - geo.pos_begin;      // token index in the chunk
                float s[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const bool vis = in && r < rows_here &&
                                     (!masked || tc >= kMaskTokens || ((mask[r] >> (tc & 63)) & 1ull));
                    s[r] = vis ? __uint_as_float((h & 1) ? sr[R + r] : sr[r]) : -INFINITY;
                }
                // V rows outside the chunk may hold stale or non-finite values:
                // zero them before P V multiplies them by P = 0
                if (tpos < geo.pos_begin || tpos + kThinTT > geo.pos_end) {
                    const int vs = g % VST;
                    // V of tile g - 2 has landed (its P V finished) before the stage's
                    // full barrier is waited on for tile g: with two V stages that
                    // barrier could otherwise still be two phases back, where its
                    // parity reads the same as tile g's
                    if (!wait_prev_pv()) { ok = false; break; }
                    if (!__all_sync(0xffffffffu, mbar_wait(v_full + 8 * vs, (g / VST) & 1, P.status))) { ok = false; break; }
                    if (!in) {
#pragma unroll
                        for (int sl_i = 0; sl_i < L::NSLAB; ++sl_i) {
                            uint8_t* vrow = base + L::kV + vs * L::kOp + sl_i * L::kSlab + ell * 128;
#pragma unroll
                            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + 16 * c) = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                // tile maxima of head h's rows: over its 16 tokens (a half-warp)
                float mt[R];
                {
                    float a[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) a[r] = s[r];
                    HRed<8, R, true>::run(a, lane);
#pragma unroll
                    for (int r = 0; r < R; ++r) mt[r] = __shfl_sync(0xffffffffu, a[0], (lane & 16) | (r << kSh));
                }
                // running max, moved only when a row's maximum grows by more than
                // 2^8 (the 16 lanes of a head take the same decisions)
                float alpha[R];
                bool resc = false;
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float mts = mt[r] * sl;
                    const bool grow = (m_ref[r] == -INFINITY) ? (mt[r] != -INFINITY) : (mts > m_ref[r] + kThinLazy);
                    alpha[r] = 1.f;
                    if (grow) {
                        alpha[r] = fast_exp2(m_ref[r] - mts);   // 0 when nothing was accumulated
                        resc = resc || m_ref[r] != -INFINITY;
                        lp[r] *= alpha[r];
                        m_ref[r] = mts;
                    }
                }
                if (j >= 2) {
                    if (!wait_prev_pv()) { ok = false; break; }
                    // a rescale of O^T touches every lane (channel): the group's heads
                    // vote. The vote area alternates, so the vote after next reuses it
                    // when every thread has read it.
                    float* vb = vote + (n_vote & 1) * HB * (R + 1);
                    if (t == 0) {
                        vb[h * (R + 1)] = resc ? 1.f : 0.f;
#pragma unroll
                        for (int r = 0; r < R; ++r) vb[h * (R + 1) + 1 + r] = alpha[r];
                    }
                    mbar_arrive(vote_bar + 8 * w);
                    if (!__all_sync(0xffffffffu, mbar_wait(vote_bar + 8 * w, n_vote++ & 1, P.status))) { ok = false; break; }
                    bool any = false;
#pragma unroll
                    for (int h2 = 0; h2 < HB; ++h2) any = any || vb[h2 * (R + 1)] != 0.f;
                    if (any) {
#pragma unroll 1
                        for (int h2 = 0; h2 < HB; ++h2) {
                            uint32_t o[16];
                            umma::ld16(lane_addr + L::colO(w) + 16 * h2, o);
                            umma::wait_ld();
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                const float a = vb[h2 * (R + 1) + 1 + r];
                                o[r] = __float_as_uint(__uint_as_float(o[r]) * a);
                                o[R + r] = __float_as_uint(__uint_as_float(o[R + r]) * a);
                            }
                            umma::st16(lane_addr + L::colO(w) + 16 * h2, o);
                        }
                        umma::wait_st();
                    }
                }
                // P^T = 2^(s sl - m) into shared memory as bf16, hi in row r and lo in
                // row R + r (K-major: lane ell at slab ell / 64, 16-byte unit (ell % 64) / 8)
                {
                    uint8_t* pb = base + L::kP + w * L::kPBuf + (ell / 64) * L::kPSlab + (ell % 8) * 2;
                    const int pc = (ell % 64) / 8;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const float mu = m_ref[r] == -INFINITY ? 0.f : m_ref[r];
                        const float p = fast_exp2(fmaf(s[r], sl, -mu));
                        lp[r] += p;
                        const __nv_bfloat16 hi = __float2bfloat16_rn(p);
                        const __nv_bfloat16 lo = __float2bfloat16_rn(p - __bfloat162float(hi));
                        *reinterpret_cast<__nv_bfloat16*>(pb + swz(r, pc)) = hi;
                        *reinterpret_cast<__nv_bfloat16*>(pb + swz(R + r, pc)) = lo;
                    }
                }
                fence_proxy_async_smem();   // P^T and zeroed V rows are read by the tensor core
                umma::fence_before_sync();
                mbar_arrive(p_full + 8 * w);
            }
            if (!ok) break;
            // ---- epilogue: each group's row sums and maxima, then the two
            // accumulators merged; group 0 writes heads 0-3, group 1 heads 4-7
            float* sums = reinterpret_cast<float*>(base + L::kSum) + (n_done & 1) * 2 * 2 * HB * R;   // [group][2][head][R]
            {
                float a[R];
#pragma unroll
                for (int r = 0; r < R; ++r) a[r] = lp[r];
                HRed<8, R, false>::run(a, lane);
                float* mine = sums + w * 2 * HB * R;
                if ((lane & ((1 << kSh) - 1)) == 0) mine[h * R + ((lane & 15) >> kSh)] = a[0];
                if (t == 0) {
#pragma unroll
                    for (int r = 0; r < R; ++r) mine[HB * R + h * R + r] = m_ref[r];
                }
            }
            mbar_arrive(lsum_bar);
            if (!__all_sync(0xffffffffu, mbar_wait(lsum_bar, n_done & 1, P.status))) { ok = false; break; }
            if (!__all_sync(0xffffffffu, mbar_wait(o_full, n_done & 1, P.status))) { ok = false; break; }
            umma::fence_after_sync();
            const bool has1 = n >= 2;   // the groups that saw a tile of the item
            const bool has0 = true;
#pragma unroll 1
            for (int h2 = 4 * w; h2 < 4 * w + 4; ++h2) {
                uint32_t o0[16], o1[16];
                if (has0) umma::ld16(lane_addr + L::colO(0) + 16 * h2, o0);
                if (has1) umma::ld16(lane_addr + L::colO(1) + 16 * h2, o1);
                umma::wait_ld();
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    if (r >= rows_here) break;
                    const float l0 = sums[h2 * R + r], m0 = sums[HB * R + h2 * R + r];
                    const float l1 = sums[2 * HB * R + h2 * R + r], m1 = sums[3 * HB * R + h2 * R + r];
                    const float M = fmaxf(has0 ? m0 : -INFINITY, has1 ? m1 : -INFINITY);
                    const float Mu = M == -INFINITY ? 0.f : M;
                    const float w0 = has0 ? fast_exp2(m0 - Mu) : 0.f, w1 = has1 ? fast_exp2(m1 - Mu) : 0.f;
                    const float Lr = (has0 ? l0 * w0 : 0.f) + (has1 ? l1 * w1 : 0.f);
                    float acc = 0.f;
                    if (has0) acc += (__uint_as_float(o0[r]) + __uint_as_float(o0[R + r])) * w0;
                    if (has1) acc += (__uint_as_float(o1[r]) + __uint_as_float(o1[R + r])) * w1;
                    const int row = row0 + r;
                    const int64_t prow =
                        (int64_t)C.part_base + (int64_t)(row / G) * Hq + (it.kv_head + h2) * G + row % G;
                    P.part_o[prow * D + ell] = Lr > 0.f ? acc / Lr : 0.f;
                    if (ell == 0) P.part_lse[prow] = Lr > 0.f ? M + __log2f(Lr) : -INFINITY;
                }
            }
            // the next item's first P V of either group overwrites an accumulator
            // the other group may still be reading
            mbar_arrive(epi_bar);
            if (!__all_sync(0xffffffffu, mbar_wait(epi_bar, n_done & 1, P.status))) { ok = false; break; }
            gbase += n;
            ++n_done;
        }
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int R>
cudaError_t launch_thin_r(const DevPlan& P, const CUtensorMap* tk, const CUtensorMap* tv, const void* Q, int n_items,
                          int item_off, int counter, cudaStream_t st, bool pdl) {
    const size_t smem = 1024 + ThinLayout<R>::kBytes;
    static DeviceOnce once;   // per device: the shared-memory limit, the SM count
    int sms = 0;
    cudaError_t e = per_device(once, &sms, nullptr, [&](int dev_id, int* a, int*) {
        cudaError_t r = cudaFuncSetAttribute(pac_thin_kernel<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (r != cudaSuccess) return r;
        return cudaDeviceGetAttribute(a, cudaDevAttrMultiProcessorCount, dev_id);
    });
    if (e != cudaSuccess) return e;
    const int grid = std::min(n_items, sms);
    return launch_kernel(pac_thin_kernel<R>, dim3(grid), dim3(kThinThreads), smem, st, pdl, P, *tk, *tv,
                         static_cast<const __nv_bfloat16*>(Q), item_off, n_items, counter);
}

}  // namespace dev

// rows_per_head: the items' row block (4 or 8); tk5 / tv5: the pools' 5-D maps
cudaError_t launch_pac_thin(const DevPlan& P, const void* tk5, const void* tv5, const void* Q, int rows_per_head,
                            int n_items, int item_off, int counter, cudaStream_t st, bool pdl) {
    if (P.d != 128 || P.n_kv_heads % kThinHeads) return cudaErrorInvalidValue;
    if (n_items <= 0) return cudaSuccess;
    const CUtensorMap* k = static_cast<const CUtensorMap*>(tk5);
    const CUtensorMap* v = static_cast<const CUtensorMap*>(tv5);
    return rows_per_head == 4 ? dev::launch_thin_r<4>(P, k, v, Q, n_items, item_off, counter, st, pdl)
                              : dev::launch_thin_r<8>(P, k, v, Q, n_items, item_off, counter, st, pdl);
}

}  // namespace pst
