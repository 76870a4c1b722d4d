// CUDA-core partial attention computation (PAC) for thin chunks: fewer than
// 16 query rows (aggregated queries x GQA group) per kv head.
//
// CoDec, "intra-block primitives": a PAC computes attention between the
// queries aggregated on a KV node and that node's K/V, loading each K/V tile
// into shared memory once for all of them, and emits a partial output with
// its softmax statistics. CoDec, "KV cache management": node-local
// stabilisation -- per row a running max m and sum of e^{s-m}, rescaled to
// the larger max when a new block is folded in.
//
// Layout of the work: one thread block per (chunk, kv head, row block of up
// to 8 rows). A producer warp streams the chunk's pages with TMA into a
// 2-stage ring (128B-swizzled 16-row boxes). Each of 4 compute warps owns 16
// rows of every 64-token tile; inside a warp, groups of LPT lanes each take
// one token at a time with the channels split across the group's lanes
// (16-byte vector reads of the staged rows). Dot products are reduced across
// the group with a transposing butterfly, so each lane ends up holding the
// score of one row; every group keeps its own running (m, l, O) and the
// groups, then the warps, are merged with the same rescaling rule at the end.
#include <algorithm>

#include "dev_common.cuh"

namespace pst {
namespace dev {

constexpr int kCcWarps = 4;
constexpr int kCcStages = 2;

template <typename T>
struct ElemTraits;
template <>
struct ElemTraits<__nv_bfloat16> {
    static constexpr int kBytes = 2;
    // 16-byte chunk -> 8 floats
    __device__ __forceinline__ static void unpack(const uint4& v, float* out) {
        out[0] = bf16lo(v.x); out[1] = bf16hi(v.x);
        out[2] = bf16lo(v.y); out[3] = bf16hi(v.y);
        out[4] = bf16lo(v.z); out[5] = bf16hi(v.z);
        out[6] = bf16lo(v.w); out[7] = bf16hi(v.w);
    }
    // 16-byte chunk -> 4 packed pairs (element order kept)
    __device__ __forceinline__ static void unpack2(const uint4& v, u64* out) {
        out[0] = pk2(bf16lo(v.x), bf16hi(v.x));
        out[1] = pk2(bf16lo(v.y), bf16hi(v.y));
        out[2] = pk2(bf16lo(v.z), bf16hi(v.z));
        out[3] = pk2(bf16lo(v.w), bf16hi(v.w));
    }
};
template <>
struct ElemTraits<float> {
    static constexpr int kBytes = 4;
    __device__ __forceinline__ static void unpack(const uint4& v, float* out) {
        out[0] = __uint_as_float(v.x); out[1] = __uint_as_float(v.y);
        out[2] = __uint_as_float(v.z); out[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static void unpack2(const uint4& v, u64* out) {
        out[0] = (u64)v.x | ((u64)v.y << 32);
        out[1] = (u64)v.z | ((u64)v.w << 32);
    }
};

// Sum RT per-lane values over the LPT lanes of a group; afterwards lane j of
// the group holds the total of value index j >> (log2 LPT - log2 RT). Each
// butterfly stage with N > 1 live values sends half of them to the partner
// lane and keeps the other half (transposing as it reduces); once one value
// is left the remaining stages are plain sums.
template <int OFF, int N>
struct ReduceStep {
    template <int RT>
    __device__ __forceinline__ static void run(float (&a)[RT], int j) {
        if constexpr (OFF >= 1) {
            if constexpr (N > 1) {
                constexpr int H = N / 2;
                const bool up = (j & OFF) != 0;
#pragma unroll
                for (int i = 0; i < H; ++i) {
                    const float send = up ? a[i] : a[i + H];
                    const float keep = up ? a[i + H] : a[i];
                    a[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
                }
                ReduceStep<OFF / 2, H>::run(a, j);
            } else {
                a[0] += __shfl_xor_sync(0xffffffffu, a[0], OFF);
                ReduceStep<OFF / 2, 1>::run(a, j);
            }
        }
    }
};

template <int LPT, int RT>
__device__ __forceinline__ float reduce_transpose(float (&a)[RT], int j) {
    ReduceStep<LPT / 2, RT>::run(a, j);
    return a[0];
}

template <int LPT, int RT>
__device__ __forceinline__ constexpr int owner_shift() {
    return (LPT == 8 ? 3 : LPT == 16 ? 4 : 5) - (RT == 1 ? 0 : RT == 2 ? 1 : RT == 4 ? 2 : 3);
}
static_assert(owner_shift<8, 8>() == 0, "owner shift");

// One chunk x kv head x row block on the compute warps; `tbase` tiles went
// through the ring before it. Returns false if a wait gave up.
template <typename T, int D, int LPT, int RT>
__device__ __forceinline__ bool cc_consume(const DevPlan& P, const DevChunk& C, int head, int rb, const T* __restrict__ Q,
                           uint32_t ring, const uint8_t* ring_ptr, uint32_t bar_full, uint32_t bar_empty,
                           float* scratch, int tbase) {
    constexpr int EB = ElemTraits<T>::kBytes;
    constexpr int ROWB = D * EB;            // bytes per K/V row
    constexpr int NSLAB = ROWB / 128;
    constexpr int CHUNKS = ROWB / 16;
    constexpr int CPL = CHUNKS / LPT;       // 16-byte chunks per lane
    constexpr int EPC = 16 / EB;            // elements per chunk
    constexpr int EPL = CPL * EPC;          // elements per lane
    constexpr int TPI = 32 / LPT;           // tokens per warp step
    constexpr int BT = 16 / TPI;            // tokens per group per tile
    constexpr int SH = owner_shift<LPT, RT>();
    constexpr uint32_t kSlabBytes = kTileTokens * 128;
    constexpr uint32_t kHalf = NSLAB * kSlabBytes;
    static_assert(CPL >= 1, "lane mapping");

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int grp = lane / LPT, j = lane % LPT;
    const int G = P.group, Hq = P.n_q_heads;
    const int rows_total = C.n_q * G;
    const int own = j >> SH;                // row whose score this lane holds

    // ---- queries of this row block, channels of this lane, pre-scaled to log2
    // units, kept as packed pairs for the f32x2 FMA
    constexpr int EP2 = EPL / 2;
    u64 q2[RT][EP2];
    uint64_t own_mask = ~0ull;
#pragma unroll
    for (int r = 0; r < RT; ++r) {
        const int row = rb * RT + r;
        float qf[EPL];
        if (row < rows_total) {
            const int qi = row / G, gh = row % G;
            const int qid = P.chunk_q[C.q_base + qi];
            const T* qrow = Q + ((int64_t)qid * Hq + head * G + gh) * D;
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
                const int gc = j + k * LPT;
                const uint4 v = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(qrow) + gc * 16);
                ElemTraits<T>::unpack(v, qf + k * EPC);
            }
#pragma unroll
            for (int e = 0; e < EPL; ++e) qf[e] *= P.scale_log2;
            if (r == own && C.mask_base >= 0) own_mask = P.masks[C.mask_base + qi];
        } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) qf[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < EP2; ++e) q2[r][e] = pk2(qf[2 * e], qf[2 * e + 1]);
    }

    u64 o2[RT][EP2];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int e = 0; e < EP2; ++e) o2[r][e] = 0ull;
    float m_run = -INFINITY, l_run = 0.f;

    const ChunkGeo g = chunk_geo(C);
    const int owner_base = grp * LPT;
    // shared-memory byte offsets of this lane's chunks in the rows it reads
    // (row & 7 only depends on grp and b, the tile base is 1024-aligned)
    uint32_t off[BT][CPL];
#pragma unroll
    for (int b = 0; b < BT; ++b)
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            const int row = warp * 16 + grp + TPI * b, gc = j + k * LPT;
            off[b][k] = (gc / 8) * kSlabBytes + swz(row, gc % 8);
        }
    bool ok = true;
    for (int i = 0; i < g.n_tiles; ++i) {
        const int s = (tbase + i) % kCcStages;
        if (!mbar_wait(bar_full + 8 * s, ((tbase + i) / kCcStages) & 1, P.status)) { ok = false; break; }
        const uint8_t* kb = ring_ptr + s * 2 * kHalf;
        const uint8_t* vb = kb + kHalf;
        const int tpos = g.tile0 + i * kTileTokens;
        const bool edge = tpos < g.pos_begin || tpos + kTileTokens > g.pos_end || C.mask_base >= 0;

        float sc[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            u64 k2[EP2];
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
                const uint4 v = *reinterpret_cast<const uint4*>(kb + off[b][k]);
                ElemTraits<T>::unpack2(v, k2 + k * (EPC / 2));
            }
            float pd[RT];
#pragma unroll
            for (int r = 0; r < RT; ++r) {
                u64 acc = fma2(q2[r][0], k2[0], 0ull);
#pragma unroll
                for (int e = 1; e < EP2; ++e) acc = fma2(q2[r][e], k2[e], acc);
                float a0, a1;
                upk2(acc, a0, a1);
                pd[r] = a0 + a1;
            }
            const float sv = reduce_transpose<LPT, RT>(pd, j);
            sc[b] = sv;
            if (edge) {
                const int pos = tpos + warp * 16 + grp + TPI * b;
                const int t = pos - g.pos_begin;
                bool valid = pos >= g.pos_begin && pos < g.pos_end;
                if (valid && t < 64) valid = (own_mask >> t) & 1ull;
                sc[b] = valid ? sv : -INFINITY;
            }
        }
        float mb = sc[0];
#pragma unroll
        for (int b = 1; b < BT; ++b) mb = fmaxf(mb, sc[b]);
        const float m_new = fmaxf(m_run, mb);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = fast_exp2(m_run - m_use);
        float p[BT];
        float ps = 0.f;
#pragma unroll
        for (int b = 0; b < BT; ++b) { p[b] = fast_exp2(sc[b] - m_use); ps += p[b]; }
        l_run = l_run * alpha + ps;
        m_run = m_new;
#pragma unroll
        for (int r = 0; r < RT; ++r) {
            const float ar = __shfl_sync(0xffffffffu, alpha, owner_base + (r << SH));
            const u64 a2 = pk2(ar, ar);
#pragma unroll
            for (int e = 0; e < EP2; ++e) o2[r][e] = mul2(o2[r][e], a2);
        }
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            float pr[RT];
#pragma unroll
            for (int r = 0; r < RT; ++r) pr[r] = __shfl_sync(0xffffffffu, p[b], owner_base + (r << SH));
            bool tok_ok = true;
            if (edge) {
                const int pos = tpos + warp * 16 + grp + TPI * b;
                tok_ok = pos >= g.pos_begin && pos < g.pos_end;
            }
            if (tok_ok) {
                u64 v2[EP2];
#pragma unroll
                for (int k = 0; k < CPL; ++k) {
                    const uint4 v = *reinterpret_cast<const uint4*>(vb + off[b][k]);
                    ElemTraits<T>::unpack2(v, v2 + k * (EPC / 2));
                }
#pragma unroll
                for (int r = 0; r < RT; ++r) {
                    const u64 p2 = pk2(pr[r], pr[r]);
#pragma unroll
                    for (int e = 0; e < EP2; ++e) o2[r][e] = fma2(p2, v2[e], o2[r][e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
    float o[RT][EPL];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int e = 0; e < EP2; ++e) upk2(o2[r][e], o[r][2 * e], o[r][2 * e + 1]);

    // ---- merge the groups of this warp (butterfly over the group bits)
    float mr[RT], lr[RT];
#pragma unroll
    for (int r = 0; r < RT; ++r) {
        mr[r] = __shfl_sync(0xffffffffu, m_run, owner_base + (r << SH));
        lr[r] = __shfl_sync(0xffffffffu, l_run, owner_base + (r << SH));
    }
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
        for (int r = 0; r < RT; ++r) {
            const float m2 = __shfl_xor_sync(0xffffffffu, mr[r], off);
            const float l2 = __shfl_xor_sync(0xffffffffu, lr[r], off);
            const float M = fmaxf(mr[r], m2);
            const float Mu = M == -INFINITY ? 0.f : M;
            const float a1 = fast_exp2(mr[r] - Mu), a2 = fast_exp2(m2 - Mu);
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                const float o2 = __shfl_xor_sync(0xffffffffu, o[r][e], off);
                o[r][e] = o[r][e] * a1 + o2 * a2;
            }
            lr[r] = lr[r] * a1 + l2 * a2;
            mr[r] = M;
        }
    }
    // ---- across warps through shared memory: per warp [RT][D] O, [RT] m, [RT] l
    float* so = scratch + warp * RT * (D + 2);
    if (grp == 0) {
#pragma unroll
        for (int r = 0; r < RT; ++r)
#pragma unroll
            for (int k = 0; k < CPL; ++k)
#pragma unroll
                for (int e = 0; e < EPC; ++e) so[r * D + (j + k * LPT) * EPC + e] = o[r][k * EPC + e];
    }
    if (lane < RT) {
        so[RT * D + lane] = mr[lane];
        so[RT * D + RT + lane] = lr[lane];
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCcWarps * 32) : "memory");
    for (int r = warp; r < RT && ok; r += kCcWarps) {
        const int row = rb * RT + r;
        if (row >= rows_total) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCcWarps; ++w) M = fmaxf(M, scratch[w * RT * (D + 2) + RT * D + r]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float wts[kCcWarps], L = 0.f;
#pragma unroll
        for (int w = 0; w < kCcWarps; ++w) {
            const float* sw = scratch + w * RT * (D + 2);
            wts[w] = fast_exp2(sw[RT * D + r] - Mu);
            L += sw[RT * D + RT + r] * wts[w];
        }
        const int qi = row / G, gh = row % G;
        const int64_t prow = (int64_t)C.part_base + (int64_t)qi * Hq + head * G + gh;
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int dd = lane; dd < D; dd += 32) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kCcWarps; ++w) acc += scratch[w * RT * (D + 2) + r * D + dd] * wts[w];
            P.part_o[prow * D + dd] = acc * inv;
        }
        if (lane == 0) P.part_lse[prow] = L > 0.f ? M + __log2f(L) : -INFINITY;
    }
    // the next item reuses the scratch
    asm volatile("bar.sync 1, %0;" ::"r"(kCcWarps * 32) : "memory");
    return ok;
}

// Persistent: each block takes items (largest first) from a work queue, so
// blocks that start late, when tensor-core blocks leave their SMs, still
// share the work evenly. The producer warp claims the next item and hands
// its index to the compute warps through a 2-deep queue in shared memory.
template <typename T, int D, int RT>
__global__ void __launch_bounds__((kCcWarps + 1) * 32)
pac_cc_kernel(DevPlan P, const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
              const T* __restrict__ Q, int item_off, int n_items, int counter) {
    constexpr int EB = ElemTraits<T>::kBytes;
    constexpr int NSLAB = D * EB / 128;
    constexpr uint32_t kStage = 2 * NSLAB * kTileTokens * 128;
    extern __shared__ uint8_t smem_raw[];
    pdl_launch_dependents();   // the next launch group may take the SMs this grid leaves
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring = smem_u32(base);
    float* scratch = reinterpret_cast<float*>(base + kCcStages * kStage);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + kCcStages * kStage + kCcWarps * RT * (D + 2) * 4);
    const uint32_t bar_full = smem_u32(bars), bar_empty = smem_u32(bars + kCcStages);
    const uint32_t item_full = smem_u32(bars + 2 * kCcStages), item_empty = item_full + 16;
    volatile int* item_idx = reinterpret_cast<volatile int*>(bars + 2 * kCcStages + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kCcStages; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, kCcWarps);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(item_full + 8 * q, 1);
            mbar_init(item_empty + 8 * q, kCcWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == kCcWarps) {
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            int tbase = 0;
            for (int q = 0;; ++q) {
                const int slot = q & 1;
                if (q >= 2 && !mbar_wait(item_empty + 8 * slot, ((q >> 1) - 1) & 1, P.status)) break;
                const int idx = atomicAdd(P.counters + counter, 1);
                item_idx[slot] = idx < n_items ? idx : -1;
                mbar_arrive(item_full + 8 * slot);   // release: the index store is visible to the waiters
                if (idx >= n_items) break;
                const DevItem it = P.items[item_off + idx];
                const DevChunk C = P.chunks[it.chunk];
                if (!produce_chunk<NSLAB, kCcStages, 128 / EB>(P, C, it.kv_head, ring, bar_full, bar_empty, &tk, &tv,
                                                              tbase)) {
                    tbase = -1;
                    break;
                }
                tbase += chunk_geo(C).n_tiles;
            }
            if (tbase >= 0) producer_done<kCcStages>(bar_full, tbase, P.status);
        }
        return;
    }
    // lanes per token: 8 for one row, 16 for 2-4 rows, up to 32 for 8 rows,
    // never more than the 16-byte chunks of a row
    constexpr int CH = D * EB / 16;
    constexpr int LW = RT == 1 ? 8 : RT <= 4 ? 16 : 32;
    constexpr int LPT = CH < LW ? CH : LW;
    int tbase = 0;
    for (int q = 0;; ++q) {
        const int slot = q & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(item_full + 8 * slot, (q >> 1) & 1, P.status))) break;
        const int idx = item_idx[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(item_empty + 8 * slot);
        if (idx < 0) break;
        const DevItem it = P.items[item_off + idx];
        const DevChunk C = P.chunks[it.chunk];
        if (!cc_consume<T, D, LPT, RT>(P, C, it.kv_head, it.row_block, Q, ring, base, bar_full, bar_empty, scratch,
                                       tbase))
            break;
        tbase += chunk_geo(C).n_tiles;
    }
}

template <typename T, int D, int RT>
size_t cc_smem_bytes() {
    constexpr int EB = ElemTraits<T>::kBytes;
    constexpr int NSLAB = D * EB / 128;
    return 1024 + kCcStages * 2 * NSLAB * kTileTokens * 128 + kCcWarps * RT * (D + 2) * 4 + 2 * kCcStages * 8 + 48;
}

// Blocks that fit on the current device at once; sets the kernel's
// shared-memory limit on first use on each device. 0 if the runtime cannot say.
template <typename T, int D, int RT>
int cc_resident_blocks(int* per_sm_out = nullptr) {
    static DeviceOnce once;   // per device: resident blocks, blocks per SM
    int resident = 0, per_sm = 0;
    const cudaError_t e = per_device(once, &resident, &per_sm, [&](int dev, int* a, int* b) {
        const size_t smem = cc_smem_bytes<T, D, RT>();
        cudaError_t r = cudaFuncSetAttribute(pac_cc_kernel<T, D, RT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (r != cudaSuccess) return r;
        int n = 0, sms = 0;
        r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pac_cc_kernel<T, D, RT>, (kCcWarps + 1) * 32, smem);
        if (r != cudaSuccess) return r;
        r = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (r != cudaSuccess) return r;
        *b = std::max(1, n);
        *a = *b * std::max(1, sms);
        return cudaSuccess;
    });
    if (e != cudaSuccess) return 0;
    if (per_sm_out) *per_sm_out = per_sm;
    return resident;
}

template <typename T, int D, int RT>
cudaError_t launch_cc_rt(const DevPlan& P, const CUtensorMap* tk, const CUtensorMap* tv, const void* Q,
                         int n_items, int item_off, int counter, cudaStream_t st, bool pdl) {
    const size_t smem = cc_smem_bytes<T, D, RT>();
    const int resident = cc_resident_blocks<T, D, RT>();
    if (!resident) return cudaErrorInvalidConfiguration;
    const int grid = std::min(n_items, resident);
    return launch_kernel(pac_cc_kernel<T, D, RT>, dim3(grid), dim3((kCcWarps + 1) * 32), smem, st, pdl, P, *tk, *tv,
                         static_cast<const T*>(Q), item_off, n_items, counter);
}

template <typename T, int D>
int cc_per_sm_t(int r_tile) {
    int n = 0;
    switch (r_tile) {
        case 1: cc_resident_blocks<T, D, 1>(&n); break;
        case 2: cc_resident_blocks<T, D, 2>(&n); break;
        case 4: cc_resident_blocks<T, D, 4>(&n); break;
        default: cc_resident_blocks<T, D, 8>(&n); break;
    }
    return n > 0 ? n : -1;
}

template <typename T, int D>
cudaError_t launch_cc_t(const DevPlan& P, const CUtensorMap* tk, const CUtensorMap* tv, const void* Q, int r_tile,
                        int n_items, int item_off, int counter, cudaStream_t st, bool pdl) {
    switch (r_tile) {
        case 1: return launch_cc_rt<T, D, 1>(P, tk, tv, Q, n_items, item_off, counter, st, pdl);
        case 2: return launch_cc_rt<T, D, 2>(P, tk, tv, Q, n_items, item_off, counter, st, pdl);
        case 4: return launch_cc_rt<T, D, 4>(P, tk, tv, Q, n_items, item_off, counter, st, pdl);
        default: return launch_cc_rt<T, D, 8>(P, tk, tv, Q, n_items, item_off, counter, st, pdl);
    }
}

}  // namespace dev

int cc_blocks_per_sm(pst_dtype dt, int d, int r_tile) {
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
        cudaGetLastError();   // leave no sticky error behind
        return -1;
    }
    if (dt == PST_BF16) return d == 128 ? dev::cc_per_sm_t<__nv_bfloat16, 128>(r_tile) : dev::cc_per_sm_t<__nv_bfloat16, 64>(r_tile);
    return d == 128 ? dev::cc_per_sm_t<float, 128>(r_tile) : dev::cc_per_sm_t<float, 64>(r_tile);
}

cudaError_t launch_pac_cc(const DevPlan& P, pst_dtype dt, const void* tk, const void* tv, const void* Q,
                          int r_tile, int n_items, int item_off, int counter, cudaStream_t st, bool pdl) {
    const CUtensorMap* k = static_cast<const CUtensorMap*>(tk);
    const CUtensorMap* v = static_cast<const CUtensorMap*>(tv);
    if (dt == PST_BF16) {
        if (P.d == 128) return dev::launch_cc_t<__nv_bfloat16, 128>(P, k, v, Q, r_tile, n_items, item_off, counter, st, pdl);
        return dev::launch_cc_t<__nv_bfloat16, 64>(P, k, v, Q, r_tile, n_items, item_off, counter, st, pdl);
    }
    if (P.d == 128) return dev::launch_cc_t<float, 128>(P, k, v, Q, r_tile, n_items, item_off, counter, st, pdl);
    return dev::launch_cc_t<float, 64>(P, k, v, Q, r_tile, n_items, item_off, counter, st, pdl);
}

}  // namespace pst
