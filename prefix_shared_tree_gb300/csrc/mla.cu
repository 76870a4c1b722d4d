// pst_mla_reconstruct: per-head K/V blocks rebuilt from a latent KV cache
// (multi-head latent attention), after which the same prefix-aware PAC and
// POR pipeline runs on them (CoDec, "supplementary details": the kernel module
// paragraph on MLA models).
//
// Every token j of the tree has a latent vector c_j of d_c channels; kv head h
// has up-projections W_UK[h], W_UV[h] of d x d_c, and
//     k_{h,j} = W_UK[h] c_j,   v_{h,j} = W_UV[h] c_j,
// stored as bf16 in the pools' layout [page][head][row][d]. Each page the
// tree uses is rebuilt once, however many queries share it: the prefix
// sharing of the attention carries over to the rebuild.
//
// One thread block takes 8 pages (128 latent rows: the M side of a tcgen05
// MMA) and a range of kv heads. The latent tile stays in shared memory (one
// TMA box of 16 rows x 64 channels per page and 128-byte slab); the weight
// rows of each (head, K or V) stream through a three-stage ring, two slabs per
// stage, as the N x K operand (N = d output channels); the products
// accumulate in tensor memory, double-buffered so that four epilogue warps
// convert one head's rows to bf16 and store them while the next head's MMAs
// run. Warp roles: 0 TMA producer, 1 tensor-memory owner and MMA issuer,
// 2-5 epilogue (tensor-memory lane quarter = warp % 4).
#include <string>

#include "dev_common.cuh"
#include "umma.cuh"

namespace pst {

int encode_bf16_map(void* out, int rank, const void* base, const uint64_t* dims, const uint64_t* strides,
                    const uint32_t* box);
int device_sm_count(int* out);

namespace dev {

constexpr int kMlaRows = 128;                     // latent rows per block (MMA M)
constexpr int kMlaPages = kMlaRows / kBoxRows;    // 8 pages of 16 rows
constexpr int kMlaStages = 3;                     // weight ring
constexpr int kMlaSlabsPerStage = 2;              // 128 latent channels per stage
constexpr int kMlaMaxSlabs = 8;                   // d_c <= 512
constexpr int kMlaThreads = 6 * 32;

template <int D>
struct MlaLayout {
    static constexpr uint32_t kASlab = kMlaRows * 128;                 // [128 rows][128 B]
    static constexpr uint32_t kBSlab = D * 128;                        // [D rows][128 B]
    static constexpr uint32_t kBStage = kMlaSlabsPerStage * kBSlab;
    static constexpr uint32_t kA = 0;
    static constexpr uint32_t kB = kA + kMlaMaxSlabs * kASlab;
    static constexpr uint32_t kBars = kB + kMlaStages * kBStage;
    // a_full, b_full[ST], b_empty[ST], acc_full[2], acc_empty[2], mma_done
    static constexpr int kNumBars = 1 + 2 * kMlaStages + 5;
    static constexpr uint32_t kTslot = kBars + 8 * kNumBars;
    static constexpr uint32_t kPages = kTslot + 16;                     // int32 [8]
    static constexpr uint32_t kBytes = kPages + 4 * kMlaPages;
    static_assert(kBytes + 1024 <= 232448, "shared memory");
    static constexpr uint32_t kTmemCols = 2 * D;                        // two accumulators
};

struct MlaArgs {
    const int32_t* pages;   // the tree's pages, ascending
    int32_t n_pages;
    int32_t d_c;            // latent channels (a multiple of 128, at most 512)
    int32_t n_kv_heads;
    int32_t heads_per_block;
    int32_t page_size;
    __nv_bfloat16* k_pool;
    __nv_bfloat16* v_pool;
    int32_t* status;
};

template <int D>
__global__ void __launch_bounds__(kMlaThreads, 1)
mla_rebuild_kernel(MlaArgs A, const __grid_constant__ CUtensorMap tc, const __grid_constant__ CUtensorMap tuk,
                   const __grid_constant__ CUtensorMap tuv) {
    using L = MlaLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(base);
    const uint32_t sA = sbase + L::kA, sB = sbase + L::kB;
    const uint32_t a_full = sbase + L::kBars;
    const uint32_t b_full = a_full + 8, b_empty = b_full + 8 * kMlaStages;
    const uint32_t acc_full = b_empty + 8 * kMlaStages, acc_empty = acc_full + 16, mma_done = acc_empty + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L::kTslot);
    int32_t* tile_pages = reinterpret_cast<int32_t*>(base + L::kPages);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h0 = blockIdx.y * A.heads_per_block;
    const int n_pairs = 2 * A.heads_per_block;         // (head, K or V) products of this block
    const int n_slabs = A.d_c / 64;
    const int n_chunks = n_slabs / kMlaSlabsPerStage;  // weight stages per product

    if (threadIdx.x < kMlaPages) {
        const int i = blockIdx.x * kMlaPages + threadIdx.x;
        tile_pages[threadIdx.x] = i < A.n_pages ? A.pages[i] : -1;
    }
    if (threadIdx.x == 0) {
        mbar_init(a_full, 1);
        for (int s = 0; s < kMlaStages; ++s) {
            mbar_init(b_full + 8 * s, 1);
            mbar_init(b_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + 8 * b, 1);
            mbar_init(acc_empty + 8 * b, 128);
        }
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

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tc);
            prefetch_tmap(&tuk);
            prefetch_tmap(&tuv);
            int valid = 0;
            for (int p = 0; p < kMlaPages; ++p) valid += tile_pages[p] >= 0;
            // the latent tile: page p's rows land at rows 16p.. of every slab
            mbar_arrive_expect_tx(a_full, (uint32_t)(valid * n_slabs * kBoxRows * 128));
            for (int p = 0; p < kMlaPages; ++p) {
                const int page = tile_pages[p];
                if (page < 0) continue;
                for (int s = 0; s < n_slabs; ++s)
                    tma_load_3d(sA + s * L::kASlab + p * kBoxRows * 128, &tc, 64 * s, 0, page, a_full);
            }
            // weight rows of each product, two slabs per stage
            int issued = 0;
            bool ok = true;
            for (int pr = 0; pr < n_pairs && ok; ++pr) {
                const CUtensorMap* w = (pr & 1) ? &tuv : &tuk;
                const int h = h0 + pr / 2;
                for (int c = 0; c < n_chunks; ++c, ++issued) {
                    const int s = issued % kMlaStages;
                    if (issued >= kMlaStages &&
                        !mbar_wait(b_empty + 8 * s, ((issued / kMlaStages) - 1) & 1, A.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(b_full + 8 * s, L::kBStage);
                    for (int j = 0; j < kMlaSlabsPerStage; ++j)
                        tma_load_3d(sB + s * L::kBStage + j * L::kBSlab, w, 64 * (kMlaSlabsPerStage * c + j), 0, h,
                                    b_full + 8 * s);
                }
            }
            // every load issued has landed before the block can leave
            mbar_wait(a_full, 0, A.status);
            drain_ring<kMlaStages>(b_full, issued, A.status);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = umma::idesc_bf16_f32(kMlaRows, D, 0, 0);
            const uint64_t da = umma::smem_desc_sw128(sA, 16, 1024);
            const uint64_t db = umma::smem_desc_sw128(sB, 16, 1024);
            bool ok = mbar_wait(a_full, 0, A.status);
            umma::fence_after_sync();
            int used = 0;
            for (int pr = 0; pr < n_pairs && ok; ++pr) {
                const int buf = pr & 1;
                if (pr >= 2 && !mbar_wait(acc_empty + 8 * buf, ((pr >> 1) - 1) & 1, A.status)) { ok = false; break; }
                umma::fence_after_sync();
                const uint32_t dst = tmem + buf * D;
                for (int c = 0; c < n_chunks; ++c, ++used) {
                    const int s = used % kMlaStages;
                    if (!mbar_wait(b_full + 8 * s, (used / kMlaStages) & 1, A.status)) { ok = false; break; }
                    umma::fence_after_sync();
#pragma unroll
                    for (int j = 0; j < kMlaSlabsPerStage; ++j) {
                        const int slab = kMlaSlabsPerStage * c + j;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma::mma_bf16_ss(dst, da + ((slab * L::kASlab + kk * 32) >> 4),
                                              db + ((s * L::kBStage + j * L::kBSlab + kk * 32) >> 4), idesc,
                                              (c | j | kk) ? 1u : 0u);
                    }
                    umma::commit(b_empty + 8 * s);
                }
                if (!ok) break;
                umma::commit(acc_full + 8 * buf);
            }
            // every MMA issued has finished before tensor memory is released
            // (also when a wait above gave up)
            umma::commit(mma_done);
            mbar_wait(mma_done, 0, A.status);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp % 4;
        const int r = 32 * quarter + lane;                 // latent row = tensor-memory lane
        const int page = tile_pages[r / kBoxRows];
        const int prow = r % kBoxRows;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
        for (int pr = 0; pr < n_pairs; ++pr) {
            const int buf = pr & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(acc_full + 8 * buf, (pr >> 1) & 1, A.status))) break;
            umma::fence_after_sync();
            const int h = h0 + pr / 2;
            __nv_bfloat16* pool = (pr & 1) ? A.v_pool : A.k_pool;
            uint4* dst = page >= 0 ? reinterpret_cast<uint4*>(
                                         pool + (((int64_t)page * A.n_kv_heads + h) * A.page_size + prow) * D)
                                   : nullptr;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                float v[32];
                umma::ld32(lane_addr + buf * D + 32 * c, v);
                umma::wait_ld();
                if (dst) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint4 q;
                        __nv_bfloat162 b0 = __floats2bfloat162_rn(v[8 * u + 0], v[8 * u + 1]);
                        __nv_bfloat162 b1 = __floats2bfloat162_rn(v[8 * u + 2], v[8 * u + 3]);
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * u + 4], v[8 * u + 5]);
                        __nv_bfloat162 b3 = __floats2bfloat162_rn(v[8 * u + 6], v[8 * u + 7]);
                        q.x = *reinterpret_cast<uint32_t*>(&b0);
                        q.y = *reinterpret_cast<uint32_t*>(&b1);
                        q.z = *reinterpret_cast<uint32_t*>(&b2);
                        q.w = *reinterpret_cast<uint32_t*>(&b3);
                        dst[4 * c + u] = q;
                    }
                }
            }
            umma::fence_before_sync();
            mbar_arrive(acc_empty + 8 * buf);
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
cudaError_t launch_mla_d(const MlaArgs& a, const CUtensorMap* tc, const CUtensorMap* tuk, const CUtensorMap* tuv,
                         int tiles, int splits, cudaStream_t st) {
    const size_t smem = 1024 + MlaLayout<D>::kBytes;
    static DeviceOnce once;   // per device: the shared-memory limit
    cudaError_t e = per_device(once, nullptr, nullptr, [&](int, int* x, int*) {
        *x = 1;
        return cudaFuncSetAttribute(mla_rebuild_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (e != cudaSuccess) return e;
    return launch_kernel(mla_rebuild_kernel<D>, dim3(tiles, splits), dim3(kMlaThreads), smem, st, false, a, *tc,
                         *tuk, *tuv);
}

}  // namespace dev
}  // namespace pst

using namespace pst;

extern "C" int pst_mla_reconstruct(const pst_plan* p, const void* C_pool, int32_t d_c, const void* W_uk,
                                   const void* W_uv, void* K_pool, void* V_pool, void* stream) {
    if (!p) return fail(PST_EINVAL, "mla_reconstruct: plan is null");
    if (!p->d_ws) return fail(PST_EWORKSPACE, "mla_reconstruct: plan has no uploaded workspace");
    if (!C_pool || !W_uk || !W_uv || !K_pool || !V_pool) return fail(PST_EINVAL, "mla_reconstruct: null pointer");
    if (p->dtype != PST_BF16) return fail(PST_EUNSUPPORTED, "mla_reconstruct: bf16 plans only");
    if (d_c < 128 || d_c > 512 || d_c % 128)
        return fail(PST_EUNSUPPORTED, "mla_reconstruct: d_c must be 128, 256, 384 or 512");
    if (p->page_size != kBoxRows) return fail(PST_EUNSUPPORTED, "mla_reconstruct: page size must be 16");
    if ((reinterpret_cast<uintptr_t>(C_pool) | reinterpret_cast<uintptr_t>(W_uk) | reinterpret_cast<uintptr_t>(W_uv) |
         reinterpret_cast<uintptr_t>(K_pool) | reinterpret_cast<uintptr_t>(V_pool)) % 16)
        return fail(PST_EINVAL, "mla_reconstruct: every pointer must be 16-byte aligned");
    const int64_t n_pages = (int64_t)p->tree_pages.size();
    if (n_pages == 0) return PST_OK;
    // latent pool [num_pages][page_size][d_c]; weights [Hkv][d][d_c]
    alignas(64) unsigned char tc[128], tuk[128], tuv[128];
    {
        const uint64_t dims[3] = {(uint64_t)d_c, (uint64_t)p->page_size, (uint64_t)p->num_pages};
        const uint64_t str[2] = {(uint64_t)d_c * 2, (uint64_t)p->page_size * d_c * 2};
        const uint32_t box[3] = {64, (uint32_t)kBoxRows, 1};
        int rc = encode_bf16_map(tc, 3, C_pool, dims, str, box);
        if (rc) return rc;
    }
    for (int k = 0; k < 2; ++k) {
        const uint64_t dims[3] = {(uint64_t)d_c, (uint64_t)p->d, (uint64_t)p->hkv};
        const uint64_t str[2] = {(uint64_t)d_c * 2, (uint64_t)p->d * d_c * 2};
        const uint32_t box[3] = {64, (uint32_t)p->d, 1};
        int rc = encode_bf16_map(k ? tuv : tuk, 3, k ? W_uv : W_uk, dims, str, box);
        if (rc) return rc;
    }
    dev::MlaArgs a;
    a.pages = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(p->d_ws) + p->ws.tree_pages);
    a.n_pages = (int32_t)n_pages;
    a.d_c = d_c;
    a.n_kv_heads = p->hkv;
    a.page_size = p->page_size;
    a.k_pool = static_cast<__nv_bfloat16*>(K_pool);
    a.v_pool = static_cast<__nv_bfloat16*>(V_pool);
    a.status = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(p->d_ws) + p->ws.status);
    // blocks: page tiles x head ranges, the heads split (in halves) until the
    // grid has about two blocks per SM or a block holds one head
    const int tiles = (int)((n_pages + dev::kMlaPages - 1) / dev::kMlaPages);
    int sms = 0;
    if (device_sm_count(&sms) != 0 || sms <= 0) sms = 148;
    int splits = 1;
    while ((int64_t)tiles * splits < 2LL * sms && p->hkv % (2 * splits) == 0) splits *= 2;
    a.heads_per_block = p->hkv / splits;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e =
        p->d == 128
            ? dev::launch_mla_d<128>(a, reinterpret_cast<const CUtensorMap*>(tc),
                                     reinterpret_cast<const CUtensorMap*>(tuk), reinterpret_cast<const CUtensorMap*>(tuv),
                                     tiles, splits, st)
            : dev::launch_mla_d<64>(a, reinterpret_cast<const CUtensorMap*>(tc),
                                    reinterpret_cast<const CUtensorMap*>(tuk), reinterpret_cast<const CUtensorMap*>(tuv),
                                    tiles, splits, st);
    if (e != cudaSuccess)
        return fail(PST_ECUDA, std::string("mla_reconstruct: launch: ") + cudaGetErrorName(e) + " (" +
                                   cudaGetErrorString(e) + ")");
    return PST_OK;
}
