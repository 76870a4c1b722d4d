// Partial output reduction (POR) and the host side of pst_decode_attn:
// workspace binding, TMA descriptors, launches, timing and status.
//
// CoDec, "intra-block primitives", POR: two partial outputs O1, O2 of the same
// query with maxima m1, m2 and sums s1, s2 merge to m = max(m1, m2),
// s = s1 e^{m1-m} + s2 e^{m2-m}, O = (O1 s1 e^{m1-m} + O2 s2 e^{m2-m}) / s.
// CoDec, "inter-block launch and tree reduction": the merge is associative and
// commutative and the reductions of different queries are independent, so the
// tree reduction becomes one independent chain per query. Here each partial
// carries its log-sum-exp (base 2) lse_i = m_i + log2 s_i, which folds the
// two statistics into one: weights w_i = 2^{lse_i - max lse}; one warp per
// (query, q-head) merges all of the query's partials at once.
#include <cudaTypedefs.h>

#include <algorithm>
#include <chrono>
#include <cstdint>
#include <cmath>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "dev_common.cuh"

namespace pst {

cudaError_t launch_pac_cc(const DevPlan& P, pst_dtype dt, const void* tk, const void* tv, const void* Q,
                          int r_tile, int n_items, int item_off, int counter, cudaStream_t st, bool pdl);
cudaError_t launch_pac_tc(const DevPlan& P, const void* tk, const void* tv, const void* Q, int n_items,
                          int item_off, cudaStream_t st, bool pdl);
cudaError_t launch_pac_umma(const DevPlan& P, const void* tk, const void* tv, const void* tq, const void* Q,
                            int n_items, int item_off, bool exact_p, bool split_rows, cudaStream_t st, bool pdl);
cudaError_t launch_pac_thin(const DevPlan& P, const void* tk5, const void* tv5, const void* Q, int rows_per_head,
                            int n_items, int item_off, int counter, cudaStream_t st, bool pdl);

// Tensor-core PAC launch group g (pst_plan::tc_group_cnt): P rounded once
// (g < 2) or exact, more than 128 rows per block (even g) or at most 128.
// The mma.sync engine has all its items in group 1.
cudaError_t launch_tc_group(const pst_plan* p, const DevPlan& dp, const void* tk, const void* tv, const void* tq,
                            const void* Q, int g, LaunchSeq& ls) {
    int64_t off = 0;
    for (int k = 0; k < g; ++k) off += p->tc_group_cnt[k];
    const int n = (int)p->tc_group_cnt[g];
    if (n == 0) return cudaSuccess;
    if (p->opts.tc_engine == 1) return launch_pac_tc(dp, tk, tv, Q, n, (int)off, ls.st, ls.next_pdl());
    // d = 128: V in 4 KB page boxes (the pool's second 5-D view)
    const void* tv_umma = p->d == 128 ? static_cast<const void*>(static_cast<const unsigned char*>(tv) + 256) : tv;
    return launch_pac_umma(dp, tk, tv_umma, tq, Q, n, (int)off, g >= 2, (g & 1) == 0, ls.st, ls.next_pdl());
}

// Thin chunks: tcgen05 thin PAC launches for row blocks of 8 and of 4 (work
// counters 4, 5; the pools' 5-D maps follow their 3-D maps), or one CUDA-core
// launch per row tile (counters 0-3).
cudaError_t launch_cc_group(const pst_plan* p, const DevPlan& dp, const void* tk, const void* tv, const void* Q,
                            LaunchSeq& ls) {
    if (p->thin) {
        for (int k = 0; k < 2; ++k) {
            if (p->cc_class_cnt[k] == 0) continue;
            cudaError_t e = launch_pac_thin(dp, static_cast<const unsigned char*>(tk) + 128,
                                            static_cast<const unsigned char*>(tv) + 128, Q, k == 0 ? 8 : 4,
                                            (int)p->cc_class_cnt[k], (int)p->cc_class_off[k], 4 + k, ls.st,
                                            ls.next_pdl());
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    for (int k = 0; k < 4; ++k) {
        if (p->cc_class_cnt[k] == 0) continue;
        cudaError_t e = launch_pac_cc(dp, p->dtype, tk, tv, Q, 8 >> k, (int)p->cc_class_cnt[k],
                                      (int)p->cc_class_off[k], k, ls.st, ls.next_pdl());
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

namespace dev {

constexpr int kPorWarps = 8;

template <int D>
__global__ void __launch_bounds__(kPorWarps * 32) por_kernel(DevPlan P, float* __restrict__ O, float* __restrict__ LSE) {
    constexpr int EPL = D / 32;
    pdl_wait();   // launched early behind the PAC grids: wait for all of them
    // every PAC launch of this call has finished: rearm their work queues
    if (blockIdx.x == 0 && threadIdx.x < kNumCounters) P.counters[threadIdx.x] = 0;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t w = (int64_t)blockIdx.x * kPorWarps + warp;
    const int Hq = P.n_q_heads;
    if (w >= (int64_t)P.n_queries * Hq) return;
    const int q = (int)(w / Hq), h = (int)(w % Hq);
    const int e0 = P.merge_ptr[q], e1 = P.merge_ptr[q + 1];
    // One pass over the query's partials, 32 at a time: lane i holds entry
    // i's row and log-sum-exp; the running max M rescales what was summed.
    float M = -INFINITY, W = 0.f;
    float acc[EPL];
#pragma unroll
    for (int k = 0; k < EPL; ++k) acc[k] = 0.f;
    for (int b = e0; b < e1; b += 32) {
        const int cnt = min(32, e1 - b);
        int64_t my_row = 0;
        float my_lse = -INFINITY;
        if (lane < cnt) {
            my_row = (int64_t)P.merge_row[b + lane] + h;
            my_lse = P.part_lse[my_row];
        }
        float m = my_lse;
#pragma unroll
        for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        const float M2 = fmaxf(M, m);
        const float Mu = M2 == -INFINITY ? 0.f : M2;
        const float a = fast_exp2(M - Mu);   // rescales the earlier sum (0 when empty)
        const float my_w = lane < cnt ? fast_exp2(my_lse - Mu) : 0.f;
        float ws = my_w;
#pragma unroll
        for (int off = 16; off; off >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, off);
        W = W * a + ws;
#pragma unroll
        for (int k = 0; k < EPL; ++k) acc[k] *= a;
        M = M2;
        // eight partial rows in flight at a time
        for (int i = 0; i < cnt; i += 8) {
            float v[8][EPL];
            float wt[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int src_lane = min(i + u, cnt - 1);
                const int64_t row = __shfl_sync(0xffffffffu, my_row, src_lane);
                wt[u] = i + u < cnt ? __shfl_sync(0xffffffffu, my_w, src_lane) : 0.f;
                const float* src = P.part_o + row * D + lane * EPL;
                if constexpr (EPL == 4) {
                    const float4 x = *reinterpret_cast<const float4*>(src);
                    v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2*>(src);
                    v[u][0] = x.x; v[u][1] = x.y;
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
#pragma unroll
                for (int k = 0; k < EPL; ++k) acc[k] = fmaf(wt[u], v[u][k], acc[k]);
        }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    float* dst = O + w * D + lane * EPL;
    if constexpr (EPL == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    } else {
        *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0) LSE[w] = (M + __log2f(W)) * 0.69314718055994530942f;
}

}  // namespace dev

int device_sm_count(int* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return 0;
}

static int cuda_fail(const char* what, cudaError_t e) {
    return fail(PST_ECUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// TMA descriptors over a pool [num_pages][Hkv][page_size][d], 128B swizzle:
// out[0, 128): 3-D (d, page row, page*Hkv + head), boxes of one 128-byte slab
// x 16 rows; bf16 with d = 128 also gets two 5-D views (64 channels, page row,
// head, slab, page) with the slab stride 128 bytes: out[128, 256) for thin
// plans, boxes of 16 rows x 8 heads x 2 slabs landing as [slab][head][row];
// out[256, 384), boxes of 16 rows x 2 slabs of one head ([slab][row], 4 KB).
static int make_pool_map(const pst_plan* p, const void* pool, unsigned char* out) {
    auto fn = encode_fn();
    if (!fn) return fail(PST_ECUDA, "decode_attn: cuTensorMapEncodeTiled is unavailable");
    const int eb = p->dtype == PST_BF16 ? 2 : 4;
    cuuint64_t dims[3] = {(cuuint64_t)p->d, (cuuint64_t)p->page_size, (cuuint64_t)p->num_pages * p->hkv};
    cuuint64_t strides[2] = {(cuuint64_t)p->d * eb, (cuuint64_t)p->page_size * p->d * eb};
    cuuint32_t box[3] = {(cuuint32_t)(128 / eb), (cuuint32_t)kBoxRows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(reinterpret_cast<CUtensorMap*>(out),
                    p->dtype == PST_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                    const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PST_ECUDA, "decode_attn: cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    if (p->dtype == PST_BF16 && p->d == 128) {
        cuuint64_t d5[5] = {64, (cuuint64_t)p->page_size, (cuuint64_t)p->hkv, 2, (cuuint64_t)p->num_pages};
        cuuint64_t s5[4] = {(cuuint64_t)p->d * eb, (cuuint64_t)p->page_size * p->d * eb, 128,
                            (cuuint64_t)p->hkv * p->page_size * p->d * eb};
        cuuint32_t e5[5] = {1, 1, 1, 1, 1};
        for (int v = 0; v < 2; ++v) {
            if (v == 0 && !p->thin) continue;
            cuuint32_t b5[5] = {64, (cuuint32_t)kBoxRows, v == 0 ? (cuuint32_t)kThinHeads : 1u, 2, 1};
            r = fn(reinterpret_cast<CUtensorMap*>(out + 128 * (v + 1)), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                   const_cast<void*>(pool), d5, s5, b5, e5, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS)
                return fail(PST_ECUDA, "decode_attn: cuTensorMapEncodeTiled (5-D) failed (" + std::to_string((int)r) + ")");
        }
    }
    return PST_OK;
}

// For entry points that run a plan out of device memory other than its bound
// workspace (same layout, base `ws`).
int encode_pool_map(const pst_plan* p, const void* pool, unsigned char* out) { return make_pool_map(p, pool, out); }

int encode_bf16_map(void* out, int rank, const void* base, const uint64_t* dims, const uint64_t* strides,
                    const uint32_t* box);

// Q [B][Hq][d] as (channel, q-head, query) with boxes of 64 channels x G
// heads x 128/G queries: the 128 rows of one tcgen05-PAC row half (query-major,
// then the G heads of one kv head), 128-byte swizzle. Used for bf16 with G up
// to 16 and dividing 128: measured on GB300, the TMA copy made document QA
// (G = 4) 1.6 % and few-shot 6 % faster per step, but tree-of-thought MQA
// (G = 32) 2 % slower than staging Q row by row.
bool q_map_fits(const pst_plan* p) { return p->dtype == PST_BF16 && p->group <= 16 && 128 % p->group == 0; }

int encode_q_map(const pst_plan* p, const void* Q, unsigned char* out) {
    const uint64_t dims[3] = {(uint64_t)p->d, (uint64_t)p->hq, (uint64_t)p->n_queries};
    const uint64_t str[2] = {(uint64_t)p->d * 2, (uint64_t)p->hq * p->d * 2};
    const uint32_t box[3] = {64, (uint32_t)p->group, (uint32_t)(128 / p->group)};
    return encode_bf16_map(out, 3, Q, dims, str, box);
}

// A bf16 tensor map with 128-byte swizzle for the library's other launchers:
// `rank` dims (innermost first), strides in bytes of dims 1.., box extents.
int encode_bf16_map(void* out, int rank, const void* base, const uint64_t* dims, const uint64_t* strides,
                    const uint32_t* box) {
    auto fn = encode_fn();
    if (!fn) return fail(PST_ECUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    CUresult r = fn(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base),
                    d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PST_ECUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
    return PST_OK;
}

DevPlan dev_plan_at(const pst_plan* p, void* ws) {
    uint8_t* b = static_cast<uint8_t*>(ws);
    DevPlan d;
    d.items = reinterpret_cast<const DevItem*>(b + p->ws.items);
    d.chunks = reinterpret_cast<const DevChunk*>(b + p->ws.chunks);
    d.pages = reinterpret_cast<const int32_t*>(b + p->ws.pages);
    d.chunk_q = reinterpret_cast<const int32_t*>(b + p->ws.chunk_q);
    d.masks = reinterpret_cast<const uint64_t*>(b + p->ws.masks);
    d.merge_ptr = reinterpret_cast<const int32_t*>(b + p->ws.merge_ptr);
    d.merge_row = reinterpret_cast<const int32_t*>(b + p->ws.merge_row);
    d.part_o = reinterpret_cast<float*>(b + p->ws.part_o);
    d.part_lse = reinterpret_cast<float*>(b + p->ws.part_lse);
    d.status = reinterpret_cast<int32_t*>(b + p->ws.status);
    d.counters = d.status + 4;
    d.n_queries = p->n_queries;
    d.n_q_heads = p->hq;
    d.n_kv_heads = p->hkv;
    d.group = p->group;
    d.d = p->d;
    d.page_size = p->page_size;
    d.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p->d));
    d.debug_stall = p->opts.debug_stall;
    return d;
}

static DevPlan dev_plan(const pst_plan* p) { return dev_plan_at(p, p->d_ws); }

cudaError_t launch_por(const DevPlan& dp, float* O, float* LSE, LaunchSeq& ls) {
    const int64_t warps = (int64_t)dp.n_queries * dp.n_q_heads;
    const int blocks = (int)((warps + dev::kPorWarps - 1) / dev::kPorWarps);
    const bool pdl = ls.next_pdl();
    if (dp.d == 128)
        return launch_kernel(dev::por_kernel<128>, dim3(blocks), dim3(dev::kPorWarps * 32), 0, ls.st, pdl, dp, O, LSE);
    return launch_kernel(dev::por_kernel<64>, dim3(blocks), dim3(dev::kPorWarps * 32), 0, ls.st, pdl, dp, O, LSE);
}

}  // namespace pst

// Per recorded call, events: [0] start, [1..5] end of each PAC launch group
// (tensor core P once / two row-block modes, exact P / two modes, CUDA core;
// each on the stream that ran it), [6] POR start (after the join), [7] POR
// end. The PAC slots report time from the call's start to the end of their
// groups (the groups run side by side); the POR slot reports POR alone.
struct pst_timer {
    int32_t max_calls = 0;
    int32_t calls = 0;
    std::vector<cudaEvent_t> ev;         // max_calls x kEvents
    std::vector<uint8_t> ran;            // max_calls x 5: launch group g had work in call c
    static constexpr int kEvents = 8;
};

using namespace pst;

extern "C" int pst_plan_upload(pst_plan* p, void* d_ws, int64_t bytes, void* stream) {
    if (!p) return fail(PST_EINVAL, "plan_upload: plan is null");
    if (!d_ws) return fail(PST_EWORKSPACE, "plan_upload: workspace is null");
    if (reinterpret_cast<uintptr_t>(d_ws) % 256) return fail(PST_EWORKSPACE, "plan_upload: workspace must be 256-byte aligned");
    if (bytes < p->ws.total) return fail(PST_EWORKSPACE, "plan_upload: workspace too small (need " + std::to_string(p->ws.total) + " bytes)");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(d_ws, p->meta_blob.data(), p->meta_blob.size(), cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail("plan_upload: cudaMemcpyAsync", e);
    // the host image stays alive with the plan; make the copy complete before returning so the
    // caller may free nothing early
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail("plan_upload: cudaStreamSynchronize", e);
    p->d_ws = d_ws;
    p->tmap_k_ptr = p->tmap_v_ptr = nullptr;
    return PST_OK;
}

static int decode_impl(const pst_plan* p, const void* Q, const void* K, const void* V, float* O, float* LSE,
                       void* stream, pst_timer* timer) {
    if (!p) return fail(PST_EINVAL, "decode_attn: plan is null");
    if (!p->d_ws) return fail(PST_EWORKSPACE, "decode_attn: plan has no uploaded workspace");
    if (!Q || !K || !V || !O || !LSE) return fail(PST_EINVAL, "decode_attn: null tensor pointer");
    if ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(Q) |
         reinterpret_cast<uintptr_t>(O)) % 16)
        return fail(PST_EINVAL, "decode_attn: Q, K_pool, V_pool and O must be 16-byte aligned");
    if (p->tmap_k_ptr != K) {
        int rc = make_pool_map(p, K, p->tmap_k);
        if (rc) return rc;
        p->tmap_k_ptr = K;
    }
    if (p->tmap_v_ptr != V) {
        int rc = make_pool_map(p, V, p->tmap_v);
        if (rc) return rc;
        p->tmap_v_ptr = V;
    }
    const bool q_map = q_map_fits(p);
    if (q_map && p->tmap_q_ptr != Q) {
        int rc = encode_q_map(p, Q, p->tmap_q);
        if (rc) return rc;
        p->tmap_q_ptr = Q;
    }
    const void* tq = q_map ? static_cast<const void*>(p->tmap_q) : nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const DevPlan dp = dev_plan(p);
    cudaEvent_t* ev = nullptr;
    if (timer) {
        if (timer->calls >= timer->max_calls) return fail(PST_EINVAL, "decode_attn_timed: timer is full");
        ev = timer->ev.data() + (size_t)timer->calls * pst_timer::kEvents;
        cudaEventRecord(ev[0], st);
    }
    cudaError_t e;
    // The PAC launch groups (four tensor-core ones, the thin one) write
    // disjoint partial rows, so they may run side by side; POR merges after
    // all of them. Two ways to let them share the SMs:
    //  - one stream, every launch after the first with a programmatic
    //    dependency on the one before (the default): a group's blocks start
    //    once every block of the groups launched before it has started, so the
    //    SMs fill in launch order (tensor-core groups first), which is the
    //    order the planner's list schedule assumes, and no event crosses
    //    streams; POR waits for all of them on the device;
    //  - the first non-empty group on `st`, the others on side streams forked
    //    from it and joined before POR (also the timed path: its events
    //    between launches would break a chain).
    constexpr int kGroups = 5;
    bool has[kGroups];
    for (int g = 0; g < 4; ++g) has[g] = p->tc_group_cnt[g] > 0;
    has[4] = p->n_cc_items > 0;
    const bool chain = p->opts.side_streams == 0 && !ev;
    if (chain) {
        LaunchSeq ls(st, true);
        for (int g = 0; g < kGroups; ++g) {
            if (!has[g]) continue;
            e = g < 4 ? launch_tc_group(p, dp, p->tmap_k, p->tmap_v, tq, Q, g, ls)
                      : launch_cc_group(p, dp, p->tmap_k, p->tmap_v, Q, ls);
            if (e != cudaSuccess) return cuda_fail(g < 4 ? "decode_attn: PAC (tensor core) launch"
                                                         : "decode_attn: PAC (thin chunks) launch", e);
        }
        e = launch_por(dp, O, LSE, ls);
        if (e != cudaSuccess) return cuda_fail("decode_attn: POR launch", e);
        return PST_OK;
    }
    cudaStream_t gst[kGroups] = {st, st, st, st, st};
    int n_side = 0;
    bool first = true;
    for (int g = 0; g < kGroups; ++g) {
        if (!has[g]) continue;
        if (first) { first = false; continue; }
        if (!p->side_stream[n_side]) {
            cudaStream_t s2;
            cudaEvent_t j;
            if ((e = cudaStreamCreateWithFlags(&s2, cudaStreamNonBlocking)) != cudaSuccess)
                return cuda_fail("decode_attn: side stream", e);
            if ((e = cudaEventCreateWithFlags(&j, cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail("decode_attn: join event", e);
            p->side_stream[n_side] = s2;
            p->ev_join[n_side] = j;
        }
        if (!p->ev_fork) {
            cudaEvent_t f;
            if ((e = cudaEventCreateWithFlags(&f, cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail("decode_attn: fork event", e);
            p->ev_fork = f;
        }
        gst[g] = static_cast<cudaStream_t>(p->side_stream[n_side++]);
    }
    if (n_side > 0) {
        cudaEventRecord(static_cast<cudaEvent_t>(p->ev_fork), st);
        for (int k = 0; k < n_side; ++k)
            cudaStreamWaitEvent(static_cast<cudaStream_t>(p->side_stream[k]), static_cast<cudaEvent_t>(p->ev_fork), 0);
    }
    for (int g = 0; g < kGroups; ++g) {
        if (!has[g]) continue;
        LaunchSeq ls(gst[g], false);
        e = g < 4 ? launch_tc_group(p, dp, p->tmap_k, p->tmap_v, tq, Q, g, ls)
                  : launch_cc_group(p, dp, p->tmap_k, p->tmap_v, Q, ls);
        if (e != cudaSuccess) return cuda_fail(g < 4 ? "decode_attn: PAC (tensor core) launch"
                                                     : "decode_attn: PAC (thin chunks) launch", e);
        if (ev) cudaEventRecord(ev[1 + g], gst[g]);
    }
    if (ev)
        for (int g = 0; g < kGroups; ++g) timer->ran[(size_t)timer->calls * kGroups + g] = has[g] ? 1 : 0;
    for (int k = 0; k < n_side; ++k) {
        cudaEventRecord(static_cast<cudaEvent_t>(p->ev_join[k]), static_cast<cudaStream_t>(p->side_stream[k]));
        cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(p->ev_join[k]), 0);
    }
    if (ev) cudaEventRecord(ev[6], st);
    LaunchSeq lpor(st, false);
    e = launch_por(dp, O, LSE, lpor);
    if (e != cudaSuccess) return cuda_fail("decode_attn: POR launch", e);
    if (ev) {
        cudaEventRecord(ev[7], st);
        timer->calls++;
    }
    return PST_OK;
}

namespace pst {
void release_plan_streams(pst_plan* p) {
    for (int k = 0; k < 4; ++k) {
        if (p->side_stream[k]) cudaStreamDestroy(static_cast<cudaStream_t>(p->side_stream[k]));
        if (p->ev_join[k]) cudaEventDestroy(static_cast<cudaEvent_t>(p->ev_join[k]));
        p->side_stream[k] = p->ev_join[k] = nullptr;
    }
    if (p->ev_fork) cudaEventDestroy(static_cast<cudaEvent_t>(p->ev_fork));
    p->ev_fork = nullptr;
}
}  // namespace pst

extern "C" int pst_decode_attn(const pst_plan* p, const void* Q, const void* K, const void* V, float* O, float* LSE,
                               void* stream) {
    return decode_impl(p, Q, K, V, O, LSE, stream, nullptr);
}

extern "C" int pst_decode_attn_timed(const pst_plan* p, const void* Q, const void* K, const void* V, float* O,
                                     float* LSE, void* stream, pst_timer* timer) {
    if (!timer) return fail(PST_EINVAL, "decode_attn_timed: timer is null");
    return decode_impl(p, Q, K, V, O, LSE, stream, timer);
}

extern "C" int pst_plan_check_status(const pst_plan* p, void* stream, int32_t* code) {
    if (!p || !p->d_ws) return fail(PST_EWORKSPACE, "check_status: plan has no workspace");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t word = 0;
    int32_t* dstatus = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(p->d_ws) + p->ws.status);
    cudaError_t e = cudaMemcpyAsync(&word, dstatus, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dstatus, 0, 4, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail("check_status", e);
    if (code) *code = word;
    if (word) return fail(PST_EDEVICE, "check_status: device status word " + std::to_string(word));
    return PST_OK;
}

extern "C" int pst_timer_create(int32_t max_calls, pst_timer** out) {
    if (!out || max_calls <= 0) return fail(PST_EINVAL, "timer_create: bad argument");
    pst_timer* t = new (std::nothrow) pst_timer();
    if (!t) return fail(PST_ENOMEM, "timer_create: out of memory");
    t->max_calls = max_calls;
    t->ev.resize((size_t)max_calls * pst_timer::kEvents, nullptr);
    t->ran.assign((size_t)max_calls * 5, 0);
    for (auto& e : t->ev) {
        cudaError_t r = cudaEventCreate(&e);
        if (r != cudaSuccess) {
            for (auto& x : t->ev) if (x) cudaEventDestroy(x);
            delete t;
            return cuda_fail("timer_create: cudaEventCreate", r);
        }
    }
    *out = t;
    return PST_OK;
}

extern "C" void pst_timer_destroy(pst_timer* t) {
    if (!t) return;
    for (auto& e : t->ev) if (e) cudaEventDestroy(e);
    delete t;
}

extern "C" int pst_timer_read(pst_timer* t, float* ms, int32_t n, int32_t* calls) {
    if (!t) return fail(PST_EINVAL, "timer_read: timer is null");
    for (int k = 0; k < n; ++k) ms[k] = 0.f;
    const int stride = pst_timer::kEvents;
    if (t->calls > 0) {
        cudaError_t e = cudaEventSynchronize(t->ev[(size_t)(t->calls - 1) * stride + stride - 1]);
        if (e != cudaSuccess) return cuda_fail("timer_read: cudaEventSynchronize", e);
    }
    // slot k covers launch groups grp[k][0..1] (end events 1 + g); a slot
    // whose groups had no work in a call adds 0 for that call
    static const int grp[3][2] = {{0, 1}, {2, 3}, {4, 4}};
    for (int c = 0; c < t->calls; ++c) {
        const cudaEvent_t* e0 = t->ev.data() + (size_t)c * stride;
        const uint8_t* ran = t->ran.data() + (size_t)c * 5;
        for (int k = 0; k < 4 && k < n; ++k) {
            float x = 0.f;
            cudaError_t e = cudaSuccess;
            if (k == 3) {
                e = cudaEventElapsedTime(&x, e0[6], e0[7]);
            } else {
                for (int g : grp[k]) {
                    if (!ran[g]) continue;
                    float y = 0.f;
                    e = cudaEventElapsedTime(&y, e0[0], e0[1 + g]);
                    if (e != cudaSuccess) break;
                    x = std::max(x, y);
                }
            }
            if (e != cudaSuccess) return cuda_fail("timer_read: cudaEventElapsedTime", e);
            ms[k] += x;
        }
    }
    if (calls) *calls = t->calls;
    t->calls = 0;
    return PST_OK;
}

extern "C" const char* pst_timer_kernel_name(int32_t slot) {
    switch (slot) {
        case 0: return "pac_tc";
        case 1: return "pac_tc_exact";
        case 2: return "pac_thin";
        case 3: return "por";
        default: return "";
    }
}
