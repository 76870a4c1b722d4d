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

#include <chrono>
#include <cmath>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "dev_common.cuh"

namespace pst {

cudaError_t launch_pac_cc(const DevPlan& P, pst_dtype dt, const void* tk, const void* tv, const void* Q,
                          int r_tile, int n_items, int item_off, cudaStream_t st);
cudaError_t launch_pac_tc(const DevPlan& P, const void* tk, const void* tv, const void* Q, int n_items,
                          int item_off, cudaStream_t st);
cudaError_t launch_pac_umma(const DevPlan& P, const void* tk, const void* tv, const void* Q, int n_items,
                            int item_off, cudaStream_t st);

namespace dev {

constexpr int kPorWarps = 8;

template <int D>
__global__ void __launch_bounds__(kPorWarps * 32) por_kernel(DevPlan P, float* __restrict__ O, float* __restrict__ LSE) {
    constexpr int EPL = D / 32;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t w = (int64_t)blockIdx.x * kPorWarps + warp;
    const int Hq = P.n_q_heads;
    if (w >= (int64_t)P.n_queries * Hq) return;
    const int q = (int)(w / Hq), h = (int)(w % Hq);
    const int e0 = P.merge_ptr[q], e1 = P.merge_ptr[q + 1];
    // the query's partials, 32 at a time: lane i holds entry i's row and weight
    float M = -INFINITY;
    for (int e = e0 + lane; e < e1; e += 32) M = fmaxf(M, P.part_lse[P.merge_row[e] + h]);
#pragma unroll
    for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float Mu = M == -INFINITY ? 0.f : M;
    float acc[EPL];
#pragma unroll
    for (int k = 0; k < EPL; ++k) acc[k] = 0.f;
    float W = 0.f;
    for (int b = e0; b < e1; b += 32) {
        const int cnt = min(32, e1 - b);
        int64_t my_row = 0;
        float my_w = 0.f;
        if (lane < cnt) {
            my_row = (int64_t)P.merge_row[b + lane] + h;
            my_w = fast_exp2(P.part_lse[my_row] - Mu);
        }
        float ws = my_w;
#pragma unroll
        for (int off = 16; off; off >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, off);
        W += ws;
        // four partial rows in flight at a time
        for (int i = 0; i < cnt; i += 4) {
            float v[4][EPL];
            float wt[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
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
            for (int u = 0; u < 4; ++u)
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

// TMA descriptor over a pool [num_pages][Hkv][page_size][d] viewed as 3-D
// (d, page row, page*Hkv + head); boxes of one 128-byte slab x 16 rows with the
// 128B swizzle.
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
    return PST_OK;
}

static DevPlan dev_plan(const pst_plan* p) {
    uint8_t* b = static_cast<uint8_t*>(p->d_ws);
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
    d.n_queries = p->n_queries;
    d.n_q_heads = p->hq;
    d.n_kv_heads = p->hkv;
    d.group = p->group;
    d.d = p->d;
    d.page_size = p->page_size;
    d.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p->d));
    return d;
}

// For entry points that run a plan out of device memory other than its bound
// workspace (same layout, base `ws`).
int encode_pool_map(const pst_plan* p, const void* pool, unsigned char* out) { return make_pool_map(p, pool, out); }

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
    d.n_queries = p->n_queries;
    d.n_q_heads = p->hq;
    d.n_kv_heads = p->hkv;
    d.group = p->group;
    d.d = p->d;
    d.page_size = p->page_size;
    d.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)p->d));
    return d;
}

cudaError_t launch_por(const DevPlan& dp, float* O, float* LSE, cudaStream_t st) {
    const int64_t warps = (int64_t)dp.n_queries * dp.n_q_heads;
    const int blocks = (int)((warps + dev::kPorWarps - 1) / dev::kPorWarps);
    if (dp.d == 128) dev::por_kernel<128><<<blocks, dev::kPorWarps * 32, 0, st>>>(dp, O, LSE);
    else dev::por_kernel<64><<<blocks, dev::kPorWarps * 32, 0, st>>>(dp, O, LSE);
    return cudaGetLastError();
}

}  // namespace pst

struct pst_timer {
    int32_t max_calls = 0;
    int32_t calls = 0;
    int32_t n_slots = 0;                 // kernels per call in the recorded calls
    int32_t forked = 0;                  // the CUDA-core PAC ran beside the tensor-core PAC
    std::vector<cudaEvent_t> ev;         // max_calls x (1 + kMaxKernels)
    static constexpr int kMaxKernels = 4;
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
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const DevPlan dp = dev_plan(p);
    cudaEvent_t* ev = nullptr;
    if (timer) {
        if (timer->calls >= timer->max_calls) return fail(PST_EINVAL, "decode_attn_timed: timer is full");
        ev = timer->ev.data() + (size_t)timer->calls * (1 + pst_timer::kMaxKernels);
        cudaEventRecord(ev[0], st);
    }
    cudaError_t e;
    // Both PAC kernels write disjoint partial rows; when a plan has both
    // kinds, the CUDA-core PAC runs on a side stream forked from `st` so its
    // blocks fill the SMs the tensor-core blocks leave idle, and POR waits on
    // the join. Timer events: [0] start, [1] after the tensor-core PAC (st),
    // [2] after the CUDA-core PAC (its stream), [3] after POR (st).
    const bool fork = p->n_tc_items > 0 && p->n_cc_items > 0;
    cudaStream_t cc_st = st;
    if (fork) {
        if (!p->side_stream) {
            cudaStream_t s2;
            cudaEvent_t a, b;
            if ((e = cudaStreamCreateWithFlags(&s2, cudaStreamNonBlocking)) != cudaSuccess)
                return cuda_fail("decode_attn: side stream", e);
            if ((e = cudaEventCreateWithFlags(&a, cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&b, cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail("decode_attn: fork/join events", e);
            p->side_stream = s2;
            p->ev_fork = a;
            p->ev_join = b;
        }
        cc_st = static_cast<cudaStream_t>(p->side_stream);
        cudaEventRecord(static_cast<cudaEvent_t>(p->ev_fork), st);
        cudaStreamWaitEvent(cc_st, static_cast<cudaEvent_t>(p->ev_fork), 0);
    }
    if (p->n_tc_items > 0) {
        e = p->opts.tc_engine == 1 ? launch_pac_tc(dp, p->tmap_k, p->tmap_v, Q, (int)p->n_tc_items, 0, st)
                                   : launch_pac_umma(dp, p->tmap_k, p->tmap_v, Q, (int)p->n_tc_items, 0, st);
        if (e != cudaSuccess) return cuda_fail("decode_attn: PAC (tensor core) launch", e);
    }
    if (ev) cudaEventRecord(ev[1], st);
    for (int k = 0; k < 4; ++k) {
        if (p->cc_class_cnt[k] == 0) continue;
        e = launch_pac_cc(dp, p->dtype, p->tmap_k, p->tmap_v, Q, 8 >> k, (int)p->cc_class_cnt[k],
                          (int)p->cc_class_off[k], cc_st);
        if (e != cudaSuccess) return cuda_fail("decode_attn: PAC (CUDA core) launch", e);
    }
    if (ev) cudaEventRecord(ev[2], cc_st);
    if (fork) {
        cudaEventRecord(static_cast<cudaEvent_t>(p->ev_join), cc_st);
        cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(p->ev_join), 0);
    }
    int slot = 2;
    {
        const int64_t warps = (int64_t)p->n_queries * p->hq;
        const int blocks = (int)((warps + dev::kPorWarps - 1) / dev::kPorWarps);
        if (p->d == 128) dev::por_kernel<128><<<blocks, dev::kPorWarps * 32, 0, st>>>(dp, O, LSE);
        else dev::por_kernel<64><<<blocks, dev::kPorWarps * 32, 0, st>>>(dp, O, LSE);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail("decode_attn: POR launch", e);
    }
    if (ev) {
        cudaEventRecord(ev[++slot], st);
        timer->n_slots = slot;
        timer->forked = fork ? 1 : 0;
        timer->calls++;
    }
    return PST_OK;
}

namespace pst {
void release_plan_streams(pst_plan* p) {
    if (p->side_stream) cudaStreamDestroy(static_cast<cudaStream_t>(p->side_stream));
    if (p->ev_fork) cudaEventDestroy(static_cast<cudaEvent_t>(p->ev_fork));
    if (p->ev_join) cudaEventDestroy(static_cast<cudaEvent_t>(p->ev_join));
    p->side_stream = p->ev_fork = p->ev_join = nullptr;
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
    t->ev.resize((size_t)max_calls * (1 + pst_timer::kMaxKernels), nullptr);
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
    const int stride = 1 + pst_timer::kMaxKernels;
    if (t->calls > 0) {
        cudaError_t e = cudaEventSynchronize(t->ev[(size_t)(t->calls - 1) * stride + t->n_slots]);
        if (e != cudaSuccess) return cuda_fail("timer_read: cudaEventSynchronize", e);
    }
    for (int c = 0; c < t->calls; ++c) {
        for (int k = 0; k < t->n_slots && k < n; ++k) {
            float x = 0.f;
            // a forked CUDA-core PAC starts with the call, not after the tensor-core PAC
            const int from = (k == 1 && t->forked) ? 0 : k;
            cudaError_t e = cudaEventElapsedTime(&x, t->ev[(size_t)c * stride + from], t->ev[(size_t)c * stride + k + 1]);
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
        case 1: return "pac_cc";
        case 2: return "por";
        default: return "";
    }
}
