// pst_decode_attn_noalloc: tree decode attention with no device allocation
// anywhere -- neither here nor by the caller.
//
// pst_decode_attn needs a device workspace that the caller allocates once per
// plan (the plan's metadata and the partial outputs the PAC kernels hand to
// the POR merge). Some callers cannot allocate device memory at the point
// where they run attention: a plug-in inside an inference engine whose
// framework owns and pre-plans every device byte, code that must not trigger
// the device-wide synchronisation that cudaFree implies, or a process where a
// caching allocator is not available. This entry point serves them: its
// scratch lives in one fixed-size array in the library's own device memory,
// reserved when the library is loaded on a device and held until the process
// exits. The caller passes only inputs and outputs.
#include <mutex>
#include <string>

#include "dev_common.cuh"

namespace pst {

cudaError_t launch_tc_group(const pst_plan* p, const DevPlan& dp, const void* tk, const void* tv, const void* tq,
                            const void* Q, int g, LaunchSeq& ls);
bool q_map_fits(const pst_plan* p);
int encode_q_map(const pst_plan* p, const void* Q, unsigned char* out);
cudaError_t launch_cc_group(const pst_plan* p, const DevPlan& dp, const void* tk, const void* tv, const void* Q,
                            LaunchSeq& ls);
cudaError_t launch_por(const DevPlan& dp, float* O, float* LSE, LaunchSeq& ls);
int encode_pool_map(const pst_plan* p, const void* pool, unsigned char* out);
DevPlan dev_plan_at(const pst_plan* p, void* ws);

// The scratch: a plan's metadata image followed by its partial outputs.
constexpr int64_t kStaticWorkspaceBytes = PST_NOALLOC_WORKSPACE_BYTES;
static __device__ __align__(256) unsigned char g_static_ws[kStaticWorkspaceBytes];

namespace {
constexpr int kMaxDevices = 256;
std::mutex g_mu;
void* g_ws_addr[kMaxDevices] = {};  // device address of g_static_ws, per device ordinal
}  // namespace

// Host code cannot pass g_static_ws to a kernel: on the host that name is only
// a stand-in for the device array. The device address is looked up once per
// device, with that device current, and cached.
static int static_ws_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(PST_ECUDA, std::string("decode_attn_noalloc: cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(PST_EUNSUPPORTED, "decode_attn_noalloc: device ordinal too large");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ws_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess || !p)
            return fail(PST_ECUDA, std::string("decode_attn_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
        g_ws_addr[dev] = p;
    }
    *out = g_ws_addr[dev];
    return PST_OK;
}

}  // namespace pst

using namespace pst;

extern "C" int pst_decode_attn_noalloc(const pst_plan* p, const void* Q, const void* K, const void* V, float* O,
                                       float* LSE, void* stream) {
    if (!p) return fail(PST_EINVAL, "decode_attn_noalloc: plan is null");
    if (!Q || !K || !V || !O || !LSE) return fail(PST_EINVAL, "decode_attn_noalloc: null tensor pointer");
    if ((reinterpret_cast<uintptr_t>(K) | reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(Q) |
         reinterpret_cast<uintptr_t>(O)) % 16)
        return fail(PST_EINVAL, "decode_attn_noalloc: Q, K_pool, V_pool and O must be 16-byte aligned");
    if (p->ws.total > kStaticWorkspaceBytes)
        return fail(PST_EWORKSPACE, "decode_attn_noalloc: this plan needs " + std::to_string(p->ws.total) +
                                        " bytes of scratch; the built-in scratch holds " +
                                        std::to_string(kStaticWorkspaceBytes) +
                                        " (use pst_decode_attn with a caller-allocated workspace)");
    void* ws = nullptr;
    int rc = static_ws_address(&ws);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The array keeps whatever the previous call left. The plan's metadata
    // image is written afresh each call; it also zeroes the status word. The
    // partial outputs need no clearing: every row is written before POR reads it.
    cudaError_t e = cudaMemcpyAsync(ws, p->meta_blob.data(), p->meta_blob.size(), cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess)
        return fail(PST_ECUDA, std::string("decode_attn_noalloc: metadata copy: ") + cudaGetErrorString(e));
    alignas(64) unsigned char tk[384], tv[384];
    rc = encode_pool_map(p, K, tk);
    if (rc) return rc;
    rc = encode_pool_map(p, V, tv);
    if (rc) return rc;
    alignas(64) unsigned char tq[128];
    const bool q_map = q_map_fits(p);
    if (q_map && (rc = encode_q_map(p, Q, tq)) != 0) return rc;
    const DevPlan dp = dev_plan_at(p, ws);
    // the launch groups on `stream`: chained by programmatic dependencies
    // (the default), else one after the other
    LaunchSeq ls(st, p->opts.side_streams == 0);
    for (int g = 0; g < 5; ++g) {
        e = g < 4 ? launch_tc_group(p, dp, tk, tv, q_map ? tq : nullptr, Q, g, ls)
                  : launch_cc_group(p, dp, tk, tv, Q, ls);
        if (e != cudaSuccess) return fail(PST_ECUDA, std::string("decode_attn_noalloc: PAC launch: ") + cudaGetErrorString(e));
    }
    e = launch_por(dp, O, LSE, ls);
    if (e != cudaSuccess) return fail(PST_ECUDA, std::string("decode_attn_noalloc: POR launch: ") + cudaGetErrorString(e));
    return PST_OK;
}

extern "C" int pst_noalloc_check_status(void* stream, int32_t* code) {
    void* ws = nullptr;
    int rc = static_ws_address(&ws);
    if (rc) return rc;
    // every plan's metadata image starts with the status word (offset 0)
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, ws, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, 4, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail(PST_ECUDA, std::string("noalloc_check_status: ") + cudaGetErrorString(e));
    if (code) *code = word;
    if (word) return fail(PST_EDEVICE, "noalloc_check_status: device status word " + std::to_string(word));
    return PST_OK;
}
