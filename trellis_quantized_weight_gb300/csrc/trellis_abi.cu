// The C ABI (include/trellis.h): argument validation on the host, then one
// kernel launch on the caller's stream.  No host synchronisation, no CPU
// fallback.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kernels.h"
#include "trellis.h"

namespace {

using trellis::DeviceInfo;

constexpr int kMaxDevices = 64;

int device_info(DeviceInfo& out) {
    static std::mutex mu;
    static DeviceInfo cache[kMaxDevices];
    static bool have[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TRELLIS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DeviceInfo d;
        d.device = dev;
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return TRELLIS_ERR_CUDA;
        cache[dev] = d;
        have[dev] = true;
    }
    out = cache[dev];
    return TRELLIS_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Checks shared by every entry point: T = 256, 1 <= k <= 8, k < L <= 24 (the
// page's wrapper accepts k in {2,3,4} with L = 12; the same definition holds
// for the wider set, whose windows still span at most two words); K a
// multiple of T; no fixed K or N.
int check_geometry(int K, int N, int k, int L, int T) {
    if (k < trellis::kMinK || k > trellis::kMaxK) return TRELLIS_ERR_UNSUPPORTED;
    if (L <= k || L > trellis::kMaxL || T != trellis::kT_abi) return TRELLIS_ERR_UNSUPPORTED;
    if (K <= 0 || N <= 0 || K % T != 0) return TRELLIS_ERR_SHAPE;
    // item (row, block) indices and weight offsets must fit the kernels' integer types
    const long long items = static_cast<long long>(N) * (K / T);
    if (items >= (1ll << 31)) return TRELLIS_ERR_SHAPE;
    return TRELLIS_OK;
}

// 1 <= M <= 16 runs on the CUDA cores; 16 < M <= kMaxM on the tensor cores.
constexpr int kSmallMMax = 16;
constexpr int kMaxM = 65536;
bool gemm_m_supported(int M) { return M >= 1 && M <= kMaxM; }
bool gemm_on_tensor_cores(int M) { return M > kSmallMMax; }

int check_codes(const uint32_t* codes, const uint16_t* scales) {
    if (codes == nullptr || scales == nullptr) return TRELLIS_ERR_NULL;
    if (!aligned(codes, 16) || !aligned(scales, 2)) return TRELLIS_ERR_ALIGN;
    return TRELLIS_OK;
}


}  // namespace

namespace trellis {

int check_gemm(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M, int K, int N,
               int k, int L, int T, const uint16_t* out) {
    if (x == nullptr || out == nullptr) return TRELLIS_ERR_NULL;
    int rc = check_codes(codes, scales);
    if (rc != TRELLIS_OK) return rc;
    rc = check_geometry(K, N, k, L, T);
    if (rc != TRELLIS_OK) return rc;
    if (!gemm_m_supported(M)) return TRELLIS_ERR_UNSUPPORTED;
    if (!aligned(x, 16) || !aligned(out, 2)) return TRELLIS_ERR_ALIGN;
    return TRELLIS_OK;
}

}  // namespace trellis

namespace {

using trellis::check_gemm;

}  // namespace

extern "C" {

int trellis_abi_version(void) { return TRELLIS_ABI_VERSION; }

const char* trellis_status_string(int status) {
    switch (status) {
        case TRELLIS_OK: return "TRELLIS_OK";
        case TRELLIS_ERR_NULL: return "TRELLIS_ERR_NULL: a required pointer is NULL";
        case TRELLIS_ERR_SHAPE: return "TRELLIS_ERR_SHAPE: sizes inconsistent or out of range";
        case TRELLIS_ERR_UNSUPPORTED: return "TRELLIS_ERR_UNSUPPORTED: k, L, T or M outside the accepted set";
        case TRELLIS_ERR_ALIGN: return "TRELLIS_ERR_ALIGN: a pointer misses its required alignment";
        case TRELLIS_ERR_CUDA: return "TRELLIS_ERR_CUDA: the CUDA runtime reported an error";
        case TRELLIS_ERR_TIMEOUT: return "TRELLIS_ERR_TIMEOUT: a bounded device-side wait gave up";
        case TRELLIS_ERR_WORKSPACE: return "TRELLIS_ERR_WORKSPACE: workspace missing or too small";
        default: return "TRELLIS_ERR_UNKNOWN";
    }
}

int trellis_decode(const uint32_t* codes, const uint16_t* scales, int K, int N, int k, int L, int T,
                   uint16_t* out_bf16, cudaStream_t stream) {
    int rc = check_codes(codes, scales);
    if (rc != TRELLIS_OK) return rc;
    if (out_bf16 == nullptr) return TRELLIS_ERR_NULL;
    rc = check_geometry(K, N, k, L, T);
    if (rc != TRELLIS_OK) return rc;
    if (!aligned(out_bf16, 16)) return TRELLIS_ERR_ALIGN;
    DeviceInfo dev;
    rc = device_info(dev);
    if (rc != TRELLIS_OK) return rc;
    return trellis::launch_decode(codes, scales, K, N, k, L, out_bf16, stream, dev);
}

int trellis_gemm_workspace_size(int M, int K, int N, int k, int L, int T, size_t* bytes) {
    if (bytes == nullptr) return TRELLIS_ERR_NULL;
    int rc = check_geometry(K, N, k, L, T);
    if (rc != TRELLIS_OK) return rc;
    if (!gemm_m_supported(M)) return TRELLIS_ERR_UNSUPPORTED;
    if (gemm_on_tensor_cores(M)) {   // the tensor-core path needs no workspace
        *bytes = 0;
        return TRELLIS_OK;
    }
    DeviceInfo dev;
    rc = device_info(dev);
    if (rc != TRELLIS_OK) return rc;
    *bytes = trellis::gemm_smallm_workspace_bytes(M, K, N, k, L, dev);
    return *bytes == 0 ? TRELLIS_ERR_SHAPE : TRELLIS_OK;
}

int trellis_gemm_ws(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M, int K,
                    int N, int k, int L, int T, uint16_t* out, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream) {
    int rc = check_gemm(x, codes, scales, M, K, N, k, L, T, out);
    if (rc != TRELLIS_OK) return rc;
    if (gemm_on_tensor_cores(M)) return trellis::launch_gemm_tc(x, codes, scales, M, K, N, k, L, out, stream);
    DeviceInfo dev;
    rc = device_info(dev);
    if (rc != TRELLIS_OK) return rc;
    const size_t need = trellis::gemm_smallm_workspace_bytes(M, K, N, k, L, dev);
    if (need == 0) return TRELLIS_ERR_SHAPE;
    if (workspace == nullptr || workspace_bytes < need) return TRELLIS_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return TRELLIS_ERR_ALIGN;
    return trellis::launch_gemm_smallm(x, codes, scales, M, K, N, k, L, out, workspace, workspace_bytes,
                                       stream, dev);
}

int trellis_gemm(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M, int K, int N,
                 int k, int L, int T, uint16_t* out, cudaStream_t stream) {
    int rc = check_gemm(x, codes, scales, M, K, N, k, L, T, out);
    if (rc != TRELLIS_OK) return rc;
    if (gemm_on_tensor_cores(M)) return trellis::launch_gemm_tc(x, codes, scales, M, K, N, k, L, out, stream);
    DeviceInfo dev;
    rc = device_info(dev);
    if (rc != TRELLIS_OK) return rc;
    const size_t need = trellis::gemm_smallm_workspace_bytes(M, K, N, k, L, dev);
    if (need == 0) return TRELLIS_ERR_SHAPE;
    if (need > trellis::kGemmScratchBytes) return TRELLIS_ERR_WORKSPACE;   // more than 170 SMs
    void* ws = nullptr;
    rc = trellis::gemm_static_scratch(&ws);
    if (rc != TRELLIS_OK) return rc;
    return trellis::launch_gemm_smallm(x, codes, scales, M, K, N, k, L, out, ws, trellis::kGemmScratchBytes,
                                       stream, dev);
}

int trellis_gemm_gateup_workspace_size(int M, int K, int N, int k, int L, int T, size_t* bytes) {
    if (bytes == nullptr) return TRELLIS_ERR_NULL;
    int rc = check_geometry(K, N, k, L, T);
    if (rc != TRELLIS_OK) return rc;
    if (!gemm_m_supported(M)) return TRELLIS_ERR_UNSUPPORTED;
    if (gemm_on_tensor_cores(M)) {
        *bytes = 0;
        return TRELLIS_OK;
    }
    // both matrices' rows in one launch: twice the tile-groups (rounded)
    if (static_cast<long long>(N) * 2 * (K / T) >= (1ll << 31)) return TRELLIS_ERR_SHAPE;
    DeviceInfo dev;
    rc = device_info(dev);
    if (rc != TRELLIS_OK) return rc;
    *bytes = trellis::gemm_smallm_workspace_bytes(M, K, N, k, L, dev, true);
    return *bytes == 0 ? TRELLIS_ERR_SHAPE : TRELLIS_OK;
}

int trellis_gemm_gateup(const uint16_t* x, const uint32_t* codes_gate, const uint16_t* scales_gate,
                        const uint32_t* codes_up, const uint16_t* scales_up, int M, int K, int N, int k, int L,
                        int T, uint16_t* out_gate, uint16_t* out_up, uint16_t* out_act, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
    int rc = check_gemm(x, codes_gate, scales_gate, M, K, N, k, L, T, out_gate);
    if (rc != TRELLIS_OK) return rc;
    rc = check_gemm(x, codes_up, scales_up, M, K, N, k, L, T, out_up);
    if (rc != TRELLIS_OK) return rc;
    if (out_act != nullptr && !aligned(out_act, 2)) return TRELLIS_ERR_ALIGN;
    size_t need = 0;
    rc = trellis_gemm_gateup_workspace_size(M, K, N, k, L, T, &need);
    if (rc != TRELLIS_OK) return rc;
    DeviceInfo dev;
    rc = device_info(dev);
    if (rc != TRELLIS_OK) return rc;
    if (gemm_on_tensor_cores(M)) {
        rc = trellis::launch_gemm_tc(x, codes_gate, scales_gate, M, K, N, k, L, out_gate, stream);
        if (rc == TRELLIS_OK) rc = trellis::launch_gemm_tc(x, codes_up, scales_up, M, K, N, k, L, out_up, stream);
    } else {
        if (workspace == nullptr || workspace_bytes < need) return TRELLIS_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return TRELLIS_ERR_ALIGN;
        trellis::SecondMatrix up;
        up.codes = codes_up;
        up.scales = scales_up;
        up.out = out_up;
        rc = trellis::launch_gemm_smallm(x, codes_gate, scales_gate, M, K, N, k, L, out_gate, workspace,
                                         workspace_bytes, stream, dev, up);
    }
    if (rc == TRELLIS_OK && out_act != nullptr)
        rc = trellis::launch_silu_mul(out_gate, out_up, out_act, static_cast<size_t>(M) * N, stream, dev);
    return rc;
}

int trellis_selftest_wait_timeout(cudaStream_t stream) { return trellis::launch_wait_selftest(stream); }

int trellis_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return TRELLIS_ERR_CUDA;
    unsigned int flags = 0u;
    if (trellis::tc_take_device_error(&flags) != 0) return TRELLIS_ERR_CUDA;
    return flags != 0u ? TRELLIS_ERR_TIMEOUT : TRELLIS_OK;
}

}  // extern "C"

#ifdef TRELLIS_TRACE
// Trace build only (not declared in include/trellis.h and absent from the
// shipped library): attach a device buffer of `bytes` that the small-M
// kernels fill with clock64 stamps of their phases (layout beside
// kTraceCtaWords in gemm_smallm_kernel.cuh); NULL detaches.
namespace {
unsigned long long* g_trace = nullptr;
size_t g_trace_words = 0;
}  // namespace

namespace trellis {
unsigned long long* trace_buffer(size_t* words) {
    *words = g_trace_words;
    return g_trace;
}
}  // namespace trellis

extern "C" __attribute__((visibility("default"))) int trellis_trace_attach(void* buffer, size_t bytes) {
    g_trace = static_cast<unsigned long long*>(buffer);
    g_trace_words = buffer != nullptr ? bytes / sizeof(unsigned long long) : 0;
    return TRELLIS_OK;
}
#endif
