// trellis_gemm_noalloc: the fused decode-and-multiply for callers that cannot
// allocate device memory.
//
// The product splits long rows over several CTAs and needs scratch memory for
// their fp32 partial sums and per-tile counters.  trellis_gemm allocates that
// scratch itself on first use and trellis_gemm_ws takes it from the caller.
// Some callers can do neither: code that runs where cudaMalloc is not allowed
// or not wanted (inside an allocator or a memory-pool callback, in a process
// whose device memory is fully reserved up front, or under a runtime that
// forbids allocation on its hot path).  This entry point takes its scratch from
// one fixed array compiled into the library instead.
//
// The array lives as long as the library is loaded, on every GPU that loads
// it, and every call shares it:
//  * its first 1 MiB holds the tile counters, which must read zero before a
//    call: the array starts zeroed, the first call on each device clears that
//    region once more, and every completed call leaves it at zero;
//  * the rest holds partial sums, which need no clearing;
//  * calls that may overlap on the same GPU (for instance on two streams)
//    race on it; each GPU has its own copy.
#include <cstdint>
#include <mutex>

#include "gemm_smallm_kernel.cuh"
#include "kernels.h"
#include "trellis.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
    bool ready = false;
    void* scratch = nullptr;          // device address of g_noalloc_scratch on this device
    trellis::DeviceInfo info;
};

// Set-up, once per device, with that device current: look up the device
// address of the array (its host-side name is only a stand-in) and clear the
// counter region.
int noalloc_device(NoAllocDevice& out) {
    static std::mutex mu;
    static NoAllocDevice devs[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TRELLIS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    NoAllocDevice& d = devs[dev];
    if (!d.ready) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return TRELLIS_ERR_CUDA;
        d.info.device = dev;
        if (cudaDeviceGetAttribute(&d.info.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return TRELLIS_ERR_CUDA;
        if (cudaMemset(p, 0, trellis::kCounterBytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
            return TRELLIS_ERR_CUDA;
        d.scratch = p;
        d.ready = true;
    }
    out = d;
    return TRELLIS_OK;
}

}  // namespace

extern "C" int trellis_gemm_noalloc(const uint16_t* x, const uint32_t* codes, const uint16_t* scales,
                                    int M, int K, int N, int k, int L, int T, uint16_t* out,
                                    cudaStream_t stream) {
    int rc = trellis::check_gemm(x, codes, scales, M, K, N, k, L, T, out);   // as trellis_gemm
    if (rc != TRELLIS_OK) return rc;
    size_t need = 0;
    rc = trellis_gemm_workspace_size(M, K, N, k, L, T, &need);
    if (rc != TRELLIS_OK) return rc;
    // Beyond the fixed array.  Defensive: the scratch grows with the SM count
    // (1 MiB of counters plus at most 18 KiB a CTA), so no accepted geometry
    // exceeds 16 MiB on a device with at most 853 SMs.
    if (need > kNoAllocScratchBytes) return TRELLIS_ERR_WORKSPACE;
    if (M > 16) return trellis::launch_gemm_tc(x, codes, scales, M, K, N, k, L, out, stream);   // no scratch
    NoAllocDevice d;
    rc = noalloc_device(d);
    if (rc != TRELLIS_OK) return rc;
    return trellis::launch_gemm_smallm(x, codes, scales, M, K, N, k, L, out, d.scratch, kNoAllocScratchBytes,
                                       stream, d.info);
}
