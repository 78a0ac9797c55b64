// Internal launch interface between the C ABI (trellis_abi.cu) and the kernel
// translation units.  Arguments reaching these functions are already validated.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace trellis {

// Accepted geometry: 256-weight blocks, k = 1..8 bits per weight, windows of
// k < L <= 24 bits.  The page's wrapper envelope (k in {2,3,4}, L = 12) runs
// on kernels specialised for it ("fast geometry": a compile-time window width
// and, for M <= 16, the shared-memory quotient table); every other (k, L)
// runs on instantiations with a run-time window mask and the computed
// quotient.
constexpr int kT_abi = 256;
constexpr int kMinK = 1, kMaxK = 8, kMaxL = 24;
inline bool fast_geometry(int k, int L) { return L == 12 && k >= 2 && k <= 4; }

#ifdef TRELLIS_TRACE
// Trace build only: the device buffer the small-M kernels stamp their phases
// into (null until trellis_trace_attach), and its size in 64-bit words.
unsigned long long* trace_buffer(size_t* words);
#endif

struct DeviceInfo {
    int device = 0;
    int num_sms = 0;
    int max_smem_optin = 0;   // bytes of dynamic shared memory a CTA may opt into
};

// Opts `kernel` into `bytes` of dynamic shared memory on the current device.
// The attribute belongs to the device, so each call site keeps one bit per
// device (`done`) and calls cudaFuncSetAttribute once per device; a race only
// repeats the call.  Returns false on a CUDA error.
template <class Kernel>
bool smem_opt_in(Kernel kernel, int bytes, std::atomic<unsigned long long>& done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    done.fetch_or(bit, std::memory_order_acq_rel);
    return true;
}

// Launch with programmatic stream serialization: the grid may begin while the
// previous kernel on the stream is still draining.  Kernels launched this way
// touch no global memory before griddepcontrol.wait, which returns once the
// previous grid has completed and its writes are visible, so stream order is
// kept for every input and output.
template <class... Params, class... Args>
cudaError_t launch_programmatic(void (*kernel)(Params...), unsigned grid, unsigned block, size_t smem,
                                cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// The argument checks of trellis_gemm, in its order (pointers, codes and
// scales, geometry, M, then the alignment of x and out); returns 0 or a
// trellis_status.  Shared by every entry point that takes trellis_gemm's
// arguments, so each rejects a call the same way.
int check_gemm(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M, int K, int N, int k,
               int L, int T, const uint16_t* out);

// trellis_gemm's split-K scratch: a static device array of kGemmScratchBytes
// (1 MiB of tile counters, then partial sums), zero when loaded and left with
// zero counters by every completed call.  Writes its address on the current
// device to *ptr; no allocation, no synchronisation.  Returns 0 or a
// trellis_status.
constexpr size_t kGemmScratchBytes = size_t(4) << 20;
int gemm_static_scratch(void** ptr);

// Dense decode of all N rows into out [N, K].  Returns 0 or a trellis_status.
int launch_decode(const uint32_t* codes, const uint16_t* scales, int K, int N, int k, int L,
                  uint16_t* out, cudaStream_t stream, const DeviceInfo& dev);

// A second weight matrix [N, K] sharing x with the first (gate and up
// projections), multiplied in the same launch; codes == nullptr: none.
struct SecondMatrix {
    const uint32_t* codes = nullptr;
    const uint16_t* scales = nullptr;
    uint16_t* out = nullptr;
};

// Fused decode-and-multiply for 1 <= M <= 16 (CUDA cores).  Both matrices
// of a SecondMatrix share one launch only for the fast geometry; otherwise
// the caller runs two launches.
size_t gemm_smallm_workspace_bytes(int M, int K, int N, int k, int L, const DeviceInfo& dev, bool two = false);
int launch_gemm_smallm(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M,
                       int K, int N, int k, int L, uint16_t* out, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream, const DeviceInfo& dev, const SecondMatrix& second = SecondMatrix{});

// act[i] = bf16(silu(g[i]) * u[i]) for count bf16 elements (silu(v) = v / (1 + e^-v),
// in fp32 from the bf16 inputs).  Returns 0 or a trellis_status.
int launch_silu_mul(const uint16_t* g, const uint16_t* u, uint16_t* act, size_t count, cudaStream_t stream,
                    const DeviceInfo& dev);

// Fused decode-and-multiply for M > 16 on the tensor cores (tcgen05): one
// launch per up to 256 activation rows.
int launch_gemm_tc(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M, int K, int N, int k,
                   int L, uint16_t* out, cudaStream_t stream);
// Copies of up to kCopyBatch contiguous runs of bf16 elements (count[g]
// elements from src[g] to dst[g]) in one launch, chained by programmatic
// launch: the gather and scatter of trellis_gemm_packed.  Returns 0 or a
// trellis_status.
constexpr int kCopyBatch = 64;
struct CopyBatch {
    const uint16_t* src[kCopyBatch];
    uint16_t* dst[kCopyBatch];
    unsigned long long count[kCopyBatch];
};
int launch_copy_groups(const CopyBatch& batch, int groups, cudaStream_t stream, const DeviceInfo& dev);

// Launches one thread whose bounded wait on an mbarrier runs out (nothing
// arrives), which sets the device error word exactly as a product wait that
// gives up would.  Returns 0 or a trellis_status.
int launch_wait_selftest(cudaStream_t stream);
// Reads and clears the tensor-core kernel's device error word (bit 0: a
// bounded wait gave up).  Returns 0 or a trellis_status.
int tc_take_device_error(unsigned int* flags);

}  // namespace trellis
