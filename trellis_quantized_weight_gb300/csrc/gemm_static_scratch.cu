// Split-K scratch of trellis_gemm: a fixed region of static device memory in
// the library image, so that trellis_gemm neither allocates nor synchronises.
//
// The small-M product balances work over all SMs by splitting rows' K-ranges
// across CTAs; the split rows' fp32 partial sums and per-tile counters need
// scratch memory (the layout of trellis_gemm_ws's workspace: counters at
// offset 0, then partial sums).  trellis_gemm takes no workspace argument, so
// this array is its scratch:
//  * it is zero when the module is loaded (a __device__ array without an
//    initializer is zero-initialised, like any object of static storage
//    duration), and every completed call leaves its counter region at zero;
//    the partial sums need no clearing;
//  * the only host-side step is looking up its device address, once per
//    device, which neither allocates nor synchronises;
//  * every trellis_gemm call on a device shares it, so calls that may overlap
//    on the GPU race (trellis_gemm_ws with separate workspaces serves
//    concurrent streams);
//  * its size covers 1 MiB of counters plus up to 18 KiB of partial sums per SM
//    (M = 16 at 12 warps) for up to 170 SMs; on a device with more SMs the
//    shapes that need more are rejected, and trellis_gemm_ws serves them.
#include <cstdint>
#include <mutex>

#include "gemm_smallm_kernel.cuh"
#include "kernels.h"
#include "trellis.h"

namespace trellis {

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_gemm_scratch[kGemmScratchBytes];

}  // namespace

int gemm_static_scratch(void** ptr) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TRELLIS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        // the host-side name of the array only stands in for it: ask the
        // runtime for its address on this device
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gemm_scratch) != cudaSuccess) return TRELLIS_ERR_CUDA;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return TRELLIS_OK;
}

}  // namespace trellis
