// Gather / scatter of token groups for trellis_gemm_packed: each group is one
// contiguous run of bf16 elements on both sides (a group's rows are contiguous
// in its own buffer and in the packed buffer), so one launch copies up to
// kCopyBatch groups, blockIdx.y selecting the group.  16-byte vectors when
// both ends of a group are 16-byte aligned, 2-byte elements otherwise.
#include "kernels.h"
#include "trellis_device.cuh"

namespace trellis {

namespace {

__global__ void __launch_bounds__(256) copy_groups_kernel(CopyBatch b) {
    griddep_wait();   // the sources may be the previous kernel's output
    const int g = blockIdx.y;
    const uint16_t* __restrict__ src = b.src[g];
    uint16_t* __restrict__ dst = b.dst[g];
    const unsigned long long n = b.count[g];
    const unsigned long long stride = static_cast<unsigned long long>(gridDim.x) * blockDim.x;
    const unsigned long long t0 = static_cast<unsigned long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    unsigned long long done = 0;
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0) {
        const unsigned long long nv = n / 8;
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        uint4* d4 = reinterpret_cast<uint4*>(dst);
        for (unsigned long long i = t0; i < nv; i += stride) d4[i] = s4[i];
        done = nv * 8;
    }
    for (unsigned long long i = done + t0; i < n; i += stride) dst[i] = src[i];
    griddep_launch_dependents();
}

}  // namespace

int launch_copy_groups(const CopyBatch& batch, int groups, cudaStream_t stream, const DeviceInfo& dev) {
    if (groups < 1 || groups > kCopyBatch) return -3;
    unsigned long long most = 0;
    for (int g = 0; g < groups; ++g) most = batch.count[g] > most ? batch.count[g] : most;
    // 16-byte vectors: 2048 elements a CTA pass; enough CTAs that the largest
    // group spreads over the SMs, at most 4 per SM per group
    unsigned long long gx = (most + 2047) / 2048;
    const unsigned long long cap = static_cast<unsigned long long>(dev.num_sms) * 4;
    if (gx > cap) gx = cap;
    if (gx < 1) gx = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(groups));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, copy_groups_kernel, batch) == cudaSuccess ? 0 : -5;
}

}  // namespace trellis
