// Internal launch interface between the C ABI (trellis_abi.cu) and the kernel
// translation units.  Arguments reaching these functions are already validated.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace trellis {

// The geometry the kernels are compiled for (the envelope of the page's
// wrapper: 12-bit windows, 256-weight blocks).
constexpr int kL_abi = 12;
constexpr int kT_abi = 256;

struct DeviceInfo {
    int device = 0;
    int num_sms = 0;
    int max_smem_optin = 0;   // bytes of dynamic shared memory a CTA may opt into
};

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

// Dense decode of all N rows into out [N, K].  Returns 0 or a trellis_status.
int launch_decode(const uint32_t* codes, const uint16_t* scales, int K, int N, int k,
                  uint16_t* out, cudaStream_t stream, const DeviceInfo& dev);

// A second weight matrix [N, K] sharing x with the first (gate and up
// projections), multiplied in the same launch; codes == nullptr: none.
struct SecondMatrix {
    const uint32_t* codes = nullptr;
    const uint16_t* scales = nullptr;
    uint16_t* out = nullptr;
};

// Fused decode-and-multiply for 1 <= M <= 16 (CUDA cores).
size_t gemm_smallm_workspace_bytes(int M, int K, int N, int k, const DeviceInfo& dev, bool two = false);
int launch_gemm_smallm(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M,
                       int K, int N, int k, uint16_t* out, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream, const DeviceInfo& dev, const SecondMatrix& second = SecondMatrix{});

// act[i] = bf16(silu(g[i]) * u[i]) for count bf16 elements (silu(v) = v / (1 + e^-v),
// in fp32 from the bf16 inputs).  Returns 0 or a trellis_status.
int launch_silu_mul(const uint16_t* g, const uint16_t* u, uint16_t* act, size_t count, cudaStream_t stream,
                    const DeviceInfo& dev);

// Fused decode-and-multiply for M > 16 on the tensor cores (tcgen05), in
// chunks of 64 activation rows.
int launch_gemm_tc(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M, int K, int N, int k,
                   uint16_t* out, cudaStream_t stream);
// Reads and clears the tensor-core kernel's device error word (bit 0: a
// bounded wait gave up).  Returns 0 or a trellis_status.
int tc_take_device_error(unsigned int* flags);

}  // namespace trellis
