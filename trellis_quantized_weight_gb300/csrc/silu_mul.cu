// Gate/up activation: act = bf16(silu(g) * u) elementwise over bf16 arrays, with
// silu(v) = v / (1 + e^-v) computed in fp32 from the bf16 inputs (the SiLU-gated
// product of the two projections that share x).  HBM bound: 6 bytes per element.
#include "kernels.h"
#include "trellis_device.cuh"

namespace trellis {

namespace {

__device__ __forceinline__ uint16_t silu_mul_one(uint16_t g, uint16_t u) {
    const float v = bf16_bits_to_f32(g);
    const float s = v / (1.0f + expf(-v));
    return bf16_bits_rn(s * bf16_bits_to_f32(u));
}

__global__ void __launch_bounds__(256) silu_mul_kernel(const uint16_t* __restrict__ g,
                                                       const uint16_t* __restrict__ u,
                                                       uint16_t* __restrict__ act, size_t count, int vec) {
    griddep_wait();   // g and u are written by the preceding kernels on the stream
    const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t done = 0;
    if (vec) {   // all three arrays 16-byte aligned: 8 elements per access
        const size_t nvec = count / 8;
        for (size_t i = tid; i < nvec; i += nthreads) {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(g) + i);
            const uint4 b = __ldg(reinterpret_cast<const uint4*>(u) + i);
            const uint32_t ga[4] = {a.x, a.y, a.z, a.w}, ub[4] = {b.x, b.y, b.z, b.w};
            uint32_t r[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const uint16_t lo = silu_mul_one(static_cast<uint16_t>(ga[h]), static_cast<uint16_t>(ub[h]));
                const uint16_t hi = silu_mul_one(static_cast<uint16_t>(ga[h] >> 16), static_cast<uint16_t>(ub[h] >> 16));
                r[h] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            }
            reinterpret_cast<uint4*>(act)[i] = make_uint4(r[0], r[1], r[2], r[3]);
        }
        done = nvec * 8;
    }
    for (size_t i = done + tid; i < count; i += nthreads) act[i] = silu_mul_one(g[i], u[i]);
    griddep_launch_dependents();
}

}  // namespace

int launch_silu_mul(const uint16_t* g, const uint16_t* u, uint16_t* act, size_t count, cudaStream_t stream,
                    const DeviceInfo& dev) {
    if (count == 0) return 0;
    const bool vec = ((reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(u) |
                       reinterpret_cast<uintptr_t>(act)) & 15u) == 0;
    const size_t work = vec ? count / 8 + 8 : count;
    size_t blocks = (work + 255) / 256;
    const size_t max_blocks = static_cast<size_t>(dev.num_sms) * 8;
    if (blocks > max_blocks) blocks = max_blocks;
    const cudaError_t e = launch_programmatic(silu_mul_kernel, static_cast<unsigned>(blocks), 256u, 0, stream,
                                              g, u, act, count, vec ? 1 : 0);
    return e == cudaSuccess ? 0 : -5;
}

}  // namespace trellis
