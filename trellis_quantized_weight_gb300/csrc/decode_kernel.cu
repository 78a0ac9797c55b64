// Dense decode: packed codes -> bf16 [N, K] ("expand" mode).
//
// Flat view: a (row, block) pair is one "item" of T = 256 weights.  Because
// codes and the output are both row-major with K a multiple of T, item i
// reads words [i*wpb, (i+1)*wpb) of `codes` and writes weights
// [i*256, (i+1)*256) of `out`.  One warp decodes 4 items per step: lane l works
// on item (step*4 + l/8), group g = l%8 (32 weights).  The lookahead word of a
// group is the first word of group g-1, which lane l-1 holds (lane l+7 for
// g = 0, whose window tails wrap to word 0 of the block), so it comes by one
// shuffle.  Each lane writes its 32 weights as 64 contiguous bytes.
//
// Bound: HBM.  Per item it reads 32*k bytes and writes 512 bytes; the decode is
// about 10 integer/fp32 instructions per weight, below the HBM time on GB300.
#include "kernels.h"
#include "trellis_device.cuh"

namespace trellis {

template <int KB>
__global__ void __launch_bounds__(256)
decode_kernel(const uint32_t* __restrict__ codes, const uint16_t* __restrict__ scales,
              uint32_t items, FastDiv blocks_per_row, uint16_t* __restrict__ out) {
    constexpr int WPB = kGroupsPerBlock * KB;
    const int lane = threadIdx.x & 31;
    const int g = lane & 7;
    const int sub = lane >> 3;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    const int src_lane = (g == 0) ? lane + 7 : lane - 1;

    for (uint32_t base = warp * 4u; base < items; base += nwarps * 4u) {
        const uint32_t item = base + sub;
        const bool valid = item < items;
        uint32_t w[KB + 1];
        float s = 0.0f;
        if (valid) {
            const uint32_t* p = codes + static_cast<size_t>(item) * WPB + (kGroupsPerBlock - 1 - g) * KB;
            if constexpr (KB == 4) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
                w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            } else if constexpr (KB == 2) {
                const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
                w[0] = v.x; w[1] = v.y;
            } else {
#pragma unroll
                for (int i = 0; i < KB; ++i) w[i] = __ldg(p + i);
            }
            s = bf16_bits_to_f32(__ldg(scales + blocks_per_row.div(item)));
        } else {
#pragma unroll
            for (int i = 0; i < KB; ++i) w[i] = 0u;
        }
        w[KB] = __shfl_sync(0xffffffffu, w[0], src_lane);
        if (!valid) continue;

        uint32_t packed[16];
#pragma unroll
        for (int jp = 0; jp < 16; ++jp) {
            const float a = __fmul_rn(window_value(group_window<KB>(w, 2 * jp)), s);
            const float b = __fmul_rn(window_value(group_window<KB>(w, 2 * jp + 1)), s);
            packed[jp] = pack_bf16x2(a, b);
        }
        uint4* dst = reinterpret_cast<uint4*>(out + static_cast<size_t>(item) * kT + 32 * g);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
    }
}

int launch_decode(const uint32_t* codes, const uint16_t* scales, int K, int N, int k,
                  uint16_t* out, cudaStream_t stream, const DeviceInfo& dev) {
    const uint32_t blocks_per_row = static_cast<uint32_t>(K / kT);
    const uint64_t items64 = static_cast<uint64_t>(N) * blocks_per_row;
    const uint32_t items = static_cast<uint32_t>(items64);
    const uint32_t warps_needed = (items + 3u) / 4u;
    const uint32_t ctas_needed = (warps_needed + 7u) / 8u;
    const uint32_t max_ctas = static_cast<uint32_t>(dev.num_sms) * 8u;
    const uint32_t grid = ctas_needed < max_ctas ? ctas_needed : max_ctas;
    const FastDiv fd(blocks_per_row);
    switch (k) {
        case 2: decode_kernel<2><<<grid, 256, 0, stream>>>(codes, scales, items, fd, out); break;
        case 3: decode_kernel<3><<<grid, 256, 0, stream>>>(codes, scales, items, fd, out); break;
        case 4: decode_kernel<4><<<grid, 256, 0, stream>>>(codes, scales, items, fd, out); break;
        default: return -3;
    }
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

}  // namespace trellis
