// Dense decode: packed codes -> bf16 [N, K] ("expand" mode).
//
// Flat view: a (row, block) pair is one "item" of T = 256 weights.  Because
// codes and the output are both row-major with K a multiple of T, item i
// reads words [i*wpb, (i+1)*wpb) of `codes` and writes weights
// [i*256, (i+1)*256) of `out`.  One warp decodes 4 consecutive items per step:
// lane l works on item (step*4 + l/8), group g = l%8 (32 weights).  The
// lookahead word of a group is the first word of group g-1, which lane l-1
// holds (lane l+7 for g = 0, whose window tails wrap to word 0 of the block),
// so it comes by one shuffle.
//
// Stores: each lane's 32 weights (64 bytes) go to a per-warp shared-memory
// buffer laid out exactly like the warp's 2 KB of output, and one lane hands
// the buffer to the TMA engine as a single bulk copy (cp.async.bulk), double
// buffered.  The next step's codes are loaded before the current step is
// decoded.
//
// Bound: HBM.  Per item it reads 32*k bytes and writes 512 bytes.
#include "kernels.h"
#include "trellis_device.cuh"

namespace trellis {

constexpr int kDecodeWarps = 8;
constexpr int kDecodeStageBytes = 4 * kT * 2;   // 4 items of bf16 = 2 KB per warp and buffer

// LL: window width fixed at compile time (12), or 0 for the run-time width
// given by lmask = 2^L - 1.
template <int KB, int LL>
__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_kernel(const uint32_t* __restrict__ codes, const uint16_t* __restrict__ scales,
              uint32_t items, FastDiv blocks_per_row, uint32_t lmask, uint16_t* __restrict__ out) {
    constexpr int WPB = kGroupsPerBlock * KB;
    __shared__ __align__(128) unsigned char stage[kDecodeWarps][2][kDecodeStageBytes];

    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int g = lane & 7;
    const int sub = lane >> 3;
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
    const int src_lane = (g == 0) ? lane + 7 : lane - 1;

    auto load = [&](uint32_t base, uint32_t (&w)[KB], float& s) {
        const uint32_t item = base + sub;
        if (item < items) {
            ldg_group<KB>(codes + static_cast<size_t>(item) * WPB + (kGroupsPerBlock - 1 - g) * KB, w);
            s = bf16_bits_to_f32(__ldg(scales + blocks_per_row.div(item)));
        } else {
#pragma unroll
            for (int i = 0; i < KB; ++i) w[i] = 0u;
            s = 0.0f;
        }
    };

    griddep_wait();   // no global memory is touched before the previous grid's writes are visible
    uint32_t cw[KB];
    float cs = 0.0f;
    uint32_t base = warp * 4u;
    if (base < items) load(base, cw, cs);
    int buf = 0;
    const uint32_t stage_lane =
        static_cast<uint32_t>(__cvta_generic_to_shared(&stage[wib][0][0])) + static_cast<uint32_t>(lane) * 64u;

    for (; base < items; base += nwarps * 4u) {
        const uint32_t next = base + nwarps * 4u;
        uint32_t nw[KB];
        float ns = 0.0f;
        if (next < items) {
            load(next, nw, ns);
        } else {
#pragma unroll
            for (int i = 0; i < KB; ++i) nw[i] = 0u;
        }

        uint32_t w[KB + 1];
#pragma unroll
        for (int i = 0; i < KB; ++i) w[i] = cw[i];
        w[KB] = __shfl_sync(0xffffffffu, w[0], src_lane);

        uint32_t packed[16];
#pragma unroll
        for (int jp = 0; jp < 16; ++jp) {
            const float2 v = __fmul2_rn(window_value2(group_window<KB, LL>(w, 2 * jp, lmask),
                                                      group_window<KB, LL>(w, 2 * jp + 1, lmask)),
                                        make_float2(cs, cs));
            packed[jp] = pack_bf16x2(v.x, v.y);
        }

        // The bulk copy issued two steps ago from this buffer must have read it.
        if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncwarp();
        const uint32_t dst = stage_lane + static_cast<uint32_t>(buf) * kDecodeStageBytes;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         :: "r"(dst + q * 16u), "r"(packed[4 * q]), "r"(packed[4 * q + 1]),
                            "r"(packed[4 * q + 2]), "r"(packed[4 * q + 3]) : "memory");
        // make the generic-proxy stores visible to the bulk copy (async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
            const uint32_t nvalid = (items - base) < 4u ? (items - base) : 4u;
            uint16_t* gdst = out + static_cast<size_t>(base) * kT;
            const uint32_t src = static_cast<uint32_t>(__cvta_generic_to_shared(&stage[wib][buf][0]));
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                         :: "l"(gdst), "r"(src), "r"(nvalid * static_cast<uint32_t>(kT * 2)) : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        buf ^= 1;
#pragma unroll
        for (int i = 0; i < KB; ++i) cw[i] = nw[i];
        cs = ns;
    }
    griddep_launch_dependents();
    // the shared buffers must outlive the bulk copies that read them
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

namespace {

template <int KB, int LL>
cudaError_t launch_decode_instance(unsigned grid, cudaStream_t stream, const uint32_t* codes,
                                   const uint16_t* scales, uint32_t items, FastDiv fd, uint32_t lmask,
                                   uint16_t* out) {
    return launch_programmatic(decode_kernel<KB, LL>, grid, kDecodeWarps * 32, 0, stream, codes, scales, items, fd,
                               lmask, out);
}

}  // namespace

int launch_decode(const uint32_t* codes, const uint16_t* scales, int K, int N, int k, int L,
                  uint16_t* out, cudaStream_t stream, const DeviceInfo& dev) {
    const uint32_t blocks_per_row = static_cast<uint32_t>(K / kT);
    const uint64_t items64 = static_cast<uint64_t>(N) * blocks_per_row;
    const uint32_t items = static_cast<uint32_t>(items64);
    const uint32_t warps_needed = (items + 3u) / 4u;
    const uint32_t ctas_needed = (warps_needed + kDecodeWarps - 1u) / kDecodeWarps;
    // Up to 24 CTAs a SM, about three times what fits at once (7 with 32 KB of
    // staging each): CTAs that finish are replaced by waiting ones, which
    // balances the end of the launch.  Measured on the 17408 x 5120 decode, as
    // CTAs a SM / us: 6 / 37.8, 7 / 40.8 (one wave, 10 or 11 steps a warp),
    // 8 / 37.1, 12 / 35.5, 16 / 34.9, 24 / 34.4, 32 / 35.4, uncapped / 39.4.
    const uint32_t max_ctas = static_cast<uint32_t>(dev.num_sms) * 24u;
    const unsigned grid = ctas_needed < max_ctas ? ctas_needed : max_ctas;
    const FastDiv fd(blocks_per_row);
    const uint32_t lmask = (1u << L) - 1u;
    cudaError_t e;
    if (fast_geometry(k, L)) {
        switch (k) {
            case 2: e = launch_decode_instance<2, kL>(grid, stream, codes, scales, items, fd, lmask, out); break;
            case 3: e = launch_decode_instance<3, kL>(grid, stream, codes, scales, items, fd, lmask, out); break;
            default: e = launch_decode_instance<4, kL>(grid, stream, codes, scales, items, fd, lmask, out); break;
        }
    } else {
        switch (k) {
            case 1: e = launch_decode_instance<1, 0>(grid, stream, codes, scales, items, fd, lmask, out); break;
            case 2: e = launch_decode_instance<2, 0>(grid, stream, codes, scales, items, fd, lmask, out); break;
            case 3: e = launch_decode_instance<3, 0>(grid, stream, codes, scales, items, fd, lmask, out); break;
            case 4: e = launch_decode_instance<4, 0>(grid, stream, codes, scales, items, fd, lmask, out); break;
            case 5: e = launch_decode_instance<5, 0>(grid, stream, codes, scales, items, fd, lmask, out); break;
            case 6: e = launch_decode_instance<6, 0>(grid, stream, codes, scales, items, fd, lmask, out); break;
            case 7: e = launch_decode_instance<7, 0>(grid, stream, codes, scales, items, fd, lmask, out); break;
            case 8: e = launch_decode_instance<8, 0>(grid, stream, codes, scales, items, fd, lmask, out); break;
            default: return -3;
        }
    }
    return e == cudaSuccess ? 0 : -5;
}

}  // namespace trellis
