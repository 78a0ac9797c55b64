// Instantiations of the small-M fused decode-and-multiply for k = 2 bits and
// a run-time window width L (every geometry outside k in {2,3,4} with L = 12),
// one translation unit per bit width so the build compiles them in parallel.
#include "gemm_smallm_kernel.cuh"

namespace trellis {

template <>
int launch_smallm_g_k<2>(int M, int L, const uint16_t* x, const uint32_t* codes, const uint16_t* scales,
                         int K, int N, uint16_t* out, void* ws, size_t ws_bytes, cudaStream_t stream,
                         const DeviceInfo& dev) {
    switch (M) {
#define TRELLIS_CASE(MV) \
    case MV: return launch_smallm_instance<typename SmallMDefault<MV>::template general<2>, 2, 0>(x, codes, scales, K, N, out, ws, ws_bytes, stream, dev, SecondMatrix{}, L);
        TRELLIS_CASE(1) TRELLIS_CASE(2) TRELLIS_CASE(3) TRELLIS_CASE(4)
        TRELLIS_CASE(5) TRELLIS_CASE(6) TRELLIS_CASE(7) TRELLIS_CASE(8)
        TRELLIS_CASE(9) TRELLIS_CASE(10) TRELLIS_CASE(11) TRELLIS_CASE(12)
        TRELLIS_CASE(13) TRELLIS_CASE(14) TRELLIS_CASE(15) TRELLIS_CASE(16)
#undef TRELLIS_CASE
        default: return -3;
    }
}

}  // namespace trellis
