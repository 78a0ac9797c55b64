// Host dispatch of the small-M fused decode-and-multiply (plan, workspace size,
// bit-width switch).  The kernels live in gemm_smallm_k{2,3,4}.cu (k in {2,3,4},
// L = 12), gemm_smallm2_k{2,3,4}.cu (the same, two matrices) and
// gemm_smallm_g_k{1..8}.cu (every other geometry).
#include "gemm_smallm_kernel.cuh"

namespace trellis {

// 0 when the geometry needs more tile counters than the workspace layout holds.
template <class C>
static size_t ws_bytes_of(int K, int N, int k, const DeviceInfo& dev, bool two) {
    const SmallMPlan p = plan_smallm<C>(K, N, k, dev, two);
    return smallm_fits_counters<C>(p) ? smallm_workspace_bytes<C>(p) : 0;
}

template <int MM>
static size_t ws_bytes_for(int K, int N, int k, int L, const DeviceInfo& dev, bool two) {
    if (fast_geometry(k, L))
        return two ? ws_bytes_of<typename SmallMDefault<MM>::two>(K, N, k, dev, true)
                   : ws_bytes_of<typename SmallMDefault<MM>::type>(K, N, k, dev, false);
    // other geometries run the two matrices of a pair as two launches, one
    // after the other on the stream, through the same workspace
    switch (k) {
#define TRELLIS_GK(KV) \
    case KV: return ws_bytes_of<typename SmallMDefault<MM>::template general<KV>>(K, N, k, dev, false);
        TRELLIS_GK(1) TRELLIS_GK(2) TRELLIS_GK(3) TRELLIS_GK(4)
        TRELLIS_GK(5) TRELLIS_GK(6) TRELLIS_GK(7) TRELLIS_GK(8)
#undef TRELLIS_GK
        default: return 0;
    }
}

size_t gemm_smallm_workspace_bytes(int M, int K, int N, int k, int L, const DeviceInfo& dev, bool two) {
    switch (M) {
#define TRELLIS_CASE(MV) \
    case MV: return ws_bytes_for<MV>(K, N, k, L, dev, two);
        TRELLIS_CASE(1) TRELLIS_CASE(2) TRELLIS_CASE(3) TRELLIS_CASE(4)
        TRELLIS_CASE(5) TRELLIS_CASE(6) TRELLIS_CASE(7) TRELLIS_CASE(8)
        TRELLIS_CASE(9) TRELLIS_CASE(10) TRELLIS_CASE(11) TRELLIS_CASE(12)
        TRELLIS_CASE(13) TRELLIS_CASE(14) TRELLIS_CASE(15) TRELLIS_CASE(16)
#undef TRELLIS_CASE
        default: return 0;
    }
}

namespace {

int launch_general(int M, int K, int N, int k, int L, const uint16_t* x, const uint32_t* codes,
                   const uint16_t* scales, uint16_t* out, void* ws, size_t ws_bytes, cudaStream_t stream,
                   const DeviceInfo& dev) {
    switch (k) {
        case 1: return launch_smallm_g_k<1>(M, L, x, codes, scales, K, N, out, ws, ws_bytes, stream, dev);
        case 2: return launch_smallm_g_k<2>(M, L, x, codes, scales, K, N, out, ws, ws_bytes, stream, dev);
        case 3: return launch_smallm_g_k<3>(M, L, x, codes, scales, K, N, out, ws, ws_bytes, stream, dev);
        case 4: return launch_smallm_g_k<4>(M, L, x, codes, scales, K, N, out, ws, ws_bytes, stream, dev);
        case 5: return launch_smallm_g_k<5>(M, L, x, codes, scales, K, N, out, ws, ws_bytes, stream, dev);
        case 6: return launch_smallm_g_k<6>(M, L, x, codes, scales, K, N, out, ws, ws_bytes, stream, dev);
        case 7: return launch_smallm_g_k<7>(M, L, x, codes, scales, K, N, out, ws, ws_bytes, stream, dev);
        case 8: return launch_smallm_g_k<8>(M, L, x, codes, scales, K, N, out, ws, ws_bytes, stream, dev);
        default: return -3;
    }
}

}  // namespace

int launch_gemm_smallm(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M,
                       int K, int N, int k, int L, uint16_t* out, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream, const DeviceInfo& dev, const SecondMatrix& second) {
    if (!fast_geometry(k, L)) {
        int rc = launch_general(M, K, N, k, L, x, codes, scales, out, workspace, workspace_bytes, stream, dev);
        if (rc == 0 && second.codes != nullptr)
            rc = launch_general(M, K, N, k, L, x, second.codes, second.scales, second.out, workspace,
                                workspace_bytes, stream, dev);
        return rc;
    }
    if (second.codes != nullptr) {
        switch (k) {
            case 2: return launch_smallm2_k<2>(M, x, codes, scales, K, N, out, workspace, workspace_bytes, stream, dev, second);
            case 3: return launch_smallm2_k<3>(M, x, codes, scales, K, N, out, workspace, workspace_bytes, stream, dev, second);
            case 4: return launch_smallm2_k<4>(M, x, codes, scales, K, N, out, workspace, workspace_bytes, stream, dev, second);
            default: return -3;
        }
    }
    switch (k) {
        case 2: return launch_smallm_k<2>(M, x, codes, scales, K, N, out, workspace, workspace_bytes, stream, dev);
        case 3: return launch_smallm_k<3>(M, x, codes, scales, K, N, out, workspace, workspace_bytes, stream, dev);
        case 4: return launch_smallm_k<4>(M, x, codes, scales, K, N, out, workspace, workspace_bytes, stream, dev);
        default: return -3;
    }
}

}  // namespace trellis
