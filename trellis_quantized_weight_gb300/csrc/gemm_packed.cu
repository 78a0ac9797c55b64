// Token packing (trellis_gemm_packed): several groups of activation rows
// multiplied by the same weights in one product (mapPackedTokens on the page
// "mlx-bun 0.4.0 -> 0.5.0", token-groups.ts): the groups are gathered into a
// packed x by one copy launch (copy_groups.cu, up to 64 groups a launch), the
// product runs once through trellis_gemm_ws, and one more copy launch scatters
// the packed output rows back to each group's output.
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"
#include "trellis.h"

using trellis::DeviceInfo;

namespace {

constexpr long long kMaxPackedM = 65536;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// Total rows of the groups, or a negative status.
long long packed_rows(const int* rows, int groups) {
    if (rows == nullptr) return TRELLIS_ERR_NULL;
    if (groups < 1) return TRELLIS_ERR_SHAPE;
    long long M = 0;
    for (int g = 0; g < groups; ++g) {
        if (rows[g] < 1) return TRELLIS_ERR_SHAPE;
        M += rows[g];
        if (M > kMaxPackedM) return TRELLIS_ERR_UNSUPPORTED;
    }
    return M;
}

// Workspace layout: the product's own workspace at offset 0, then packed x
// [M, K] and packed out [M, N].  The product keeps per-tile counters in the
// first 1 MiB of its workspace and leaves them at zero; that region is always
// reserved (even when this M needs none, as on the tensor cores), so the
// copies never land on it and one workspace serves any sequence of calls.
constexpr size_t kCounterRegion = size_t(1) << 20;

struct PackedLayout {
    size_t x_off = 0, out_off = 0, gemm_bytes = 0, total = 0;
};

int packed_layout(int M, int K, int N, int k, int L, int T, bool single, PackedLayout* lay) {
    size_t gemm = 0;
    const int rc = trellis_gemm_workspace_size(M, K, N, k, L, T, &gemm);
    if (rc != TRELLIS_OK) return rc;
    PackedLayout l;
    l.gemm_bytes = gemm;
    if (single) {
        l.total = gemm;
    } else {
        l.x_off = round256(gemm > kCounterRegion ? gemm : kCounterRegion);
        l.out_off = l.x_off + round256(static_cast<size_t>(M) * K * 2);
        l.total = l.out_off + round256(static_cast<size_t>(M) * N * 2);
    }
    *lay = l;
    return TRELLIS_OK;
}

}  // namespace

extern "C" {

int trellis_gemm_packed_workspace_size(const int* rows, int groups, int K, int N, int k, int L, int T,
                                       size_t* bytes) {
    if (bytes == nullptr) return TRELLIS_ERR_NULL;
    const long long M = packed_rows(rows, groups);
    if (M < 0) return static_cast<int>(M);
    PackedLayout lay;
    const int rc = packed_layout(static_cast<int>(M), K, N, k, L, T, groups == 1, &lay);
    if (rc != TRELLIS_OK) return rc;
    *bytes = lay.total;
    return TRELLIS_OK;
}

int trellis_gemm_packed(const uint16_t* const* xs, const int* rows, int groups, const uint32_t* codes,
                        const uint16_t* scales, int K, int N, int k, int L, int T, uint16_t* const* outs,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (xs == nullptr || outs == nullptr || codes == nullptr || scales == nullptr) return TRELLIS_ERR_NULL;
    const long long M = packed_rows(rows, groups);
    if (M < 0) return static_cast<int>(M);
    for (int g = 0; g < groups; ++g) {
        if (xs[g] == nullptr || outs[g] == nullptr) return TRELLIS_ERR_NULL;
        if (!aligned(xs[g], 16) || !aligned(outs[g], 2)) return TRELLIS_ERR_ALIGN;
    }
    PackedLayout lay;
    int rc = packed_layout(static_cast<int>(M), K, N, k, L, T, groups == 1, &lay);
    if (rc != TRELLIS_OK) return rc;
    if (!aligned(codes, 16) || !aligned(scales, 2)) return TRELLIS_ERR_ALIGN;
    if (lay.total > 0 && (workspace == nullptr || workspace_bytes < lay.total)) return TRELLIS_ERR_WORKSPACE;
    if (workspace != nullptr && !aligned(workspace, 256)) return TRELLIS_ERR_ALIGN;
    char* ws = static_cast<char*>(workspace);
    void* gemm_ws = lay.gemm_bytes > 0 ? ws : nullptr;
    if (groups == 1)
        return trellis_gemm_ws(xs[0], codes, scales, static_cast<int>(M), K, N, k, L, T, outs[0], gemm_ws,
                               lay.gemm_bytes, stream);

    DeviceInfo dev;
    if (cudaGetDevice(&dev.device) != cudaSuccess ||
        cudaDeviceGetAttribute(&dev.num_sms, cudaDevAttrMultiProcessorCount, dev.device) != cudaSuccess)
        return TRELLIS_ERR_CUDA;
    uint16_t* px = reinterpret_cast<uint16_t*>(ws + lay.x_off);
    uint16_t* pout = reinterpret_cast<uint16_t*>(ws + lay.out_off);
    // gather: group g's rows to packed rows pos_g .., kCopyBatch groups a launch
    size_t pos = 0;
    for (int g0 = 0; g0 < groups; g0 += trellis::kCopyBatch) {
        const int nb = groups - g0 < trellis::kCopyBatch ? groups - g0 : trellis::kCopyBatch;
        trellis::CopyBatch b;
        for (int j = 0; j < nb; ++j) {
            const size_t n = static_cast<size_t>(rows[g0 + j]);
            b.src[j] = xs[g0 + j];
            b.dst[j] = px + pos * K;
            b.count[j] = n * K;
            pos += n;
        }
        rc = trellis::launch_copy_groups(b, nb, stream, dev);
        if (rc != TRELLIS_OK) return rc;
    }
    rc = trellis_gemm_ws(px, codes, scales, static_cast<int>(M), K, N, k, L, T, pout, gemm_ws, lay.gemm_bytes,
                         stream);
    if (rc != TRELLIS_OK) return rc;
    // scatter: packed output rows back to each group's output
    pos = 0;
    for (int g0 = 0; g0 < groups; g0 += trellis::kCopyBatch) {
        const int nb = groups - g0 < trellis::kCopyBatch ? groups - g0 : trellis::kCopyBatch;
        trellis::CopyBatch b;
        for (int j = 0; j < nb; ++j) {
            const size_t n = static_cast<size_t>(rows[g0 + j]);
            b.src[j] = pout + pos * N;
            b.dst[j] = outs[g0 + j];
            b.count[j] = n * N;
            pos += n;
        }
        rc = trellis::launch_copy_groups(b, nb, stream, dev);
        if (rc != TRELLIS_OK) return rc;
    }
    return TRELLIS_OK;
}

}  // extern "C"
