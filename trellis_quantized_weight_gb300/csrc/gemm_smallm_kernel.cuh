// Fused decode-and-multiply for 1 <= M <= 16 on the CUDA cores (sm_103a).
//
// What it computes: out[m, n] = bf16( sum_k w[n, k] * x[m, k] ), with w the
// decoded bf16 weights, products and sums in fp32 (the wide-prefill kernel on
// the page "mlx-bun 0.2.0 -> 0.4.0", trellis-wide-prefill.ts: decode each row
// once and share it across every activation row).
//
// Mapping (GB300-first, not the page's simdgroup layout):
//  * lane = output row.  A warp owns a "tile" of 32*R rows (lane l holds rows
//    l, l+32, ...), so all lanes of a warp sit at the same k at the same time
//    and every activation value it needs is one broadcast shared-memory read,
//    reused by the R rows and both weights of an f32x2 FMA.
//  * WARPS tiles form a "tile-group".  Work units are (tile-group, 32-wide
//    k-group) pairs, numbered tile-group-major, and CTA c takes the contiguous
//    unit range [c*U/P, (c+1)*U/P): every SM gets the same number of weights
//    whatever N and K are (stream-K split), and all warps of a CTA walk the
//    same k-groups, so the CTA stages the matching slice of x once, as fp32,
//    in shared memory.
//  * A row whose K-range is split over several CTAs writes fp32 partial sums
//    to the workspace; the last CTA to finish a tile (ticket from a per-tile
//    counter) adds the partials in CTA order, rounds to bf16, stores and resets
//    the counter.  The sum order is therefore fixed: identical inputs give
//    identical bits.  No CTA ever waits on another.
//  * Decode per weight: funnel shift + mask, hash IMAD, dp4a byte sum into a
//    float, the 3-op residual-corrected quotient, the scale multiply and a
//    bf16 round that keeps fp32 format; then MM/2 packed f32x2 FMAs per weight
//    pair per activation row.
#pragma once

#include <cstdint>

#include "kernels.h"
#include "trellis_device.cuh"

namespace trellis {

struct SmallMPlan {
    int M, K, N;
    int G;              // k-groups per row (K / 32)
    int row_words;      // K * k / 32
    int ntg;            // tile-groups
    int P;              // CTAs
    int units_max;      // ceil(U / P)
    long long U;        // units = ntg * G
    float* partials;    // workspace: [P][2][WARPS][M][R][32] fp32
    uint32_t* counters; // workspace: [ntg * WARPS]
};

template <int MM>
struct SmallMShape {
    static constexpr int R = 2;                       // rows per lane
    static constexpr int WARPS = (MM <= 8) ? 16 : 8;  // warps per CTA = tiles per tile-group
    static constexpr int MP = (MM == 1) ? 1 : ((MM + 1) & ~1);   // padded x rows in smem
    static constexpr int XS_UNIT = 32 * MP;           // floats of staged x per k-group
};

__device__ __forceinline__ int cta_of_unit(long long u, long long U, int P) {
    const long long c = ((u + 1) * P - 1) / U;
    return static_cast<int>(c < P - 1 ? c : P - 1);
}

template <int MM, int KB>
__global__ void __launch_bounds__(SmallMShape<MM>::WARPS * 32, 1)
gemm_smallm_kernel(const uint16_t* __restrict__ x, const uint32_t* __restrict__ codes,
                   const uint16_t* __restrict__ scales, uint16_t* __restrict__ out, SmallMPlan p) {
    using S = SmallMShape<MM>;
    constexpr int R = S::R, WARPS = S::WARPS, MP = S::MP, XS_UNIT = S::XS_UNIT;
    constexpr int WPB = kGroupsPerBlock * KB;
    constexpr int NT = WARPS * 32;
    extern __shared__ __align__(16) float xs[];

    const int c = blockIdx.x;
    const long long u0 = static_cast<long long>(c) * p.U / p.P;
    const long long u1 = static_cast<long long>(c + 1) * p.U / p.P;
    const int nunits = static_cast<int>(u1 - u0);
    const int tid = threadIdx.x;

    // ---- stage x for this CTA's k-groups: xs[q][kk/2][m][kk%2] (fp32) ----
    for (int q = 0; q < nunits; ++q) {
        const int k0 = static_cast<int>((u0 + q) % p.G) * 32;
        float* xq = xs + q * XS_UNIT;
        for (int e = tid; e < MP * 32; e += NT) {
            const int m = e >> 5, kk = e & 31;
            float v = 0.0f;
            if (m < MM) v = bf16_bits_to_f32(x[static_cast<size_t>(m) * p.K + k0 + kk]);
            xq[((kk >> 1) * MP + m) * 2 + (kk & 1)] = v;   // MP == 1 gives xq[kk]
        }
    }
    __syncthreads();

    const int warp = tid >> 5, lane = tid & 31;
    const int first_tg = static_cast<int>(u0 / p.G);

    for (long long u = u0; u < u1;) {
        const int tg = static_cast<int>(u / p.G);
        const int j0 = static_cast<int>(u - static_cast<long long>(tg) * p.G);
        const long long rest = u1 - u;
        const int len = static_cast<int>((p.G - j0) < rest ? (p.G - j0) : rest);
        const int j1 = j0 + len;
        const int q0 = static_cast<int>(u - u0);
        u += len;

        const int tile = tg * WARPS + warp;
        const int row0 = tile * 32 * R;
        if (row0 >= p.N) continue;   // whole tile beyond N: skipped by every CTA alike

        bool ok[R];
        float s[R];
        const uint32_t* rp[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int n = row0 + 32 * r + lane;
            ok[r] = n < p.N;
            s[r] = ok[r] ? bf16_bits_to_f32(__ldg(scales + n)) : 0.0f;
            rp[r] = codes + static_cast<size_t>(ok[r] ? n : 0) * p.row_words;
        }

        float2 acc[R][MM];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MM; ++m) acc[r][m] = make_float2(0.0f, 0.0f);

        uint32_t cur[R][KB + 1], nxt[R][KB + 1];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (ok[r]) {
                load_group_words<KB>(rp[r] + (j0 >> 3) * WPB, j0 & 7, cur[r]);
            } else {
#pragma unroll
                for (int i = 0; i <= KB; ++i) cur[r][i] = 0u;
            }
        }

        for (int j = j0; j < j1; ++j) {
            const int jn = j + 1;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (ok[r] && jn < j1) {
                    load_group_words<KB>(rp[r] + (jn >> 3) * WPB, jn & 7, nxt[r]);
                } else {
#pragma unroll
                    for (int i = 0; i <= KB; ++i) nxt[r][i] = 0u;
                }
            }
            const float* xq = xs + (q0 + (j - j0)) * XS_UNIT;
#pragma unroll
            for (int pp = 0; pp < 16; ++pp) {
                float2 xv[MM];
                if constexpr (MM == 1) {
                    xv[0] = *reinterpret_cast<const float2*>(xq + 2 * pp);
                } else {
#pragma unroll
                    for (int mm = 0; mm < MP / 2; ++mm) {
                        const float4 t = *reinterpret_cast<const float4*>(xq + (pp * MP + 2 * mm) * 2);
                        xv[2 * mm] = make_float2(t.x, t.y);
                        if (2 * mm + 1 < MM) xv[2 * mm + 1] = make_float2(t.z, t.w);
                    }
                }
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float wa = round_bf16_as_f32(
                        __fmul_rn(window_value(group_window<KB>(cur[r], 2 * pp)), s[r]));
                    const float wb = round_bf16_as_f32(
                        __fmul_rn(window_value(group_window<KB>(cur[r], 2 * pp + 1)), s[r]));
                    const float2 wv = make_float2(wa, wb);
#pragma unroll
                    for (int m = 0; m < MM; ++m) acc[r][m] = __ffma2_rn(wv, xv[m], acc[r][m]);
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int i = 0; i <= KB; ++i) cur[r][i] = nxt[r][i];
        }

        float v[R][MM];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MM; ++m) v[r][m] = __fadd_rn(acc[r][m].x, acc[r][m].y);

        if (j0 == 0 && j1 == p.G) {
            // this CTA owns the whole K-range of the tile-group
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (ok[r])
#pragma unroll
                    for (int m = 0; m < MM; ++m)
                        out[static_cast<size_t>(m) * p.N + row0 + 32 * r + lane] =
                            bf16_bits_rn(v[r][m]);
            continue;
        }

        // ---- split row: publish the partial, the last arriver reduces ----
        const int slot = (tg == first_tg) ? 0 : 1;
        float* mine = p.partials + ((static_cast<size_t>(c) * 2 + slot) * WARPS + warp) * (MM * R * 32);
#pragma unroll
        for (int m = 0; m < MM; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) mine[(m * R + r) * 32 + lane] = v[r][m];
        __threadfence();
        __syncwarp();
        uint32_t ticket = 0;
        if (lane == 0) ticket = atomicAdd(p.counters + tile, 1u);
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        const long long tg_u0 = static_cast<long long>(tg) * p.G;
        const int c_first = cta_of_unit(tg_u0, p.U, p.P);
        const int c_last = cta_of_unit(tg_u0 + p.G - 1, p.U, p.P);
        if (ticket != static_cast<uint32_t>(c_last - c_first)) continue;

        __threadfence();
        float sum[R][MM];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MM; ++m) sum[r][m] = 0.0f;
        for (int cc = c_first; cc <= c_last; ++cc) {
            const long long cc_u0 = static_cast<long long>(cc) * p.U / p.P;
            const int cc_slot = (tg == static_cast<int>(cc_u0 / p.G)) ? 0 : 1;
            const float* src =
                p.partials + ((static_cast<size_t>(cc) * 2 + cc_slot) * WARPS + warp) * (MM * R * 32);
#pragma unroll
            for (int m = 0; m < MM; ++m)
#pragma unroll
                for (int r = 0; r < R; ++r)
                    sum[r][m] = __fadd_rn(sum[r][m], __ldcg(src + (m * R + r) * 32 + lane));
        }
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (ok[r])
#pragma unroll
                for (int m = 0; m < MM; ++m)
                    out[static_cast<size_t>(m) * p.N + row0 + 32 * r + lane] =
                        bf16_bits_rn(sum[r][m]);
        if (lane == 0) p.counters[tile] = 0u;
    }
}

// Host-side planning shared by the per-k instantiation files.
template <int MM>
SmallMPlan plan_smallm(int K, int N, int k, const DeviceInfo& dev) {
    using S = SmallMShape<MM>;
    SmallMPlan p{};
    p.M = MM;
    p.K = K;
    p.N = N;
    p.G = K / 32;
    p.row_words = K / 32 * k;
    const int rows_per_tg = S::WARPS * 32 * S::R;
    p.ntg = (N + rows_per_tg - 1) / rows_per_tg;
    p.U = static_cast<long long>(p.ntg) * p.G;
    long long P = dev.num_sms;
    if (P > p.U) P = p.U;
    const long long bytes_per_unit = static_cast<long long>(S::XS_UNIT) * 4;
    const long long ucap = dev.max_smem_optin / bytes_per_unit;
    if ((p.U + P - 1) / P > ucap) P = (p.U + ucap - 1) / ucap;
    p.P = static_cast<int>(P);
    p.units_max = static_cast<int>((p.U + P - 1) / P);
    return p;
}

// Workspace layout: a fixed-capacity counter region at offset 0 (the same
// place for every geometry, so a workspace reused across geometries never
// finds stale partial sums where it expects counters), then the partial sums.
// Counters are left at zero by every call; partial sums need no clearing.
constexpr size_t kCounterCapacity = size_t(1) << 18;            // tiles
constexpr size_t kCounterBytes = kCounterCapacity * sizeof(uint32_t);

template <int MM>
size_t smallm_workspace_bytes(const SmallMPlan& p) {
    using S = SmallMShape<MM>;
    const size_t partials = static_cast<size_t>(p.P) * 2 * S::WARPS * MM * S::R * 32 * 4;
    return kCounterBytes + partials;
}

template <int MM>
bool smallm_fits_counters(const SmallMPlan& p) {
    return static_cast<size_t>(p.ntg) * SmallMShape<MM>::WARPS <= kCounterCapacity;
}

template <int MM, int KB>
int launch_smallm_instance(const uint16_t* x, const uint32_t* codes, const uint16_t* scales,
                           int K, int N, uint16_t* out, void* ws, size_t ws_bytes,
                           cudaStream_t stream, const DeviceInfo& dev) {
    using S = SmallMShape<MM>;
    SmallMPlan p = plan_smallm<MM>(K, N, KB, dev);
    if (!smallm_fits_counters<MM>(p)) return -2;
    const size_t need = smallm_workspace_bytes<MM>(p);
    if (ws_bytes < need || ws == nullptr) return -7;
    p.counters = static_cast<uint32_t*>(ws);
    p.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes);
    const size_t smem = static_cast<size_t>(p.units_max) * S::XS_UNIT * 4;
    static bool attr_set = false;   // idempotent; a race only repeats the call
    if (!attr_set) {
        if (cudaFuncSetAttribute(gemm_smallm_kernel<MM, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 dev.max_smem_optin) != cudaSuccess)
            return -5;
        attr_set = true;
    }
    gemm_smallm_kernel<MM, KB><<<p.P, S::WARPS * 32, smem, stream>>>(x, codes, scales, out, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

template <int KB>
int launch_smallm_k(int M, const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int K,
                    int N, uint16_t* out, void* ws, size_t ws_bytes, cudaStream_t stream,
                    const DeviceInfo& dev);

}  // namespace trellis
