// Fused decode-and-multiply for M > 16 activation rows on the 5th-generation
// tensor cores (tcgen05, sm_103a).
//
// What it computes is the same as the CUDA-core product (the wide-prefill
// kernel on the page "mlx-bun 0.2.0 -> 0.4.0", trellis-wide-prefill.ts):
// out[m, n] = bf16( sum_k w[n, k] * x[m, k] ) with w the decoded bf16 weights.
// With tens of activation rows the multiply is a real dense contraction, so
// the decoded weights go to the tensor cores instead of the FMA pipes:
//
//   D[n, m] (TMEM, fp32, 128 lanes x NB columns) += A[n, k] * B[m, k]^T
//   A = decoded weight tile, 128 rows x 16 k, bf16, K-major
//   B = activation tile,      NB rows x 16 k, bf16, K-major, shared memory
//
// NB (the MMA's N) is 64, 128 or 256: one launch serves up to NB activation
// rows, and larger M runs in NB-row chunks, each decoding the weights again.
// One CTA owns 128 weight rows and the whole K range, with 16 decode warps,
// one TMA warp and one MMA warp (one thread issues the 8 tcgen05.mma, K = 16
// each, of a 128-k stage and commits them to the stage's "empty" barrier).
// Two kernels:
//   * gemm_tca_kernel, k = 2 .. 8: the TMA thread loads each block's code
//     words (one or two 128-byte boxes a row) for the CTA's 128 rows into
//     shared memory next to the activation tiles; decode warp w takes weight
//     rows 32*(w%4) .. +31 (one row a lane) and group w/4 of each stage, reads
//     its words from shared memory and writes the decoded bf16 values straight
//     into tensor memory (tcgen05.st), where the MMA takes A from.  Four A
//     slots in tensor memory; four or six activation slots, two at NB = 256.
//   * gemm_tc_kernel, k = 1 (a block's 8 words are a quarter of a code box):
//     decode warps load their code words from global memory and write the A
//     tile to shared memory in the K-major 128-byte-swizzled layout (two
//     k-blocks of 64 k, each row of a k-block 128 bytes, and inside every 8-row
//     (1 KB) atom the 16-byte chunk c of row r stored at chunk c ^ r),
//     published to the tensor cores by a proxy fence.
// The quotient: with NB = 64 and the page's geometry (k in {2, 3, 4}, 12-bit
// windows) the tensor-memory kernel reads it from the per-lane shared-memory
// table of the CUDA-core kernel (one dp4a address and one load a window,
// indexed by the hash's byte sum; trellis_device.cuh), which its freed shared
// memory holds; otherwise it is computed on the FMA pipe (two-part
// reciprocal, two windows per f32x2 instruction).  In both kernels
// the TMA warp loads each stage's activation tile with two 2-D tensor copies
// (one per k-block, 128-byte rows, swizzled by the TMA into the MMA's layout;
// the box covers the chunk's rows rounded up to 8, and rows beyond it only feed
// accumulator columns that are never stored), and after the last stage the
// decode warps read the accumulator back with tcgen05.ld, round to bf16 and
// store out[m, n] (each store instruction writes 32 consecutive n).
//
// Every mbarrier wait is bounded; a wait that runs out records an error in a
// device word (read by trellis_device_status) and the CTA winds down without
// leaving asynchronous work behind: the TMA copies complete on barriers of
// their own, which the TMA thread waits for (bounded) before it leaves, the
// decode warps wait for their own tensor-memory stores, and the MMA thread
// always commits and waits for its last MMAs, so nothing is in flight when the
// tensor memory is released.
#include <cuda.h>
#include <cstdint>
#include <mutex>

#include "kernels.h"
#include "trellis_device.cuh"

namespace trellis {

__device__ unsigned int g_tc_error = 0u;

namespace {

constexpr int kTcRows = 128;                 // weight rows per CTA (MMA M)
constexpr int kTcStageK = 128;               // k per pipeline stage
constexpr int kTcDecodeWarps = 16;
constexpr int kTcThreads = (kTcDecodeWarps + 2) * 32;
constexpr int kTcTmaWarp = kTcDecodeWarps;
constexpr int kTcMmaWarp = kTcDecodeWarps + 1;

// The shared-memory-A kernel computes the quotient (window_value2) rather
// than reading the per-lane table of the CUDA-core kernel: its A tiles take
// the shared memory the table's 113 KB would need.

constexpr int kABytes = kTcRows * kTcStageK * 2;     // 32 KB
constexpr int kSwK = 64;                             // k per 128-byte swizzled row (one k-block)
constexpr int kSwRowBytes = kSwK * 2;                // 128
constexpr int kSwAtomBytes = 8 * kSwRowBytes;        // 8-row atom: 1 KB, the stride between 8-row groups
constexpr int kAKBlockBytes = kTcRows * kSwRowBytes; // 16 KB

// Activation rows a chunk of M rows loads per k-block: M rounded up to 8, at
// most NB (the TMA box height).
__host__ __device__ constexpr int tc_box_rows(int M, int NB) { return ((M + 7) & ~7) < NB ? ((M + 7) & ~7) : NB; }

// One pass multiplies the decoded weights by NB activation rows (the MMA's N:
// 64, 128 or 256), so a weight tile is decoded once per NB rows of x.  Stages
// in flight fill about 192 KB of shared memory: 4 at NB = 64, 3 at 128, 2 at
// 256 (each stage: a 32 KB weight tile and an NB x 128 activation tile).
template <int NB>
struct TcShape {
    static constexpr int kStages = NB == 64 ? 4 : (NB == 128 ? 3 : 2);
    static constexpr int kBBytes = NB * kTcStageK * 2;
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kABytes;
    static constexpr int kOffBar = kOffB + kStages * kBBytes;
    static constexpr int kBarFull = 0, kBarEmpty = kStages, kBarTma = 2 * kStages, kBarDone = 3 * kStages;
    static constexpr int kOffTaddr = kOffBar + (3 * kStages + 1) * 8;
    // + 1 KB so that the base can be rounded up to the 1 KB the swizzle atoms need
    static constexpr int kSmemBytes = kOffTaddr + 16 + 1024;
    static constexpr int kTmemCols = NB;   // fp32 accumulator: 128 lanes x NB columns
    // instruction descriptor: kind::f16, D fp32, A and B bf16, both K-major,
    // N = NB (bits 17-22: N/8), M = 128 (bits 24-28: M/16)
    static constexpr uint32_t kInstrDesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                           (static_cast<uint32_t>(NB >> 3) << 17) |
                                           (static_cast<uint32_t>(kTcRows >> 4) << 24);
    static_assert(NB == 64 || NB == 128 || NB == 256, "MMA N");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds 227 KB");
    static_assert(kOffA % 1024 == 0 && kOffB % 1024 == 0 && kBBytes % 1024 == 0 && kABytes % 1024 == 0,
                  "swizzle atoms must start on 1 KB boundaries");
};

// A wait gives up after kWaitNs of wall-clock time (the %globaltimer
// nanosecond clock, read every 64 polls) or, as a backstop, after
// kWaitPollCap polls, whichever comes first.
constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s
constexpr uint32_t kWaitPollCap = 1u << 26;



// ---- PTX wrappers ------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 " selp.b32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0u;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait: false (and the error word set) when it runs out.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 0; i < kWaitPollCap; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && global_ns() - t0 > limit_ns) break;
    }
    atomicOr(&g_tc_error, 1u);
    return false;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) { return mbar_wait_for(bar, parity, kWaitNs); }
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
// Shared-memory matrix descriptor, K-major with the 128-byte swizzle: start
// address, leading offset unused by this layout (encoded 1), stride between
// 8-row atoms 1 KB, descriptor version 1 (bit 46), swizzle mode 2 (bits
// 61-63).  A k step of 16 inside an atom advances the start by 32 bytes: the
// swizzle is applied to the final address bits, as the stores applied it.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) |
           (1ull << 16) |
           (static_cast<uint64_t>(kSwAtomBytes >> 4) << 32) |
           (1ull << 46) |
           (2ull << 61);
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

// The k words of group 4*(stage%2) + gi of block stage/2 of a row (zeros for
// a row past N).  The window tails of the group spill into one more word; for
// gi = 1..3 that is the neighbouring lane's first word, and for groups 0 and 4
// (gi = 0) it is the first word of group 7 or 3 of the same block, which the
// gi = 3 lane of the same row loads for the other stage of the block: both
// arrive by shuffles (a second load here would double the loads in flight).
template <int KB>
__device__ __forceinline__ void tc_load_group(const uint32_t* __restrict__ row_codes, bool ok, int stage,
                                              int gi, uint32_t (&w)[KB]) {
    constexpr int WPB = kGroupsPerBlock * KB;
    const int b = stage >> 1, g = 4 * (stage & 1) + gi;
    if (ok) {
        ldg_group<KB>(row_codes + b * WPB + (kGroupsPerBlock - 1 - g) * KB, w);
    } else {
#pragma unroll
        for (int i = 0; i < KB; ++i) w[i] = 0u;
    }
}

// LL: window width fixed at compile time (12), or 0 for the run-time width
// given by lmask = 2^L - 1.
template <int KB, int NB, int LL>
__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tc_kernel(const uint32_t* __restrict__ codes, const uint16_t* __restrict__ scales,
               uint16_t* __restrict__ out, int M, int K, int N, int row_words, uint32_t lmask,
               const __grid_constant__ CUtensorMap x_map) {
    using S = TcShape<NB>;
    constexpr int kTcStages = S::kStages;
    constexpr int kBBytes = S::kBBytes;
    constexpr int kOffA = S::kOffA, kOffB = S::kOffB, kOffBar = S::kOffBar, kOffTaddr = S::kOffTaddr;
    constexpr int kBarFull = S::kBarFull, kBarEmpty = S::kBarEmpty, kBarDone = S::kBarDone;
    constexpr int kBarTma = S::kBarTma;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sraw = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    unsigned char* const smem = smem_raw + (sbase - sraw);
    const uint32_t bar_full = sbase + kOffBar + 8 * kBarFull;
    const uint32_t bar_empty = sbase + kOffBar + 8 * kBarEmpty;
    const uint32_t bar_done = sbase + kOffBar + 8 * kBarDone;
    const uint32_t bar_tma = sbase + kOffBar + 8 * kBarTma;
    const int nstages = K / kTcStageK;
    const int n0 = blockIdx.x * kTcRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(bar_full + 8 * s, kTcDecodeWarps);   // one arrival per decode warp
            mbar_init(bar_empty + 8 * s, 1);               // the MMAs' commit
            mbar_init(bar_tma + 8 * s, 1);                 // the TMA thread's expect_tx, then the bytes
        }
        mbar_init(bar_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_shared();
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(sbase + kOffTaddr), "r"(S::kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t taddr = *reinterpret_cast<volatile uint32_t*>(smem + kOffTaddr);
    // Before the wait for the previous grid: L2 prefetches of the code words
    // of the first stages (no data reaches registers; L2 is where every write
    // becomes visible, so a line fetched now cannot go stale), so that the
    // first loads after the wait hit L2.
    if (warp < kTcDecodeWarps) {
        const int prow = n0 + warp * 8 + (lane & 7);
        const int pgi = (lane >> 3) & 3;
        if (prow < N) {
            const uint32_t* rc = codes + static_cast<size_t>(prow) * row_words;
            constexpr int WPB = kGroupsPerBlock * KB;
#pragma unroll
            for (int st = 0; st < 4; ++st)
                if (st < nstages)
                    asm volatile("prefetch.global.L2 [%0];"
                                 :: "l"(rc + (st >> 1) * WPB + (kGroupsPerBlock - 1 - (4 * (st & 1) + pgi)) * KB));
        }
    }
    // everything above touches no global memory but L2 prefetches; loads only after this
    griddep_wait();

    if (warp < kTcDecodeWarps) {
        // ---------------------------------------------------------------- decode
        const int row_local = warp * 8 + (lane & 7);
        const int gi = (lane >> 3) & 3;
        const int row = n0 + row_local;
        const bool ok = row < N;
        const float sr = ok ? bf16_bits_to_f32(__ldg(scales + row)) : 0.0f;
        const float2 s2 = make_float2(sr, sr);
        const uint32_t* row_codes = codes + static_cast<size_t>(ok ? row : 0) * row_words;
        const int src_lane = (gi == 0) ? lane : lane - 8;
        const int r8 = lane & 7;
        // this thread's 64 bytes (k = 32*gi .. 32*gi+31) inside a stage's A
        // tile: k-block gi/2, 16-byte chunks 4*(gi%2) + q, swizzled by row
        const uint32_t a_row_off = static_cast<uint32_t>((gi >> 1) * kAKBlockBytes + row_local * kSwRowBytes);
        const uint32_t a_chunk0 = static_cast<uint32_t>(4 * (gi & 1));
        const uint32_t a_rsw = static_cast<uint32_t>(row_local & 7);
        // code words travel through a 4-deep register ring: stage i+3 is
        // loaded while stage i is decoded (ring indices are compile-time
        // because the stage loop is unrolled by the ring depth)
        constexpr int D = 4;
        static_assert(D % 2 == 0, "stage and ring slot share their parity");
        uint32_t ring[D][KB];
#pragma unroll
        for (int d = 0; d < D - 1; ++d) {
            if (d < nstages) {
                tc_load_group<KB>(row_codes, ok, d, gi, ring[d]);
            } else {
#pragma unroll
                for (int q = 0; q < KB; ++q) ring[d][q] = 0u;
            }
        }
        bool alive = true;
        uint32_t carry = 0u;   // word 4k of the block, for the odd stage
        for (int i0 = 0; i0 < nstages && alive; i0 += D) {
#pragma unroll
            for (int d = 0; d < D; ++d) {
                const int i = i0 + d;
                if (i >= nstages || !alive) break;
                const int s = i % kTcStages;
                const int pre = i + D - 1;
                if (pre < nstages) tc_load_group<KB>(row_codes, ok, pre, gi, ring[(d + D - 1) % D]);
                uint32_t w[KB + 1];
#pragma unroll
                for (int q = 0; q < KB; ++q) w[q] = ring[d][q];
                const uint32_t nb = __shfl_sync(0xffffffffu, ring[d][0], src_lane);
                // the lookahead word of groups 0 and 4 (the gi == 0 lanes): word
                // 0 of the block (group 7's first word, loaded for the odd stage
                // by the gi == 3 lane of the same row and already in the ring),
                // or word 4k (group 3's first word, handed over during the even
                // stage; i and d have the same parity because D is even)
                uint32_t look;
                if ((d & 1) == 0) {
                    look = __shfl_sync(0xffffffffu, ring[(d + 1) % D][0], r8 + 24);
                    carry = __shfl_sync(0xffffffffu, ring[d][0], r8 + 24);
                } else {
                    look = carry;
                }
                w[KB] = (gi == 0) ? look : nb;

                uint32_t packed[16];
#pragma unroll
                for (int jp = 0; jp < 16; ++jp) {
                    const float2 v = window_value2(group_window<KB, LL>(w, 2 * jp, lmask),
                                                   group_window<KB, LL>(w, 2 * jp + 1, lmask));
                    const float2 ws = __fmul2_rn(v, s2);
                    packed[jp] = pack_bf16x2(ws.x, ws.y);
                }
                if constexpr (kTcStages == 4) {
                    // Four slots: an even stage i and the odd stage i + 1 go to
                    // slots 0/2 and 1/3.  Only the odd stage's slot is probed,
                    // before the pair's first write: the commit that frees it
                    // (MMAs of stage i - 3) tracks every earlier MMA, those of
                    // stage i - 4 included.  Slots 1 and 3 are probed at every
                    // one of their phases, slots 0 and 2 never, so no probe
                    // skips a phase of its barrier.
                    if ((d & 1) == 0 && i + 1 >= kTcStages)
                        alive = mbar_wait(bar_empty + 8 * ((i + 1) % kTcStages), (((i + 1) / kTcStages) + 1) & 1);
                } else {
                    if (i >= kTcStages) alive = mbar_wait(bar_empty + 8 * s, ((i / kTcStages) + 1) & 1);
                }
                if (!alive) break;
                const uint32_t dst = sbase + kOffA + s * kABytes + a_row_off;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                                 :: "r"(dst + (((a_chunk0 + q) ^ a_rsw) << 4)), "r"(packed[4 * q]),
                                    "r"(packed[4 * q + 1]), "r"(packed[4 * q + 2]), "r"(packed[4 * q + 3])
                                 : "memory");
                if (kTcStages < 3 || (d & 1)) {
                    // with three or four stages, stages come in pairs (K / 128
                    // is even): one proxy fence and both arrivals after the
                    // second (two stages leave too little slack for it)
                    fence_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        if (kTcStages >= 3) mbar_arrive(bar_full + 8 * ((i - 1) % kTcStages));
                        mbar_arrive(bar_full + 8 * s);
                    }
                }
            }
        }

        // -------------------------------------------------------------- epilogue
        const bool done = alive && mbar_wait(bar_done, 0);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        // warp w reads TMEM lanes 32*(w%4) .. +31 (its weight rows) and the
        // columns (activation rows) of quarter w/4, 16 at a time
        const int sub = warp & 3, colq = warp >> 2;
#pragma unroll
        for (int cc = 0; cc < NB / 64 && done; ++cc) {
            const int col = colq * (NB / 4) + 16 * cc;
            uint32_t r[16];
            const uint32_t ta = taddr + (static_cast<uint32_t>(32 * sub) << 16) + static_cast<uint32_t>(col);
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                "%12, %13, %14, %15}, [%16];"
                : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                  "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                  "=r"(r[14]), "=r"(r[15])
                : "r"(ta));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            const int n = n0 + 32 * sub + lane;
            if (n < N) {
                // activation rows m >= M were zero-filled by the TMA; not stored
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (col + j < M)
                        out[static_cast<size_t>(col + j) * N + n] = bf16_bits_rn(__uint_as_float(r[j]));
            }
        }
    } else if (warp == kTcTmaWarp) {
        // ------------------------------------------------------------- x via TMA
        if (lane == 0) {
            // one box per k-block: the chunk's rows rounded up to 8 (rows past
            // M zero-filled by the TMA) x 64 k, 128 bytes a row
            const int rows = tc_box_rows(M, NB);
            int issued = 0;
            for (int i = 0; i < nstages; ++i) {
                const int s = i % kTcStages;
                if (i >= kTcStages && !mbar_wait(bar_empty + 8 * s, ((i / kTcStages) + 1) & 1)) break;
                mbar_arrive_expect_tx(bar_tma + 8 * s, static_cast<uint32_t>(2 * rows * kSwRowBytes));
                const uint32_t dst = sbase + kOffB + s * kBBytes;
#pragma unroll
                for (int kb = 0; kb < kTcStageK / kSwK; ++kb)
                    tma_load_2d(dst + kb * (NB * kSwRowBytes), &x_map, i * kTcStageK + kb * kSwK, 0,
                                bar_tma + 8 * s);
                issued = i + 1;
            }
            // Before the CTA can exit, every copy it issued has landed.  The
            // copies of the last (up to) kTcStages issued stages may not have
            // been consumed yet, but their completion depends on nothing else:
            // wait (bounded) for each.  After a normal run these return at once.
            for (int i = issued > kTcStages ? issued - kTcStages : 0; i < issued; ++i)
                (void)mbar_wait(bar_tma + 8 * (i % kTcStages), (i / kTcStages) & 1);
        }
    } else {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            // The descriptors of stage slot 0 at k step 0; every other operand
            // start is a fixed byte offset from it, a multiple of 16 that adds
            // to the start-address field (bits 0-13, shared-memory offsets
            // below 256 KB never carry out of it), so one 32-bit add per MMA
            // operand replaces rebuilding the descriptor: this thread shares
            // its sub-partition's issue slots with four decode warps.
            const uint64_t da0 = smem_desc(sbase + kOffA), db0 = smem_desc(sbase + kOffB);
            const uint32_t da_hi = static_cast<uint32_t>(da0 >> 32), db_hi = static_cast<uint32_t>(db0 >> 32);
            // With four slots the decode warps publish stages in pairs (their
            // arrivals for stages i and i + 1 come together), so the pair is
            // taken as a unit: the four barrier probes are issued back to back
            // and their latencies overlap, instead of four in a row between the
            // last decode arrival and the pair's MMAs (measured slower with
            // three slots, where it stays one stage at a time).
            constexpr int P = kTcStages == 4 ? 2 : 1;
            auto issue_stage = [&](int i) {
                const int s = i % kTcStages;
                const uint32_t da_s = static_cast<uint32_t>(da0) + static_cast<uint32_t>(s * (kABytes >> 4));
                const uint32_t db_s = static_cast<uint32_t>(db0) + static_cast<uint32_t>(s * (kBBytes >> 4));
#pragma unroll
                for (int kk = 0; kk < kTcStageK / 16; ++kk) {
                    const int kb = kk / (kSwK / 16), ks = kk % (kSwK / 16);
                    const uint32_t a_lo = da_s + static_cast<uint32_t>((kb * kAKBlockBytes + ks * 32) >> 4);
                    const uint32_t b_lo = db_s + static_cast<uint32_t>((kb * (NB * kSwRowBytes) + ks * 32) >> 4);
                    mma_bf16(taddr, (static_cast<uint64_t>(da_hi) << 32) | a_lo,
                             (static_cast<uint64_t>(db_hi) << 32) | b_lo, S::kInstrDesc, (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar_empty + 8 * s);
            };
            for (int i = 0; i < nstages; i += P) {
                bool ready[2 * P];
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const int t = i + p, s = t % kTcStages, par = (t / kTcStages) & 1;
                    ready[2 * p] = mbar_try_wait(bar_tma + 8 * s, par);
                    ready[2 * p + 1] = mbar_try_wait(bar_full + 8 * s, par);
                }
                bool ok = true;
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const int t = i + p, s = t % kTcStages, par = (t / kTcStages) & 1;
                    if (ok && !ready[2 * p]) ok = mbar_wait(bar_tma + 8 * s, par);
                    if (ok && !ready[2 * p + 1]) ok = mbar_wait(bar_full + 8 * s, par);
                }
                if (!ok) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll
                for (int p = 0; p < P; ++p) issue_stage(i + p);
            }
            // tracks every MMA issued above; also waited for here, so that no
            // MMA is in flight when the tensor memory is released, whether the
            // loop ran to the end or gave up
            mma_commit(bar_done);
            (void)mbar_wait(bar_done, 0);
        }
    }

    griddep_launch_dependents();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(S::kTmemCols)
                     : "memory");
    }
}


// ---- decoded tiles in tensor memory, code tiles by TMA ---------------------
// The decode warps take their code words from shared memory, where the TMA
// thread puts each block's 128 rows x 8k words as one or two boxes of 32 words
// (128 bytes a row, 128-byte swizzled: the 16-byte chunk c of row r at chunk
// c ^ (r % 8); a box past the block's words holds the start of the next block,
// unused, or zeros past the row's end), and write the decoded bf16 tile to
// tensor memory with tcgen05.st: there the MMA reads A directly, so no
// shared-memory A tile and no generic-to-async proxy fence are needed.
// Tensor-memory lane = weight row; a 32-bit column holds two consecutive k (the
// lower k in the low half).
constexpr int kCodeTileWords = 32;                             // one TMA box: 128 bytes a row
constexpr int kCodeTileBytes = kTcRows * kCodeTileWords * 4;   // 16 KB
constexpr int kCodeSlots = 3;
// boxes a block's code words take: its 8k words (one box for k <= 4, two above)
__host__ __device__ constexpr int code_boxes(int kb) {
    return (kGroupsPerBlock * kb + kCodeTileWords - 1) / kCodeTileWords;
}

// TAB: the quotient comes from the per-lane shared-memory table (NB = 64,
// where the table, three code slots and four activation slots fit in 227 KB).
template <int NB, bool TAB, int KB>
struct TcaShape {
    // A slots (tensor memory) and activation slots (shared memory); the
    // activation ring is shallower at NB = 256, whose tiles are 64 KB
    static constexpr int kStages = TAB ? 4 : (NB == 64 ? 6 : 4);
    static constexpr int kXStages = NB == 256 ? 2 : kStages;
    static constexpr int kBBytes = NB * kTcStageK * 2;
    static constexpr int kCodeBytes = code_boxes(KB) * kCodeTileBytes;   // one code slot
    static constexpr int kOffB = 0;
    static constexpr int kOffCode = kOffB + kXStages * kBBytes;
    static constexpr int kOffTable = kOffCode + kCodeSlots * kCodeBytes;
    static constexpr int kOffBar = kOffTable + (TAB ? kQuotientTableBytes : 0);
    static constexpr int kBarFull = 0, kBarEmpty = kStages, kBarTma = 2 * kStages,
                         kBarXEmpty = 2 * kStages + kXStages, kBarCode = 2 * kStages + 2 * kXStages,
                         kBarDone = 2 * kStages + 2 * kXStages + kCodeSlots;
    static constexpr int kOffTaddr = kOffBar + (kBarDone + 1) * 8;
    static constexpr int kSmemBytes = kOffTaddr + 16 + 1024;
    static constexpr int kAColBase = NB;          // accumulator: columns [0, NB)
    static constexpr int kTmemCols = 512;
    static_assert(NB == 64 || NB == 128 || NB == 256, "MMA N");
    static_assert(NB + kStages * 64 <= kTmemCols, "tensor memory columns");
    static_assert(kStages % 2 == 0 && kXStages <= 2 * kCodeSlots, "stage pairs; code slot reuse");
    static_assert(kSmemBytes <= 232448, "shared memory per CTA exceeds 227 KB");
    static_assert(!TAB || KB <= 4, "the quotient table serves 12-bit windows of k <= 4");
    static_assert(kOffCode % 1024 == 0 && kBBytes % 1024 == 0 && kCodeBytes % 1024 == 0,
                  "swizzle atoms must start on 1 KB boundaries");
};

__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
// Word w of this row in a code slot (row base `rb` in the slot's first box,
// row index mod 8 `r7`): box w / 32, 16-byte chunk (w % 32) / 4 swizzled.
__device__ __forceinline__ uint32_t code_word_addr(uint32_t rb, uint32_t r7, int w) {
    return rb + (static_cast<uint32_t>(w >> 5) * kCodeTileBytes) + ((static_cast<uint32_t>((w >> 2) & 7) ^ r7) << 4) +
           (static_cast<uint32_t>(w & 3) << 2);
}
// The KB words of group g of the tile's block and its lookahead word (the
// next word, or word 0 of the block for group 0).
template <int KB>
__device__ __forceinline__ void tile_group_words(uint32_t rb, uint32_t r7, int g, uint32_t (&w)[KB + 1]) {
    const int w0 = (kGroupsPerBlock - 1 - g) * KB;
    if constexpr (KB == 4 || KB == 8) {
        // 16-byte aligned chunks inside one box
#pragma unroll
        for (int q = 0; q < KB; q += 4)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[q]), "=r"(w[q + 1]), "=r"(w[q + 2]), "=r"(w[q + 3])
                         : "r"(code_word_addr(rb, r7, w0 + q)));
    } else if constexpr (KB == 2) {
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(code_word_addr(rb, r7, w0)));
    } else {
#pragma unroll
        for (int q = 0; q < KB; ++q) w[q] = lds32(code_word_addr(rb, r7, w0 + q));
    }
    w[KB] = lds32(code_word_addr(rb, r7, (w0 + KB) % (kGroupsPerBlock * KB)));
}

template <int KB, int NB, bool TAB, int LL>
__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tca_kernel(const uint16_t* __restrict__ scales, uint16_t* __restrict__ out, int M, int K, int N,
                uint32_t lmask, const __grid_constant__ CUtensorMap x_map,
                const __grid_constant__ CUtensorMap code_map) {
    using S = TcaShape<NB, TAB, KB>;
    constexpr int kBoxes = code_boxes(KB);
    constexpr int kS = S::kStages;
    constexpr int kBBytes = S::kBBytes;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sraw = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
    const uint32_t sbase = (sraw + 1023u) & ~1023u;
    unsigned char* const smem = smem_raw + (sbase - sraw);
    const uint32_t bar_full = sbase + S::kOffBar + 8 * S::kBarFull;
    const uint32_t bar_empty = sbase + S::kOffBar + 8 * S::kBarEmpty;
    const uint32_t bar_tma = sbase + S::kOffBar + 8 * S::kBarTma;
    const uint32_t bar_code = sbase + S::kOffBar + 8 * S::kBarCode;
    const uint32_t bar_done = sbase + S::kOffBar + 8 * S::kBarDone;
    constexpr int kSX = S::kXStages;
    // with as many activation slots as A slots, one commit frees both
    const uint32_t bar_xempty = kSX == kS ? bar_empty : sbase + S::kOffBar + 8 * S::kBarXEmpty;
    const int nstages = K / kTcStageK;
    const int nblocks = nstages / 2;
    const int n0 = blockIdx.x * kTcRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(bar_full + 8 * s, kTcDecodeWarps);   // the decode warps' arrivals
            mbar_init(bar_empty + 8 * s, 1);               // the MMAs' commit: A slot free
        }
        for (int s = 0; s < kSX; ++s) {
            mbar_init(bar_tma + 8 * s, 1);                 // expect_tx, then the activation bytes
            if (kSX != kS) mbar_init(bar_xempty + 8 * s, 1);   // the MMAs' commit: activation slot free
        }
        for (int c = 0; c < kCodeSlots; ++c) mbar_init(bar_code + 8 * c, 1);
        mbar_init(bar_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_async_shared();
    }
    if constexpr (TAB) build_quotient_table(reinterpret_cast<float*>(smem + S::kOffTable), threadIdx.x, kTcThreads);
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(sbase + S::kOffTaddr), "r"(S::kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t taddr = *reinterpret_cast<volatile uint32_t*>(smem + S::kOffTaddr);
    if (warp == kTcTmaWarp && lane == 0) {
        // L2 prefetches of the first code tiles (no data reaches the CTA
        // before the wait for the previous grid; L2 cannot hold a stale line)
        for (int b = 0; b < kCodeSlots && b < nblocks; ++b)
#pragma unroll
            for (int q = 0; q < kBoxes; ++q)
                asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                             :: "l"(reinterpret_cast<uint64_t>(&code_map)),
                                "r"(b * kGroupsPerBlock * KB + q * kCodeTileWords), "r"(n0)
                             : "memory");
    }
    griddep_wait();

    if (warp < kTcDecodeWarps) {
        // ---------------------------------------------------------------- decode
        // warp w: tensor-memory lanes (weight rows) 32*(w%4) .. +31, group
        // gi = w/4 of each stage's four 32-k groups (A columns 16*gi .. +15)
        const int q4 = warp & 3, gi = warp >> 2;
        const int row_local = 32 * q4 + lane;
        const int row = n0 + row_local;
        const float sr = row < N ? bf16_bits_to_f32(__ldg(scales + row)) : 0.0f;
        const float2 s2 = make_float2(sr, sr);
        const uint32_t r7 = static_cast<uint32_t>(row_local & 7);
        const uint32_t rb0 = sbase + S::kOffCode + static_cast<uint32_t>(row_local * kCodeTileWords * 4);
        const uint32_t t_row = taddr + (static_cast<uint32_t>(32 * q4) << 16) +
                               static_cast<uint32_t>(S::kAColBase + 16 * gi);
        const uint32_t lane_tbl = quotient_table_lane_address(smem + S::kOffTable, lane);
        bool alive = true;
        int c = 0, cpar = 0;     // code slot of block b and its phase parity
        int se = 0;              // A slot of the even stage 2b
        int spar = 1;            // parity the odd stage's slot probe waits for
        for (int b = 0; b < nblocks; ++b) {
            // The block's code tile, and the A slot of the odd stage 2b + 1:
            // the commit that frees it (MMAs of stage 2b + 1 - kS) tracks every
            // earlier MMA, those of stage 2b - kS (the even slot's previous
            // user) included.  Odd slots are probed at every one of their
            // phases, even slots never.  Both probes are issued before either
            // result is used, so their latencies overlap.
            const bool probe_slot = 2 * b + 1 >= kS;
            const bool code_ready = mbar_try_wait(bar_code + 8 * c, static_cast<uint32_t>(cpar));
            const bool slot_ready = !probe_slot || mbar_try_wait(bar_empty + 8 * (se + 1), static_cast<uint32_t>(spar));
            if (!code_ready) alive = mbar_wait(bar_code + 8 * c, static_cast<uint32_t>(cpar));
            if (alive && !slot_ready) alive = mbar_wait(bar_empty + 8 * (se + 1), static_cast<uint32_t>(spar));
            if (!alive) break;
            const uint32_t rb = rb0 + static_cast<uint32_t>(c * S::kCodeBytes);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t w[KB + 1];
                tile_group_words<KB>(rb, r7, 4 * h + gi, w);
                uint32_t packed[16];
#pragma unroll
                for (int jp = 0; jp < 16; ++jp) {
                    float2 v;
                    if constexpr (TAB) {
                        v.x = quotient_lookup(group_window<KB, kL>(w, 2 * jp), lane_tbl);
                        v.y = quotient_lookup(group_window<KB, kL>(w, 2 * jp + 1), lane_tbl);
                    } else {
                        v = window_value2(group_window<KB, LL>(w, 2 * jp, lmask),
                                          group_window<KB, LL>(w, 2 * jp + 1, lmask));
                    }
                    const float2 ws = __fmul2_rn(v, s2);
                    packed[jp] = pack_bf16x2(ws.x, ws.y);
                }
                asm volatile(
                    "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
                    "%11, %12, %13, %14, %15, %16};"
                    :: "r"(t_row + static_cast<uint32_t>(64 * (se + h))), "r"(packed[0]), "r"(packed[1]),
                       "r"(packed[2]), "r"(packed[3]), "r"(packed[4]), "r"(packed[5]), "r"(packed[6]),
                       "r"(packed[7]), "r"(packed[8]), "r"(packed[9]), "r"(packed[10]), "r"(packed[11]),
                       "r"(packed[12]), "r"(packed[13]), "r"(packed[14]), "r"(packed[15])
                    : "memory");
                if (h == 0 && b + 1 == nblocks) {
                    // the last block's even stage is published on its own, so
                    // that its MMAs overlap the odd stage's decode
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_full + 8 * se);
                }
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                if (b + 1 < nblocks) mbar_arrive(bar_full + 8 * se);
                mbar_arrive(bar_full + 8 * (se + 1));
            }
            if (++c == kCodeSlots) { c = 0; cpar ^= 1; }
            se += 2;
            if (se == kS) se = 0;
            if (2 * b + 3 >= kS && ((2 * b + 3) % kS) == 1) spar ^= 1;
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");

        // -------------------------------------------------------------- epilogue
        const bool done = alive && mbar_wait(bar_done, 0);
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int sub = warp & 3, colq = warp >> 2;
#pragma unroll
        for (int cc = 0; cc < NB / 64 && done; ++cc) {
            const int col = colq * (NB / 4) + 16 * cc;
            uint32_t r[16];
            const uint32_t ta = taddr + (static_cast<uint32_t>(32 * sub) << 16) + static_cast<uint32_t>(col);
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
                "%12, %13, %14, %15}, [%16];"
                : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                  "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
                  "=r"(r[14]), "=r"(r[15])
                : "r"(ta));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            const int n = n0 + 32 * sub + lane;
            if (n < N) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (col + j < M)
                        out[static_cast<size_t>(col + j) * N + n] = bf16_bits_rn(__uint_as_float(r[j]));
            }
        }
    } else if (warp == kTcTmaWarp) {
        // ------------------------------------------------- x and code tiles via TMA
        if (lane == 0) {
            const int rows = tc_box_rows(M, NB);
            int code_next = 0;
            auto issue_code = [&](int b) {
                const int cs = b % kCodeSlots;
                mbar_arrive_expect_tx(bar_code + 8 * cs, static_cast<uint32_t>(S::kCodeBytes));
#pragma unroll
                for (int q = 0; q < kBoxes; ++q)
                    tma_load_2d(sbase + S::kOffCode + cs * S::kCodeBytes + q * kCodeTileBytes, &code_map,
                                b * kGroupsPerBlock * KB + q * kCodeTileWords, n0, bar_code + 8 * cs);
            };
            for (; code_next < kCodeSlots && code_next < nblocks; ++code_next) issue_code(code_next);
            int issued = 0;
            for (int i = 0; i < nstages; ++i) {
                const int s = i % kSX;
                if (i >= kSX && !mbar_wait(bar_xempty + 8 * s, ((i / kSX) + 1) & 1)) break;
                mbar_arrive_expect_tx(bar_tma + 8 * s, static_cast<uint32_t>(2 * rows * kSwRowBytes));
                const uint32_t dst = sbase + S::kOffB + s * kBBytes;
#pragma unroll
                for (int kb = 0; kb < kTcStageK / kSwK; ++kb)
                    tma_load_2d(dst + kb * (NB * kSwRowBytes), &x_map, i * kTcStageK + kb * kSwK, 0,
                                bar_tma + 8 * s);
                issued = i + 1;
                // The MMAs of stage i - kSX are complete (waited above), so the
                // decode of every stage up to i - kSX is too: block p's code
                // slot (that of block p - kCodeSlots) is free once stage
                // 2 (p - kCodeSlots) + 1 <= i - kSX.
                if (i >= kSX) {
                    const int lim = ((i - kSX - 1) >> 1) + kCodeSlots;
                    for (; code_next <= lim && code_next < nblocks; ++code_next) issue_code(code_next);
                }
            }
            // every copy issued has landed before the CTA can exit
            for (int i = issued > kSX ? issued - kSX : 0; i < issued; ++i)
                (void)mbar_wait(bar_tma + 8 * (i % kSX), (i / kSX) & 1);
            for (int b = code_next > kCodeSlots ? code_next - kCodeSlots : 0; b < code_next; ++b)
                (void)mbar_wait(bar_code + 8 * (b % kCodeSlots), (b / kCodeSlots) & 1);
        }
    } else {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint64_t db0 = smem_desc(sbase + S::kOffB);
            const uint32_t db_hi = static_cast<uint32_t>(db0 >> 32);
            auto issue_stage = [&](int i) {
                const int s = i % kS, sx = i % kSX;
                const uint32_t ta_s = taddr + static_cast<uint32_t>(S::kAColBase + 64 * s);
                const uint32_t db_s = static_cast<uint32_t>(db0) + static_cast<uint32_t>(sx * (kBBytes >> 4));
#pragma unroll
                for (int kk = 0; kk < kTcStageK / 16; ++kk) {
                    const int kb = kk / (kSwK / 16), ks = kk % (kSwK / 16);
                    const uint32_t b_lo = db_s + static_cast<uint32_t>((kb * (NB * kSwRowBytes) + ks * 32) >> 4);
                    mma_bf16_ta(taddr, ta_s + static_cast<uint32_t>(8 * kk),
                                (static_cast<uint64_t>(db_hi) << 32) | b_lo, TcShape<NB>::kInstrDesc,
                                (i > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar_empty + 8 * s);
                if constexpr (kSX != kS) mma_commit(bar_xempty + 8 * sx);
            };
            // Stages are published in pairs (the last pair stage by stage), so
            // the four barrier probes of a pair are issued back to back (their
            // latencies overlap), and each stage's MMAs go out as soon as its
            // own barriers have completed.
            for (int i = 0; i < nstages; i += 2) {
                bool ready[4];
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int t = i + p;
                    ready[2 * p] = mbar_try_wait(bar_tma + 8 * (t % kSX), (t / kSX) & 1);
                    ready[2 * p + 1] = mbar_try_wait(bar_full + 8 * (t % kS), (t / kS) & 1);
                }
                bool ok = true;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int t = i + p;
                    if (ok && !ready[2 * p]) ok = mbar_wait(bar_tma + 8 * (t % kSX), (t / kSX) & 1);
                    if (ok && !ready[2 * p + 1]) ok = mbar_wait(bar_full + 8 * (t % kS), (t / kS) & 1);
                    if (!ok) break;
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    issue_stage(t);
                }
                if (!ok) break;
            }
            mma_commit(bar_done);
            (void)mbar_wait(bar_done, 0);
        }
    }

    griddep_launch_dependents();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(S::kTmemCols)
                     : "memory");
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// x [M, K] bf16 row-major (the M <= NB rows of this chunk) as a 2-D tensor
// (k, m) with a box of 64 k (128 bytes) x `rows` rows, swizzled by the TMA
// into the MMA's K-major 128-byte-swizzle layout.  Box rows m >= M lie outside
// the tensor and are filled with zeros.
bool make_x_map(CUtensorMap* map, const uint16_t* x, int M, int K, int rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {kSwK, static_cast<cuuint32_t>(rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KB, int NB, int LL>
int launch_tc_chunks(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M, int K, int N,
                     uint32_t lmask, uint16_t* out, cudaStream_t stream) {
    static std::atomic<unsigned long long> opted{0};
    if (!smem_opt_in(gemm_tc_kernel<KB, NB, LL>, TcShape<NB>::kSmemBytes, opted)) return -5;
    const int grid = (N + kTcRows - 1) / kTcRows;
    for (int m = 0; m < M; m += NB) {
        const int m0 = (M > NB && m + NB > M) ? M - NB : m;
        const int mc = (M - m0) < NB ? (M - m0) : NB;
        CUtensorMap map;
        if (!make_x_map(&map, x + static_cast<size_t>(m0) * K, mc, K, tc_box_rows(mc, NB))) return -5;
        const cudaError_t e = launch_programmatic(gemm_tc_kernel<KB, NB, LL>, static_cast<unsigned>(grid),
                                                  static_cast<unsigned>(kTcThreads), TcShape<NB>::kSmemBytes,
                                                  stream, codes, scales, out + static_cast<size_t>(m0) * N, mc, K,
                                                  N, K / 32 * KB, lmask, map);
        if (e != cudaSuccess) return -5;
    }
    return 0;
}


// codes [N, row_words] uint32 as a 2-D tensor (word, row) with a box of 32
// words (128 bytes) x 128 rows, 128-byte swizzled; rows past N and words past
// the row's end are filled with zeros.
bool make_code_map(CUtensorMap* map, const uint32_t* codes, int N, int row_words) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_words), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_words) * 4};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kCodeTileWords), static_cast<cuuint32_t>(kTcRows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(codes), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KB, int NB, bool TAB, int LL>
int launch_tca_chunks(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M, int K, int N,
                      uint32_t lmask, uint16_t* out, cudaStream_t stream) {
    using S = TcaShape<NB, TAB, KB>;
    static std::atomic<unsigned long long> opted{0};
    if (!smem_opt_in(gemm_tca_kernel<KB, NB, TAB, LL>, S::kSmemBytes, opted)) return -5;
    const int grid = (N + kTcRows - 1) / kTcRows;
    CUtensorMap cmap;
    if (!make_code_map(&cmap, codes, N, K / 32 * KB)) return -5;
    for (int m = 0; m < M; m += NB) {
        const int m0 = (M > NB && m + NB > M) ? M - NB : m;
        const int mc = (M - m0) < NB ? (M - m0) : NB;
        CUtensorMap map;
        if (!make_x_map(&map, x + static_cast<size_t>(m0) * K, mc, K, tc_box_rows(mc, NB))) return -5;
        const cudaError_t e = launch_programmatic(gemm_tca_kernel<KB, NB, TAB, LL>, static_cast<unsigned>(grid),
                                                  static_cast<unsigned>(kTcThreads), S::kSmemBytes, stream, scales,
                                                  out + static_cast<size_t>(m0) * N, mc, K, N, lmask, map, cmap);
        if (e != cudaSuccess) return -5;
    }
    return 0;
}

// LL = kL (k in {2, 3, 4}, 12-bit windows: the quotient table at NB = 64) or 0
// (the window width from L at run time, the computed quotient).
template <int KB, int LL>
int launch_tca_instance(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M, int K, int N,
                        int L, uint16_t* out, cudaStream_t stream) {
    const uint32_t lmask = (1u << L) - 1u;
    if (M <= 64) return launch_tca_chunks<KB, 64, LL == kL, LL>(x, codes, scales, M, K, N, lmask, out, stream);
    if (M <= 128) return launch_tca_chunks<KB, 128, false, LL>(x, codes, scales, M, K, N, lmask, out, stream);
    return launch_tca_chunks<KB, 256, false, LL>(x, codes, scales, M, K, N, lmask, out, stream);
}

// The MMA's N follows M: 64 for M <= 64, 128 for M <= 128, else 256.  Above
// 256 rows the launches take 256-row chunks (each decodes the weights again;
// they are programmatically chained on the stream), and the last chunk is
// moved back to end at row M, so it is full and overlaps the one before: the
// overlapping rows are computed again with identical bits (each output is its
// own dot product) and written again after the earlier launch (stream order).
template <int KB, int LL>
int launch_tc_instance(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M, int K, int N,
                       int L, uint16_t* out, cudaStream_t stream) {
    const uint32_t lmask = (1u << L) - 1u;
    if (M <= 64) return launch_tc_chunks<KB, 64, LL>(x, codes, scales, M, K, N, lmask, out, stream);
    if (M <= 128) return launch_tc_chunks<KB, 128, LL>(x, codes, scales, M, K, N, lmask, out, stream);
    return launch_tc_chunks<KB, 256, LL>(x, codes, scales, M, K, N, lmask, out, stream);
}

}  // namespace

int launch_gemm_tc(const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int M, int K, int N, int k,
                   int L, uint16_t* out, cudaStream_t stream) {
    if (fast_geometry(k, L)) {
        switch (k) {
            case 2: return launch_tca_instance<2, kL>(x, codes, scales, M, K, N, L, out, stream);
            case 3: return launch_tca_instance<3, kL>(x, codes, scales, M, K, N, L, out, stream);
            default: return launch_tca_instance<4, kL>(x, codes, scales, M, K, N, L, out, stream);
        }
    }
    switch (k) {
        // k = 1: a block's 8 words are a quarter of a code box, and the
        // shared-memory-A kernel measured faster (30.8 against 31.9 us at M = 64)
        case 1: return launch_tc_instance<1, 0>(x, codes, scales, M, K, N, L, out, stream);
        case 2: return launch_tca_instance<2, 0>(x, codes, scales, M, K, N, L, out, stream);
        case 3: return launch_tca_instance<3, 0>(x, codes, scales, M, K, N, L, out, stream);
        case 4: return launch_tca_instance<4, 0>(x, codes, scales, M, K, N, L, out, stream);
        case 5: return launch_tca_instance<5, 0>(x, codes, scales, M, K, N, L, out, stream);
        case 6: return launch_tca_instance<6, 0>(x, codes, scales, M, K, N, L, out, stream);
        case 7: return launch_tca_instance<7, 0>(x, codes, scales, M, K, N, L, out, stream);
        case 8: return launch_tca_instance<8, 0>(x, codes, scales, M, K, N, L, out, stream);
        default: return -3;
    }
}

namespace {

// One thread waits on an mbarrier that nothing ever arrives on: the wait runs
// out after limit_ns, sets the error word and the kernel returns.  It checks
// the reporting path of the product's bounded waits without a hang or fault.
__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    (void)mbar_wait_for(b, 0, limit_ns);
}

}  // namespace

int launch_wait_selftest(cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(50000000ull);   // 50 ms
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

int tc_take_device_error(unsigned int* flags) {
    unsigned int v = 0u;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v)) != cudaSuccess) return -5;
    if (v != 0u) {
        const unsigned int zero = 0u;
        if (cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(zero)) != cudaSuccess) return -5;
    }
    *flags = v;
    return 0;
}

}  // namespace trellis
