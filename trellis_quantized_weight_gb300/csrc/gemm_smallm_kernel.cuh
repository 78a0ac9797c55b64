// Fused decode-and-multiply for 1 <= M <= 16 on the CUDA cores (sm_103a).
//
// What it computes: out[m, n] = bf16( sum_k w[n, k] * x[m, k] ), with w the
// decoded bf16 weights, products and sums in fp32 (the wide-prefill kernel on
// the page "mlx-bun 0.2.0 -> 0.4.0", trellis-wide-prefill.ts: decode each row
// once and share it across every activation row).
//
// Mapping (GB300-first, not the page's simdgroup layout):
//  * A warp's 32 lanes are 4 row slots x 8 groups: the lane decodes group g
//    (32 weights) of the rows held by its slot q.  The 8 lanes of a slot read
//    one row's 32*k-byte block together, so a warp-wide code load touches 4
//    cache lines, and the lookahead word of group g (the first word of group
//    g-1, or word 0 of the block for g = 0) arrives by one shuffle.  Lane order
//    is a per-shape choice: slot-major (l = 8q + g) or group-major
//    (l = 4g + q: the 4 slots reading the same activations are adjacent, which
//    serves a 16-byte shared load in 2 wavefronts instead of 4).  Codes are
//    always loaded slot-major, each quarter-warp reading one row's contiguous
//    block; in group-major order k + 1 shuffles per row and block then hand
//    each lane its group's words and the lookahead word.
//  * Each lane holds R rows (slot q: rows q, q+4, ...), so a warp's tile is
//    4*R rows and every activation value a lane loads from shared memory feeds
//    R rows and both weights of an f32x2 FMA.
//  * WARPS tiles form a "tile-group".  Work units are (tile-group, 256-weight
//    block) pairs, numbered tile-group-major, and CTA c takes a contiguous
//    range of floor(U/P) units, one more if c < U mod P: every SM gets the
//    same number of weights, to one unit, whatever N and K are (stream-K
//    split).  All warps of a CTA walk the same
//    blocks in step, so the CTA stages x UB blocks ahead, as fp32, through a
//    2*UB-slot shared-memory ring ([group][m][32 k], groups padded by 16 bytes
//    so the 8 groups of a load hit 8 different bank quads), with one CTA
//    barrier per UB blocks.
//  * At the end of a row segment the 8 lanes of a slot add their per-group
//    sums by butterfly shuffles (lane distances 4, 8, 16).  A row whose K-range is split over several
//    CTAs writes fp32 partial sums to the workspace as soon as its segment
//    ends; only a CTA's first and last segments can be split, and both take
//    their per-tile tickets after the CTA's last unit (one atomic instruction
//    for the two), so the loop never waits on a fence or an atomic.  The last
//    CTA to take a tile's ticket adds the partials in CTA order, rounds to
//    bf16, stores and resets the counter; partials are laid out [m][r][slot],
//    so its loads and stores run along each output row's 4R columns.  The sum
//    order is fixed: identical inputs give identical bits.  No CTA ever waits
//    on another.
//  * Decode per weight: funnel shift + mask, hash IMAD, then either the dp4a
//    byte sum into a float and the two-op quotient (trellis_device.cuh), or one
//    dp4a that turns the hash into the address of the quotient in a per-lane
//    shared-memory table (one conflict-free load).  Then a packed f32x2 scale
//    multiply, a bf16 round that keeps fp32 format, and the packed f32x2 FMAs
//    of the multiply: either MM per weight pair and row (two k at once, x
//    staged as [group][m][k]), or, for the shapes marked MP, MM/2 per weight
//    and row (two activation rows at once with the weight in both halves,
//    which the FMA takes from one register; an odd MM's last row by a scalar
//    FMA; x staged as [group][k][m]): half the fp32 sums a lane holds.
#pragma once

#include <cstdint>
#include <type_traits>

#include "kernels.h"
#include "trellis_device.cuh"

namespace trellis {

struct SmallMPlan {
    int M, K, N;
    int nblocks;        // 256-weight blocks per row (K / 256)
    int row_words;      // K * k / 32
    int ntg;            // tile-groups
    int P;              // CTAs
    int U;              // units = ntg * nblocks (below 2^31: N*K/256 is)
    int base, rem;      // CTA c takes base + (c < rem) units, c*base + min(c, rem) first
    FastDiv div_base1;  // division by base + 1
    FastDiv div_base;   // division by base
    // Two weight matrices sharing x (gate and up projections): virtual rows
    // [0, npad) are matrix 0 (the kernel's codes, scales, out), [npad, 2*npad)
    // matrix 1; npad is N rounded up to whole tile-groups, 0 for one matrix.
    int npad;
    const uint32_t* codes2;
    const uint16_t* scales2;
    uint16_t* out2;
    float* partials;    // workspace: [P][2][WARPS][R*M*4] fp32
    uint32_t* counters; // workspace: [ntg * WARPS]
    uint32_t lmask;     // 2^L - 1: the window mask of kernels built for a run-time L
#ifdef TRELLIS_TRACE
    unsigned long long* trace;   // trace build only: phase stamps (see trace_stamp)
    size_t trace_words;
#endif
};

// Trace build only (-DTRELLIS_TRACE; the shipped library is built without it):
// clock64 stamps of the kernel's phases.  CTA c owns kTraceCtaWords words from
// c * kTraceCtaWords: [0] SM id, [1] entry, [2] thread 0 leaving the loop,
// [3] units; warp w's record of 8 words at 8 + 8w: [0] leaving the loop,
// [1] tickets answered, [2] the reduction's partial sums loaded and added,
// [3] done, [4] flags (bit 0/1: split first/last segment, bit 2: in-loop
// ticket, bit 3/4: this warp reduced that tile).  Writes past the attached
// buffer are dropped.
#ifdef TRELLIS_TRACE
constexpr int kTraceCtaWords = 8 + 8 * 16;
__device__ __forceinline__ unsigned long long trace_clock() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void trace_stamp(const SmallMPlan& p, int c, int idx, unsigned long long v) {
    const size_t i = static_cast<size_t>(c) * kTraceCtaWords + idx;
    if (p.trace != nullptr && i < p.trace_words) p.trace[i] = v;
}
#endif

// Compile-time shape of one instantiation.
//   R      rows per lane (a warp's tile is 4*R rows)
//   WARPS  warps per CTA (= tiles per tile-group)
//   LUT    decode the quotient through a shared-memory table instead of the
//          two-part reciprocal multiply (same bits either way)
//   OCC    CTAs per SM
//   UB     blocks staged per CTA barrier
//   GM     group-major lane order (see the mapping notes above)
//   ET     early tickets: a split segment that ends before the CTA's last
//          unit takes its ticket inside the loop, and the segment that runs
//          to the last unit skips its ticket when the counter it read at its
//          start shows every other contributor done.  Pays when every CTA's
//          range spans a tile-group boundary (each split tile then has two
//          contributors, one finishing early); the in-loop fence costs more
//          than it saves otherwise.
//   TWO    two weight matrices sharing x (gate and up); single-matrix kernels
//          carry none of the row mapping
template <int MM_, int R_, int WARPS_, bool LUT_, int OCC_ = 1, int UB_ = 2, bool GM_ = false, bool ET_ = false,
          bool TWO_ = false, bool MP_ = false>
struct SmallMCfg {
    static constexpr int MM = MM_;
    static constexpr int R = R_;
    static constexpr int WARPS = WARPS_;
    static constexpr bool LUT = LUT_;
    static constexpr int OCC = OCC_;                              // CTAs per SM
    // MP: each f32x2 FMA takes a pair of activation rows (m, m+1) and one
    // weight in both halves; else a pair of k for one activation row
    static constexpr bool MP = MP_;
    static constexpr int MMP = MP ? (MM + 1) / 2 * 2 : MM;        // activation rows staged (even for MP)
    static constexpr int XG = 32 * MMP + 4;                       // floats per staged (block, group)
    static constexpr int XS_UNIT = 8 * XG;                        // floats of staged x per block
    static constexpr int TABLE_BYTES = LUT ? kQuotientTableBytes : 0;
    static constexpr int ROWS_PER_TILE = 4 * R;
    static constexpr int NT = WARPS * 32;
    static constexpr int XV = MM * 32;                            // 8-element x vectors per block
    static constexpr bool ODD = MP && (MM & 1);                   // the last activation row alone
    static constexpr int NACC = MP ? MM / 2 : MM;                 // f32x2 sums per row a lane holds
    static constexpr int XPT = (XV + NT - 1) / NT;                // x vectors staged per thread per block
    static constexpr int UB = UB_;                                // blocks per CTA barrier
    static constexpr int RING = 2 * UB;                           // x ring slots
    static constexpr size_t SMEM_BYTES = TABLE_BYTES + RING * XS_UNIT * sizeof(float);
    static constexpr bool GM = GM_;
    static constexpr bool ET = ET_;
    static constexpr bool TWO = TWO_;
    static constexpr int GROUP_STRIDE = GM ? 4 : 1;  // lane distance between groups of a slot
    // Split-K reduction form: 2 = a lane takes pairs of adjacent columns and
    // loads 4 contributors a round; 1 = single columns, 4 a round; 0 = single
    // columns, 8 a round.  The reduction is inlined into the kernel and moves
    // the register allocation of its loop, so the form is chosen per shape by
    // timing (single-matrix kernels; gate/up keeps form 0).
    static constexpr int RED = (TWO || MM == 1) ? 0 : ((MM == 11 || MM == 15) ? 1 : 2);
};

// The shape used by the library for each M, chosen by timing back-to-back
// calls of the M = 1, 5, 8 and 15 workloads on GB300 over R, WARPS, UB, LUT and
// CTAs per SM (M in between takes its neighbours' shape).  With k-pairs (now
// M = 1, 2 only, KWARPS) M = 11 took 8 warps: at 12 its registers (168 a
// thread) spilled, and 8 measured 7-12% faster; M = 9 and 10 measured the
// same or faster at 12.  With activation-row pairs every M >= 11 fits 12.
template <int MM>
struct SmallMDefault {
    // Pairs of activation rows per f32x2 FMA (MP) from M = 3, an odd M's last
    // row on its own (a scalar FMA): half the sums a lane holds, so more warps
    // fit.  A/B on one GB300 (K = 5120, N = 17408; k = 2 for M = 5, 6, k = 3
    // for M = 7 .. 11, else k = 4), us: M = 3 37.3 -> 35.8, 4 40.4 -> 37.7,
    // 5 42.8 -> 41.2, 6 47.3 -> 43.8, 7 52.3 -> 50.0, 8 54.5 -> 50.3,
    // 9 59.6 -> 57.2, 10 64.7 -> 58.8 (16 warps); 11 69.5 -> 67.9, 12 69.6 ->
    // 64.2, 13 72.1 -> 69.5, 15 78.7 -> 76.7, 16 82.0 -> 79.4 (12 warps; 16
    // spilled and measured slower at M = 11, 12); 14 77.2 -> 72.7 (8 warps,
    // then 12 once the split-K tail got shorter: k = 4 72.9 -> 70.3, k = 3
    // 78.0 -> 74.2, k = 2 71.5 -> 69.3).
    // M = 1, 2 keep k-pairs (a pair of rows would leave half of each FMA idle).
    static constexpr bool MPD = MM >= 3;
    static constexpr int KWARPS = (MM <= 2) ? 16 : (MM <= 10 ? 12 : 8);   // with k-pairs
    static constexpr int WARPS = MPD ? (MM <= 10 ? 16 : 12) : KWARPS;
    static constexpr int UB = (MM <= 2) ? 3 : (MM <= 11) ? 4 : 3;
    static constexpr bool GM = MM >= 6;   // activation traffic matters more than the shuffles
    // early tickets (8 warps only) measured slower at 12 warps (M = 12 64.3
    // -> 63.1 us without, 13 69.6 -> 68.7, 15 76.7 -> 75.7, 16 79.5 -> 78.9);
    // no default shape runs 8 warps any more
    static constexpr bool ET = MM >= 12 && WARPS == 8;
    using type = SmallMCfg<MM, 3, WARPS, true, 1, UB, GM, ET, false, MPD>;
    // gate and up: activation-row pairs as above (M = 5 94.2 -> 85.1 us,
    // M = 8 117.3 -> 103.3 at K = 5120, N = 17408 against k-pairs at 12 warps,
    // measured with both on a slower build; M = 12 141.4 -> 123.8, M = 15
    // 158.0 -> 147.1 against k-pairs at 8 warps with early tickets, once the
    // split-K tail got shorter)
    using two = SmallMCfg<MM, 3, WARPS, true, 1, UB, GM, false, true, MPD>;
    // any other (k, L): the quotient table only holds the byte sums that
    // 12-bit windows reach, so these compute the quotient, which needs more
    // registers.  With activation-row pairs (from M = 3): 16 warps up to
    // M = 10, 12 above; with k-pairs (M = 1, 2) 16.  A/B on one GB300 at
    // K = 5120, N = 17408 against k-pairs at 8 warps (2 rows a lane for M = 15,
    // k = 8 and M = 16, k = 4, 6, 7, where 3 spilled heavily), us: M = 8 k = 3
    // L = 16 59.5 -> 55.4, M = 8 k = 8 L = 16 62.5 -> 60.6, M = 12 k = 3 L = 16
    // 74.6 -> 70.7, M = 15 k = 4 L = 16 85.7 -> 80.7, M = 15 k = 8 L = 16
    // 90.5 -> 85.6, M = 5 k = 5 L = 20 49.2 -> 49.9.  At k = 8 the 16-warp
    // shapes of M = 6 .. 10 spill 116-286 bytes and 12 warps none: M = 8
    // 59.6 -> 55.7 us (at M = 15, 8 warps instead of 12 measured 84.9 -> 86.8).
    static constexpr int GWARPS = MPD ? (MM <= 10 ? 16 : 12) : 16;
    template <int KB>
    using general = SmallMCfg<MM, 3, (KB == 8 && MM >= 6 && MM <= 10) ? 12 : GWARPS, false, 1, UB, GM, false,
                              false, MPD>;
    static_assert(type::SMEM_BYTES <= 232448, "shared memory per CTA exceeds 227 KB");
};

// The matrix a tile-group's virtual rows belong to: its codes, scales and
// output, and the virtual row of its first row.
struct RowSrc {
    const uint32_t* codes;
    const uint16_t* scales;
    uint16_t* out;
    int first;
};
template <class C>
__device__ __forceinline__ RowSrc row_source(const SmallMPlan& p, const uint32_t* codes, const uint16_t* scales,
                                             uint16_t* out, int row0) {
    if constexpr (C::TWO) {
        if (row0 >= p.npad) return RowSrc{p.codes2, p.scales2, p.out2, p.npad};
    }
    return RowSrc{codes, scales, out, 0};
}

__device__ __forceinline__ int unit_begin(int c, const SmallMPlan& p) {
    return c * p.base + (c < p.rem ? c : p.rem);
}

__device__ __forceinline__ int cta_of_unit(int u, const SmallMPlan& p) {
    const int big = p.rem * (p.base + 1);   // units of the CTAs that take base + 1
    return u < big ? static_cast<int>(p.div_base1.div(static_cast<uint32_t>(u)))
                   : p.rem + static_cast<int>(p.div_base.div(static_cast<uint32_t>(u - big)));
}

// A tile's ticket: add 1 to its counter at GPU scope with release semantics
// (the warp's partial-sum stores, ordered before it by a warp barrier, become
// visible first) and acquire semantics (the last contributor's later loads of
// the other CTAs' partial sums see them).  Returns the previous count.
__device__ __forceinline__ uint32_t take_ticket(uint32_t* counter) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    return old;
}

// Release/acquire fence at GPU scope.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// A ticket taken inside the loop: a relaxed add after a release fence, so no
// later load waits for its reply (the count is only read after the loop).
__device__ __forceinline__ uint32_t take_ticket_relaxed(uint32_t* counter) {
    uint32_t old;
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    return old;
}

// A counter read without ordering, issued where written; its value is used
// after the loop, behind an acquire fence.
__device__ __forceinline__ uint32_t load_relaxed(const uint32_t* counter) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    return v;
}

template <int KB, int R>
__device__ __forceinline__ void load_block_group(const uint32_t* const (&rp)[R], const bool (&ok)[R], int b,
                                                 int g, uint32_t (&w)[R][KB]) {
    constexpr int WPB = kGroupsPerBlock * KB;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (ok[r]) {
            // volatile: issued where written (a block ahead of its use), never
            // sunk toward the use to shorten register lifetimes
            // (a group starts at word (7 - g) * KB of a 32-byte aligned block:
            // 16-byte aligned for KB % 4 == 0, 8-byte aligned for even KB)
            const uint32_t* p = rp[r] + b * WPB + (kGroupsPerBlock - 1 - g) * KB;
            if constexpr (KB % 4 == 0) {
#pragma unroll
                for (int i = 0; i < KB; i += 4)
                    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[r][i]), "=r"(w[r][i + 1]), "=r"(w[r][i + 2]), "=r"(w[r][i + 3])
                                 : "l"(p + i));
            } else if constexpr (KB % 2 == 0) {
#pragma unroll
                for (int i = 0; i < KB; i += 2)
                    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(w[r][i]), "=r"(w[r][i + 1]) : "l"(p + i));
            } else {
#pragma unroll
                for (int i = 0; i < KB; ++i) asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(w[r][i]) : "l"(p + i));
            }
        } else {
#pragma unroll
            for (int i = 0; i < KB; ++i) w[r][i] = 0u;
        }
    }
}

// x of one 256-weight block, 8 bf16 (16 bytes) per load: vector i of the
// block is row m = i/32, columns 8*(i%32) .. +7 ...
template <class C>
__device__ __forceinline__ void x_block_load(const uint16_t* __restrict__ x, int K, int b, int tid,
                                             uint4 (&v)[C::XPT]) {
#pragma unroll
    for (int i = 0; i < C::XPT; ++i) {
        const int e = tid + i * C::NT;
        if (e < C::XV) {
            const int m = e >> 5, c8 = e & 31;
            v[i] = __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(m) * K + b * 256 + c8 * 8));
        }
    }
}

// ... stored as fp32 in the layout [group][m][32 k] of one ring slot (the two
// floats of a k-pair are adjacent, ready for f32x2 FMAs).
template <class C>
__device__ __forceinline__ void x_block_store(float* slot, int tid, const uint4 (&v)[C::XPT]) {
#pragma unroll
    for (int i = 0; i < C::XPT; ++i) {
        const int e = tid + i * C::NT;
        if (e < C::XV) {
            const int m = e >> 5, c8 = e & 31;
            const uint32_t u[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            float f[8];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                f[2 * h] = __uint_as_float(u[h] << 16);
                f[2 * h + 1] = __uint_as_float(u[h] & 0xFFFF0000u);
            }
            if constexpr (C::MP) {
                // [group][k][m]: the activation rows of one k are adjacent
                float* dst = slot + (c8 >> 2) * C::XG + ((c8 & 3) * 8) * C::MMP + m;
#pragma unroll
                for (int j = 0; j < 8; ++j) dst[j * C::MMP] = f[j];
            } else {
                float* dst = slot + (c8 >> 2) * C::XG + m * 32 + (c8 & 3) * 8;
                *reinterpret_cast<float4*>(dst) = make_float4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<float4*>(dst + 4) = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
    }
}

// The CTAs that contribute to a tile-group, packed in one word: the first
// (bits 0-14) and the last (bits 15-29) contributing CTA, and bit 30 set when
// the first one keeps its partial sums in slot 1 (its range starts before the
// tile-group: every CTA after the first starts inside the tile-group, so the
// tile-group is its first, slot 0).  Computed when a segment starts, off the
// critical path at the end of the kernel.
__device__ __forceinline__ uint32_t contributors_info(int tg, const SmallMPlan& p) {
    const int tg_u0 = tg * p.nblocks;
    const int c_first = cta_of_unit(tg_u0, p);
    const int c_last = cta_of_unit(tg_u0 + p.nblocks - 1, p);
    const uint32_t slot1 = unit_begin(c_first, p) < tg_u0 ? 1u : 0u;
    return static_cast<uint32_t>(c_first) | (static_cast<uint32_t>(c_last) << 15) | (slot1 << 30);
}
__device__ __forceinline__ int info_first(uint32_t info) { return static_cast<int>(info & 0x7FFFu); }
__device__ __forceinline__ int info_last(uint32_t info) { return static_cast<int>((info >> 15) & 0x7FFFu); }
__device__ __forceinline__ int info_slot(uint32_t info) { return static_cast<int>(info >> 30); }

// Adds the partial sums of up to two split tiles of this warp (tile-groups
// tgs[t] where use[t], contributors infos[t]) in CTA order, rounds to bf16,
// stores, and resets the tiles' counters.  All loads of a round, for both
// tiles, are issued before the first add, so the reduction costs one round
// trip per 8 contributors.
template <class C>
__device__ __forceinline__ void reduce_split_tiles(const SmallMPlan& p, const bool (&use)[2], const int (&tgs)[2],
                                                   const uint32_t (&infos)[2], int warp, int lane,
                                                   uint16_t* __restrict__ out, int c) {
    constexpr int MM = C::MM, WARPS = C::WARPS;
    constexpr int E = C::R * MM * 4;                  // sums of one warp's tile
    constexpr int V = C::RED == 2 ? 2 : 1;            // adjacent columns a lane takes at once
    constexpr int EV = E / V;                         // ... as that many units (E is a multiple of 4)
    constexpr int EP = (EV + 31) / 32;                // units per lane
    constexpr int CR = C::RED == 0 ? 8 : 4;           // contributors loaded per round
    using VT = typename std::conditional<V == 2, float2, float>::type;
    int c_first[2], c_last[2], cf_slot[2];
    int rounds = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        c_first[t] = use[t] ? info_first(infos[t]) : 1;
        c_last[t] = use[t] ? info_last(infos[t]) : 0;
        cf_slot[t] = use[t] ? info_slot(infos[t]) : 0;
        const int r = (c_last[t] - c_first[t] + CR) / CR;
        rounds = r > rounds ? r : rounds;
    }
    float sum[2][EP][V];
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int ep = 0; ep < EP; ++ep)
#pragma unroll
            for (int h = 0; h < V; ++h) sum[t][ep][h] = 0.0f;
    for (int rd = 0; rd < rounds; ++rd) {
        VT part[2][EP][CR];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int i = 0; i < CR; ++i) {
                const int cc = c_first[t] + CR * rd + i;
                const int cs = (cc == c_first[t]) ? cf_slot[t] : 0;
                const VT* src = reinterpret_cast<const VT*>(
                    p.partials + ((static_cast<size_t>(cc) * 2 + cs) * WARPS + warp) * E);
#pragma unroll
                for (int ep = 0; ep < EP; ++ep) {
                    const int ev = lane + 32 * ep;
                    part[t][ep][i] = (cc <= c_last[t] && ev < EV) ? __ldcg(src + ev) : VT{};
                }
            }
        // contributors in CTA order, so the sums are the same whatever the form
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int i = 0; i < CR; ++i)
                if (c_first[t] + CR * rd + i <= c_last[t])
#pragma unroll
                    for (int ep = 0; ep < EP; ++ep) {
                        if constexpr (V == 2) {
                            sum[t][ep][0] = __fadd_rn(sum[t][ep][0], part[t][ep][i].x);
                            sum[t][ep][1] = __fadd_rn(sum[t][ep][1], part[t][ep][i].y);
                        } else {
                            sum[t][ep][0] = __fadd_rn(sum[t][ep][0], part[t][ep][i]);
                        }
                    }
    }
#ifdef TRELLIS_TRACE
    {
        // stamped once every sum is complete (the clock read depends on them)
        float z = 0.0f;
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int ep = 0; ep < EP; ++ep)
#pragma unroll
                for (int h = 0; h < V; ++h) z += sum[t][ep][h];
        unsigned long long t;
        asm volatile("mov.u64 %0, %%clock64;" : "=l"(t) : "f"(z));
        if (lane == 0) trace_stamp(p, c, 8 + 8 * warp + 2, t);
    }
#endif
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (!use[t]) continue;
        const int tile = tgs[t] * WARPS + warp;
        const int row0 = tile * C::ROWS_PER_TILE;
        const RowSrc rs = row_source<C>(p, nullptr, nullptr, out, row0);
#pragma unroll
        for (int ep = 0; ep < EP; ++ep) {
            const int ev = lane + 32 * ep;
            if (ev < EV) {
                // e = m * 4R + (4r + q): the tile's 4R columns of row m are
                // adjacent (a pair never crosses a row: 4R is even)
                const int e = V * ev;
                const int m = e / (4 * C::R), col = e - m * (4 * C::R);
                const int n = row0 - rs.first + col;
                uint16_t* dst = rs.out + static_cast<size_t>(m) * p.N + n;
                if constexpr (V == 2) {
                    if (n + 1 < p.N && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
                        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(sum[t][ep][0], sum[t][ep][1]);
                    } else {
                        if (n < p.N) dst[0] = bf16_bits_rn(sum[t][ep][0]);
                        if (n + 1 < p.N) dst[1] = bf16_bits_rn(sum[t][ep][1]);
                    }
                } else {
                    if (n < p.N) *dst = bf16_bits_rn(sum[t][ep][0]);
                }
            }
        }
        if (lane == 0) p.counters[tile] = 0u;
    }
}

// LL: the window width when fixed at compile time (12), or 0 for the run-time
// width of p.lmask.
template <class C, int KB, int LL>
__global__ void __launch_bounds__(C::WARPS * 32, C::OCC)
gemm_smallm_kernel(const uint16_t* __restrict__ x, const uint32_t* __restrict__ codes,
                   const uint16_t* __restrict__ scales, uint16_t* __restrict__ out, SmallMPlan p) {
    constexpr int MM = C::MM, R = C::R, WARPS = C::WARPS, XG = C::XG, XS_UNIT = C::XS_UNIT;
    constexpr int NT = C::NT;
    constexpr int UB = C::UB;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* xs = reinterpret_cast<float*>(smem_raw + C::TABLE_BYTES);   // C::RING slots of XS_UNIT floats

    const int c = blockIdx.x;
#ifdef TRELLIS_TRACE
    if (threadIdx.x == 0) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        trace_stamp(p, c, 0, smid);
        trace_stamp(p, c, 1, trace_clock());
    }
#endif
    const int u0 = unit_begin(c, p);
    const int u1 = unit_begin(c + 1, p);
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = C::GM ? lane >> 2 : lane & 7;
    const int slot = C::GM ? lane & 3 : lane >> 3;
    // the lane of the same slot holding group g - 1 (mod 8)
    const int src_lane = (g == 0) ? lane + 7 * C::GROUP_STRIDE : lane - C::GROUP_STRIDE;
    // Code loads are always slot-major (each quarter-warp reads one row's
    // contiguous block): this lane loads group lg of the rows of slot lslot.
    // In group-major order the words then move to their lane by shuffles.
    const int lslot = lane >> 3, lg = lane & 7;
    const int first_tg = u0 / p.nblocks;

    // (tile-group, block) of the current unit, advanced incrementally: no
    // divisions inside the loop
    const int nunits = u1 - u0;
    int utg = first_tg;
    int b = u0 - first_tg * p.nblocks;

    // Per-segment state of this warp's tile.
    bool ok[R];
    float2 s2[R];
    const uint32_t* rp[R];
    constexpr int NACC = C::NACC;
    float2 acc[R][NACC];
    float acc1[R];   // the last activation row when MM is odd (MP)
    uint32_t cw[R][KB];
    int tg = -1, row0 = 0, tile = 0, b_first = 0;
    bool live = false;
    // Scales of the next segment: requested, with its first block of codes,
    // during the current segment's last unit.
    float snext[R];
    // A segment starts at unit (utg, b).  Its first codes and scales are loaded
    // here, or were already requested one unit ahead (prefetched).
    uint32_t seg_info = 0;   // contributors of the current segment's tile-group
    auto begin_segment = [&](bool prefetched) {
        tg = utg;
        b_first = b;
        seg_info = contributors_info(tg, p);
        tile = tg * WARPS + warp;
        row0 = tile * C::ROWS_PER_TILE;
        const RowSrc rs = row_source<C>(p, codes, scales, out, row0);
        live = row0 - rs.first < p.N;   // whole tile beyond N: skipped by every CTA alike
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int n = row0 - rs.first + slot + 4 * r;    // this lane's row
            const int nl = row0 - rs.first + lslot + 4 * r;  // the row this lane loads codes for
            ok[r] = nl < p.N;
            float sr;
            if (prefetched)
                sr = snext[r];
            else
                sr = n < p.N ? bf16_bits_to_f32(__ldg(rs.scales + n)) : 0.0f;
            s2[r] = make_float2(sr, sr);
            rp[r] = rs.codes + static_cast<size_t>(ok[r] ? nl : 0) * p.row_words;
#pragma unroll
            for (int m = 0; m < NACC; ++m) acc[r][m] = make_float2(0.0f, 0.0f);
            acc1[r] = 0.0f;
        }
        if (live && !prefetched) load_block_group<KB, R>(rp, ok, b, lg, cw);
    };

    // Shared-memory set-up first: under a programmatic launch it overlaps the
    // previous kernel's tail, together with L2 prefetches of the first unit's
    // codes and x (L2 is coherent, so these cannot observe stale data).
    // Nothing is loaded into registers or written before griddep_wait().  Then
    // the first segment's codes and the x of the first UB units (into ring
    // slots 0 .. UB-1).
    if (nunits > 0) {
        const int prow0 = (utg * WARPS + warp) * C::ROWS_PER_TILE;
        const RowSrc prs = row_source<C>(p, codes, scales, out, prow0);
        if (lg == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int n = prow0 - prs.first + lslot + 4 * r;
                if (n < p.N)
                    asm volatile("prefetch.global.L2 [%0];"
                                 :: "l"(prs.codes + static_cast<size_t>(n) * p.row_words + b * (kGroupsPerBlock * KB)));
            }
        }
        // x of the first unit: MM rows of 512 bytes, 4 lines each
        if (tid < MM * 4)
            asm volatile("prefetch.global.L2 [%0];"
                         :: "l"(x + static_cast<size_t>(tid >> 2) * p.K + b * 256 + (tid & 3) * 64));
    }
    if constexpr (C::LUT) build_quotient_table(reinterpret_cast<float*>(smem_raw), tid, NT);
    if constexpr (C::MP && C::MMP != MM) {
        // the padding activation row (m = M) of every ring slot stays zero
        for (int i = tid; i < C::RING * 8 * 32; i += NT) {
            const int slot_i = i >> 8, gk = i & 255;
            xs[slot_i * XS_UNIT + (gk >> 5) * XG + (gk & 31) * C::MMP + MM] = 0.0f;
        }
    }
    griddep_wait();
    if (nunits > 0) begin_segment(false);
    {
        uint4 xfirst[UB][C::XPT];
#pragma unroll
        for (int j = 0; j < UB; ++j)
            if (j < nunits) {
                int bj = b + j;
                while (bj >= p.nblocks) bj -= p.nblocks;
                x_block_load<C>(x, p.K, bj, tid, xfirst[j]);
            }
#pragma unroll
        for (int j = 0; j < UB; ++j)
            if (j < nunits) x_block_store<C>(xs + j * XS_UNIT, tid, xfirst[j]);
    }
    __syncthreads();
    const uint32_t lane_tbl = quotient_table_lane_address(smem_raw, lane);

    // x of the next UB units: loaded at the start of a phase of UB units,
    // stored to the ring (into the previous phase's slots) at its end, then
    // one CTA barrier.
    uint4 xnext[UB][C::XPT];
    // Split segments (at most two per CTA: its first and its last) publish
    // their partial sums at once.  Indexed by partial slot.
    //  * A split segment that ends before the CTA's last unit takes its ticket
    //    at the next phase end, just before the barrier (the count is read
    //    after the loop).
    //  * The segment that runs to the CTA's last unit reads its tile's counter
    //    when that unit starts.  If every other contributor had already taken
    //    its ticket, this CTA is the last one by construction: it takes no
    //    ticket and goes straight to the reduction after the loop.  Otherwise
    //    it takes its ticket after the loop.
    bool pend0 = false, pend1 = false;
    int ptg0 = 0, ptg1 = 0;
    uint32_t pinfo0 = 0, pinfo1 = 0;
    bool tk_due = false, tk_taken = false;   // slot 0's in-loop ticket
    uint32_t tk0 = 0;                        // its previous count (lane 0)
    uint32_t peek = 0xFFFFFFFFu;             // counter of the CTA's last segment when it started (lane 0)

    int ph = 0, rhalf = 0;   // position in the current phase of UB units; ring half it uses
    for (int rel = 0; rel < nunits; ++rel) {
        const int ring = rhalf * UB + ph;   // ring slot of this unit's x
        const bool seg_start = (rel == 0) || (b == 0);
        const bool seg_end = (rel + 1 == nunits) || (b + 1 == p.nblocks);
        const bool phase_start = ph == 0;
        const bool phase_end = ph == UB - 1 || rel + 1 == nunits;

        if (phase_start) {
#pragma unroll
            for (int j = 0; j < UB; ++j)
                if (rel + UB + j < nunits) {
                    int bj = b + UB + j;
                    while (bj >= p.nblocks) bj -= p.nblocks;
                    x_block_load<C>(x, p.K, bj, tid, xnext[j]);
                }
        }

        if (seg_start && rel > 0) begin_segment(true);
        // the last unit of a split segment: read its tile's counter (the other
        // contributors have had the whole kernel to take their tickets)
        if (C::ET && rel + 1 == nunits && live && !(b_first == 0 && b + 1 == p.nblocks) && lane == 0)
            peek = load_relaxed(p.counters + tile);

        if (live) {
            uint32_t nw[R][KB];
            if (!seg_end) {
                load_block_group<KB, R>(rp, ok, b + 1, lg, nw);
            } else if (rel + 1 < nunits) {
                // the next unit starts tile-group utg + 1 at block 0: request
                // its codes and scales now
                const int nrow0 = ((utg + 1) * WARPS + warp) * C::ROWS_PER_TILE;
                const RowSrc nrs = row_source<C>(p, codes, scales, out, nrow0);
                bool nok[R];
                const uint32_t* nrp[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int n = nrow0 - nrs.first + slot + 4 * r;
                    const int nl = nrow0 - nrs.first + lslot + 4 * r;
                    nok[r] = nl < p.N;
                    nrp[r] = nrs.codes + static_cast<size_t>(nok[r] ? nl : 0) * p.row_words;
                    snext[r] = n < p.N ? bf16_bits_to_f32(__ldg(nrs.scales + n)) : 0.0f;
                }
                load_block_group<KB, R>(nrp, nok, 0, lg, nw);
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int i = 0; i < KB; ++i) nw[r][i] = 0u;
            }
            uint32_t w[R][KB + 1];
            if constexpr (C::GM) {
                // group g of slot's row was loaded by lane 8*slot + g; the
                // lookahead is group g - 1's first word
                const int from = 8 * slot + g, from_prev = 8 * slot + ((g + 7) & 7);
#pragma unroll
                for (int r = 0; r < R; ++r) {
#pragma unroll
                    for (int i = 0; i < KB; ++i) w[r][i] = __shfl_sync(0xffffffffu, cw[r][i], from);
                    w[r][KB] = __shfl_sync(0xffffffffu, cw[r][0], from_prev);
                }
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r) {
#pragma unroll
                    for (int i = 0; i < KB; ++i) w[r][i] = cw[r][i];
                    w[r][KB] = __shfl_sync(0xffffffffu, cw[r][0], src_lane);
                }
            }
            const float* xq = xs + ring * XS_UNIT + g * XG;
            if constexpr (C::MP) {
#pragma unroll
                for (int pp = 0; pp < 16; ++pp) {
                    // weights of k-pair pp (k = 2pp, 2pp+1 of the group) for each row
                    float2 wv[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        float2 v;
                        if constexpr (C::LUT) {
                            static_assert(LL == kL, "the quotient table covers 12-bit windows only");
                            v.x = quotient_lookup(group_window<KB, LL>(w[r], 2 * pp), lane_tbl);
                            v.y = quotient_lookup(group_window<KB, LL>(w[r], 2 * pp + 1), lane_tbl);
                        } else {
                            v = window_value2(group_window<KB, LL>(w[r], 2 * pp, p.lmask),
                                              group_window<KB, LL>(w[r], 2 * pp + 1, p.lmask));
                        }
                        const float2 ws = __fmul2_rn(v, s2[r]);
                        wv[r] = make_float2(round_bf16_as_f32(ws.x), round_bf16_as_f32(ws.y));
                    }
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const float* xk = xq + (2 * pp + kk) * C::MMP;
#pragma unroll
                        for (int q = 0; q < C::MMP / 4; ++q) {
                            const float4 t = *reinterpret_cast<const float4*>(xk + 4 * q);
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                const float wk = kk ? wv[r].y : wv[r].x;
                                if (2 * q < NACC)
                                    acc[r][2 * q] =
                                        __ffma2_rn(make_float2(wk, wk), make_float2(t.x, t.y), acc[r][2 * q]);
                                else if (C::ODD && 4 * q == MM - 1)
                                    acc1[r] = __fmaf_rn(wk, t.x, acc1[r]);
                                if (2 * q + 1 < NACC)
                                    acc[r][2 * q + 1] =
                                        __ffma2_rn(make_float2(wk, wk), make_float2(t.z, t.w), acc[r][2 * q + 1]);
                                else if (C::ODD && 4 * q + 2 == MM - 1)
                                    acc1[r] = __fmaf_rn(wk, t.z, acc1[r]);
                            }
                        }
                        if constexpr (C::MMP % 4 != 0) {
                            const float2 t2 = *reinterpret_cast<const float2*>(xk + C::MMP - 2);
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                const float wk = kk ? wv[r].y : wv[r].x;
                                if constexpr (C::ODD)
                                    acc1[r] = __fmaf_rn(wk, t2.x, acc1[r]);
                                else
                                    acc[r][NACC - 1] = __ffma2_rn(make_float2(wk, wk), t2, acc[r][NACC - 1]);
                            }
                        }
                    }
                }
            } else {
    #pragma unroll
                for (int pq = 0; pq < 8; ++pq) {
                    // k-pairs 2pq and 2pq+1 of the group: x[m][4pq .. 4pq+3]
                    float2 xa[MM], xb[MM];
    #pragma unroll
                    for (int m = 0; m < MM; ++m) {
                        const float4 t = *reinterpret_cast<const float4*>(xq + m * 32 + 4 * pq);
                        xa[m] = make_float2(t.x, t.y);
                        xb[m] = make_float2(t.z, t.w);
                    }
    #pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int pp = 2 * pq + half;
    #pragma unroll
                        for (int r = 0; r < R; ++r) {
                            float2 v;
                            if constexpr (C::LUT) {
                                static_assert(LL == kL, "the quotient table covers 12-bit windows only");
                                v.x = quotient_lookup(group_window<KB, LL>(w[r], 2 * pp), lane_tbl);
                                v.y = quotient_lookup(group_window<KB, LL>(w[r], 2 * pp + 1), lane_tbl);
                            } else {
                                v = window_value2(group_window<KB, LL>(w[r], 2 * pp, p.lmask),
                                                  group_window<KB, LL>(w[r], 2 * pp + 1, p.lmask));
                            }
                            const float2 ws = __fmul2_rn(v, s2[r]);
                            const float2 wv = make_float2(round_bf16_as_f32(ws.x), round_bf16_as_f32(ws.y));
    #pragma unroll
                            for (int m = 0; m < MM; ++m)
                                acc[r][m] = __ffma2_rn(wv, half ? xb[m] : xa[m], acc[r][m]);
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int i = 0; i < KB; ++i) cw[r][i] = nw[r][i];
        }
        if constexpr (C::TWO) {
            // A tile wholly past N does no work, but with two matrices it can
            // end the first matrix's last tile-group and be followed, in the
            // same CTA, by the second matrix's first one: request that
            // segment's codes and scales here too (with one matrix a tile past
            // N only occurs in the last tile-group, where no segment follows).
            if (!live && seg_end && rel + 1 < nunits) {
                const int nrow0 = ((utg + 1) * WARPS + warp) * C::ROWS_PER_TILE;
                const RowSrc nrs = row_source<C>(p, codes, scales, out, nrow0);
                bool nok[R];
                const uint32_t* nrp[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int n = nrow0 - nrs.first + slot + 4 * r;
                    const int nl = nrow0 - nrs.first + lslot + 4 * r;
                    nok[r] = nl < p.N;
                    nrp[r] = nrs.codes + static_cast<size_t>(nok[r] ? nl : 0) * p.row_words;
                    snext[r] = n < p.N ? bf16_bits_to_f32(__ldg(nrs.scales + n)) : 0.0f;
                }
                load_block_group<KB, R>(nrp, nok, 0, lg, cw);
            }
        }

        if (live && seg_end) {
            // ---- per-row sums: k-pair halves, then the 8 groups of the slot ----
            // Transposing butterfly over the slot's 8 lanes: each step adds
            // the partner's half of the values and keeps half as many, so
            // after three steps lane g holds the complete sums of the NV/8
            // values starting at vbase (the same pairwise sums as a plain
            // butterfly, in a third of the shuffles).  Value i = r*MM + m.
            constexpr int NV = (R * MM + 7) / 8 * 8;
            float v[NV];
#pragma unroll
            for (int i = 0; i < NV; ++i)
                if constexpr (C::MP)
                    v[i] = (i < R * MM) ? ((C::ODD && i % MM == MM - 1) ? acc1[i / MM]
                                           : ((i % MM) & 1 ? acc[i / MM][(i % MM) >> 1].y
                                                           : acc[i / MM][(i % MM) >> 1].x))
                                        : 0.0f;
                else
                    v[i] = (i < R * MM) ? __fadd_rn(acc[i / MM][i % MM].x, acc[i / MM][i % MM].y) : 0.0f;
            int vbase = 0;
#pragma unroll
            for (int step = 0; step < 3; ++step) {
                const int h = NV >> (step + 1);              // values kept after this step
                const bool upper = (g >> step) & 1;         // this lane keeps the upper half
#pragma unroll
                for (int i = 0; i < h; ++i) {
                    const float lo = v[i], hi = v[i + h];
                    const float other = __shfl_xor_sync(0xffffffffu, upper ? lo : hi, C::GROUP_STRIDE << step);
                    v[i] = __fadd_rn(upper ? hi : lo, other);
                }
                vbase += upper ? h : 0;
            }

            if (b_first == 0 && b + 1 == p.nblocks) {
                // this CTA owns the whole K-range of the tile-group
                const RowSrc rs = row_source<C>(p, codes, scales, out, row0);
#pragma unroll
                for (int j = 0; j < NV / 8; ++j) {
                    const int i = vbase + j;
                    const int r = i / MM, m = i - r * MM;
                    const int n = row0 - rs.first + slot + 4 * r;
                    if (i < R * MM && n < p.N) rs.out[static_cast<size_t>(m) * p.N + n] = bf16_bits_rn(v[j]);
                }
            } else {
                // ---- split row: publish the partial now, take the ticket after the loop ----
                // value (r, m) of row slot q sits at [(m*R + r)*4 + q]: row m's 4R
                // columns of the tile are adjacent, for the reduction's loads and stores
                const int pslot = (tg == first_tg) ? 0 : 1;
                float* mine = p.partials + ((static_cast<size_t>(c) * 2 + pslot) * WARPS + warp) * (R * MM * 4);
                if constexpr (C::LUT) {
#pragma unroll
                    for (int j = 0; j < NV / 8; ++j) {
                        const int i = vbase + j;
                        if (i < R * MM) {
                            const int r = i / MM, m = i - r * MM;
                            mine[(m * R + r) * 4 + slot] = v[j];
                        }
                    }
                } else {
                    // the same positions with (r, m) stepped along j: fewer live
                    // registers, which the run-time-window kernels need (M = 15,
                    // k = 8, L = 16: 87.5 -> 85.8 us; the fast-geometry kernels
                    // measured slower with it)
                    int r = vbase / MM, m = vbase - r * MM;
#pragma unroll
                    for (int j = 0; j < NV / 8; ++j) {
                        if (vbase + j < R * MM) mine[(m * R + r) * 4 + slot] = v[j];
                        if (++m == MM) {
                            m = 0;
                            ++r;
                        }
                    }
                }
                if (pslot == 0) {
                    pend0 = true;
                    ptg0 = tg;
                    pinfo0 = seg_info;
                    tk_due = C::ET && rel + 1 < nunits;
                } else {
                    pend1 = true;
                    ptg1 = tg;
                    pinfo1 = seg_info;
                }
            }
        }

        if (phase_end) {
            // the next phase's units use the other half of the ring
            const int pbase = rel - ph;
#pragma unroll
            for (int j = 0; j < UB; ++j)
                if (pbase + UB + j < nunits) x_block_store<C>(xs + ((rhalf ^ 1) * UB + j) * XS_UNIT, tid, xnext[j]);
            if (tk_due) {
                __syncwarp();          // the slot lanes' partial-sum stores ...
                fence_acq_rel_gpu();   // ... are visible before the ticket
                if (lane == 0) tk0 = take_ticket_relaxed(p.counters + ptg0 * WARPS + warp);
                tk_due = false;
                tk_taken = true;
            }
            __syncthreads();
        }
        if (++b == p.nblocks) {
            b = 0;
            ++utg;
        }
        if (++ph == UB) {
            ph = 0;
            rhalf ^= 1;
        }
    }

    // the next grid on the stream may be scheduled as this CTA's SM frees up
    griddep_launch_dependents();
#ifdef TRELLIS_TRACE
    if (tid == 0) {
        trace_stamp(p, c, 2, trace_clock());
        trace_stamp(p, c, 3, static_cast<unsigned long long>(nunits));
    }
    if (lane == 0) {
        trace_stamp(p, c, 8 + 8 * warp, trace_clock());
        trace_stamp(p, c, 8 + 8 * warp + 1, 0);
        trace_stamp(p, c, 8 + 8 * warp + 2, 0);
        trace_stamp(p, c, 8 + 8 * warp + 4, 0);
    }
#endif

    // ---- the last contributor of a split tile reduces it ----
    if (pend0 || pend1) {
        // The split segment that ran to the CTA's last unit, if any: slot 1,
        // or slot 0 when it had no ticket in the loop.
        const bool has_last = pend1 || !tk_taken;
        const uint32_t lneed = pend1 ? static_cast<uint32_t>(info_last(pinfo1) - info_first(pinfo1))
                                     : static_cast<uint32_t>(info_last(pinfo0) - info_first(pinfo0));
        peek = __shfl_sync(0xffffffffu, peek, 0);
        const bool by_peek = C::ET && has_last && peek == lneed;   // every other contributor is done
        const bool skip0 = by_peek && !pend1;                      // slot 0 is that segment
        __syncwarp();   // the slot lanes' partial-sum stores are ordered before the tickets
        uint32_t e0 = 0, e1 = 0;
        // one atomic instruction for both tickets: lane 0 takes slot 0's,
        // lane 1 slot 1's (two instructions would each wait for the other)
        const bool tk_mine = lane == 0 ? (pend0 && !tk_taken && !skip0) : (lane == 1 && pend1 && !by_peek);
        uint32_t ev = 0;
        if (tk_mine) ev = take_ticket(p.counters + (lane == 0 ? ptg0 : ptg1) * WARPS + warp);
        e0 = __shfl_sync(0xffffffffu, ev, 0);
        e1 = __shfl_sync(0xffffffffu, ev, 1);
#ifdef TRELLIS_TRACE
        if (lane == 0) trace_stamp(p, c, 8 + 8 * warp + 1, trace_clock());
#endif
        const uint32_t t0 = __shfl_sync(0xffffffffu, tk0, 0);
        const uint32_t need0 = static_cast<uint32_t>(info_last(pinfo0) - info_first(pinfo0));
        const uint32_t need1 = static_cast<uint32_t>(info_last(pinfo1) - info_first(pinfo1));
        const bool use[2] = {pend0 && (tk_taken ? t0 == need0 : (skip0 || e0 == need0)),
                             pend1 && (by_peek || e1 == need1)};
        const int tgs[2] = {ptg0, ptg1};
        const uint32_t infos[2] = {pinfo0, pinfo1};
        if (use[0] || use[1]) {
            // A ticket taken here is an acq_rel atomic: its acquire, then the
            // warp barrier, order the other contributors' partial sums before
            // every lane's loads.  A count read relaxed (the in-loop ticket or
            // the peek) needs the acquire fence.
            if (by_peek || (use[0] && tk_taken))
                fence_acq_rel_gpu();
            __syncwarp();
            reduce_split_tiles<C>(p, use, tgs, infos, warp, lane, out, c);
        }
#ifdef TRELLIS_TRACE
        if (lane == 0)
            trace_stamp(p, c, 8 + 8 * warp + 4,
                        (pend0 ? 1u : 0u) | (pend1 ? 2u : 0u) | (tk_taken ? 4u : 0u) | (use[0] ? 8u : 0u) |
                            (use[1] ? 16u : 0u));
#endif
    }
#ifdef TRELLIS_TRACE
    if (lane == 0) trace_stamp(p, c, 8 + 8 * warp + 3, trace_clock());
#endif
}

// Workspace layout: a fixed-capacity counter region at offset 0 (the same
// place for every geometry, so a workspace reused across geometries never
// finds stale partial sums where it expects counters), then the partial sums.
// Counters are left at zero by every call; partial sums need no clearing.
constexpr size_t kCounterCapacity = size_t(1) << 18;            // tiles
constexpr size_t kCounterBytes = kCounterCapacity * sizeof(uint32_t);

// Host-side planning.
template <class C>
SmallMPlan plan_smallm(int K, int N, int k, const DeviceInfo& dev, bool two = false) {
    SmallMPlan p{};
    p.M = C::MM;
    p.K = K;
    p.N = N;
    p.nblocks = K / 256;
    p.row_words = K / 32 * k;
    const int rows_per_tg = C::WARPS * C::ROWS_PER_TILE;
    p.ntg = (N + rows_per_tg - 1) / rows_per_tg;
    if (two) {   // the second matrix starts at the next whole tile-group
        p.npad = p.ntg * rows_per_tg;
        p.ntg *= 2;
    }
    p.U = p.ntg * p.nblocks;
    int P = dev.num_sms * C::OCC;
    if (P > p.U) P = p.U;
    p.P = P;
    p.base = p.U / P;
    p.rem = p.U % P;
    p.div_base1 = FastDiv(static_cast<uint32_t>(p.base + 1));
    p.div_base = FastDiv(static_cast<uint32_t>(p.base));
    return p;
}

template <class C>
size_t smallm_workspace_bytes(const SmallMPlan& p) {
    const size_t partials = static_cast<size_t>(p.P) * 2 * C::WARPS * C::R * C::MM * 4 * sizeof(float);
    return kCounterBytes + partials;
}

template <class C>
bool smallm_fits_counters(const SmallMPlan& p) {
    return static_cast<size_t>(p.ntg) * C::WARPS <= kCounterCapacity;
}

template <class C, int KB, int LL = kL>
int launch_smallm_instance(const uint16_t* x, const uint32_t* codes, const uint16_t* scales,
                           int K, int N, uint16_t* out, void* ws, size_t ws_bytes,
                           cudaStream_t stream, const DeviceInfo& dev, const SecondMatrix& second = SecondMatrix{},
                           int L = kL) {
    if ((second.codes != nullptr) != C::TWO) return -3;
    if (LL != 0 && L != LL) return -3;
    SmallMPlan p = plan_smallm<C>(K, N, KB, dev, C::TWO);
    p.lmask = (1u << L) - 1u;
    p.codes2 = second.codes;
    p.scales2 = second.scales;
    p.out2 = second.out;
    if (!smallm_fits_counters<C>(p)) return -2;
    if (p.P >= (1 << 15)) return -3;   // CTA indices are packed in 15 bits (contributors_info)
    const size_t need = smallm_workspace_bytes<C>(p);
    if (ws_bytes < need || ws == nullptr) return -7;
    p.counters = static_cast<uint32_t*>(ws);
    p.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + kCounterBytes);
#ifdef TRELLIS_TRACE
    p.trace = trace_buffer(&p.trace_words);
#endif
    const size_t smem = C::SMEM_BYTES;
    static std::atomic<unsigned long long> opted{0};
    if (!smem_opt_in(gemm_smallm_kernel<C, KB, LL>, static_cast<int>(C::SMEM_BYTES), opted)) return -5;
    const cudaError_t e = launch_programmatic(gemm_smallm_kernel<C, KB, LL>, static_cast<unsigned>(p.P),
                                              static_cast<unsigned>(C::WARPS * 32), smem, stream,
                                              x, codes, scales, out, p);
    return e == cudaSuccess ? 0 : -5;
}

template <int KB>
int launch_smallm_k(int M, const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int K,
                    int N, uint16_t* out, void* ws, size_t ws_bytes, cudaStream_t stream,
                    const DeviceInfo& dev);

// Any other geometry: k = KB bits, run-time window width L (instantiated in
// gemm_smallm_g_k*.cu, one translation unit per bit width).
template <int KB>
int launch_smallm_g_k(int M, int L, const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int K,
                      int N, uint16_t* out, void* ws, size_t ws_bytes, cudaStream_t stream,
                      const DeviceInfo& dev);

// The same with a second matrix sharing x (instantiated in gemm_smallm2_k*.cu).
template <int KB>
int launch_smallm2_k(int M, const uint16_t* x, const uint32_t* codes, const uint16_t* scales, int K,
                     int N, uint16_t* out, void* ws, size_t ws_bytes, cudaStream_t stream,
                     const DeviceInfo& dev, const SecondMatrix& second);

}  // namespace trellis
