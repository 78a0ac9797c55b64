// Device-side building blocks of the packed-Trellis decode (sm_103a).
//
// The per-weight arithmetic follows the wide-prefill Metal kernel on the page
// "mlx-bun 0.2.0 -> 0.4.0" (package/src/model/trellis-wide-prefill.ts): an
// L-bit window of the block's bit-string, the multiply-add hash, the sum of the
// hash's four bytes minus 510, the correctly rounded fp32 quotient by
// 147.800537109375 (the page reaches it with a residual correction; here a
// two-part reciprocal gives the same bits, see code_to_value), the per-row
// scale and a round to bf16.
//
// Work is organised in "groups" of 32 consecutive weights of one block
// (T = 256 weights, so 8 groups per block).  Group g holds weights
// t = 32g .. 32g+31, which start at bits (T-1-t)*k; those are exactly the k
// words (8-1-g)*k .. (8-g)*k-1 of the block, plus the window tails that spill
// into the next word: word (8-g)*k, which for g = 0 wraps to word 0 of the
// same block.  Inside a group the bit offset of weight j is the compile-time
// constant (31-j)*k, so every shift below folds to an immediate.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace trellis {

constexpr int kT = 256;                 // weights per block
constexpr int kL = 12;                  // window bits
constexpr int kGroupsPerBlock = kT / 32;

constexpr uint32_t kHashMul = 34038481u;
constexpr uint32_t kHashAdd = 76625530u;
// dp4a(z, 0x01010101, 0x4B400000) is the bit pattern of the float
// 1.5*2^23 + (byte sum), exactly; subtracting 1.5*2^23 + 510 leaves
// float(code) exactly (both operands share the exponent 2^23, unit ulp).
constexpr uint32_t kMagicBits = 0x4B400000u;
constexpr float kMagicPlusBias = 12583422.0f;

// Window of weight j (0..31) of a group, from the group's k words w[0..k-1]
// and the lookahead word w[k].  LL is the window width when it is fixed at
// compile time (the page's L = 12: a window inside one word needs only a
// shift); LL = 0 takes the width from `lmask` = 2^L - 1 at run time and always
// funnel-shifts (the same one instruction).  Any 1 <= k <= 8 and L <= 24 keep a
// window inside words wi and wi + 1 <= k.
template <int KB, int LL = kL>
__device__ __forceinline__ uint32_t group_window(const uint32_t (&w)[KB + 1], int j, uint32_t lmask = 0u) {
    const int o = (31 - j) * KB;     // constant after unrolling
    const int wi = o >> 5;
    const int off = o & 31;
    if constexpr (LL == 0) {
        return __funnelshift_r(w[wi], w[wi + 1], off) & lmask;
    } else {
        uint32_t win;
        if (off + LL <= 32)
            win = w[wi] >> off;
        else
            win = __funnelshift_r(w[wi], w[wi + 1], off);
        return win & ((1u << LL) - 1u);
    }
}

// The KB code words of one group, starting at p, with the widest loads its
// alignment allows: a group starts at word (7 - g) * KB of a block and blocks
// and rows start on 32-byte boundaries, so p is 16-byte aligned when KB is a
// multiple of 4 and 8-byte aligned when KB is even.
template <int KB>
__device__ __forceinline__ void ldg_group(const uint32_t* __restrict__ p, uint32_t (&w)[KB]) {
    if constexpr (KB % 4 == 0) {
#pragma unroll
        for (int i = 0; i < KB / 4; ++i) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + i);
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
    } else if constexpr (KB % 2 == 0) {
#pragma unroll
        for (int i = 0; i < KB / 2; ++i) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(p) + i);
            w[2 * i] = v.x; w[2 * i + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < KB; ++i) w[i] = __ldg(p + i);
    }
}

// float(code) -> code / 147.800537109375 rounded to nearest fp32, as a
// multiplication by the reciprocal held in two fp32 parts (the double-word
// constant multiplication of Brisebarre and Muller, "Correctly rounded
// multiplication by arbitrary precision constants", IEEE TC 2008):
// kRecipHi is 1/c to 14 significant bits (14189 * 2^-21), so code * kRecipHi
// is exact for |code| <= 510 (at most 23 bits), and kRecipLo is the fp32 of
// 1/c - kRecipHi.  One FMA adds code * kRecipLo to the exact product before
// its only rounding.  For every integer code in [-510, 510] the result is the
// correctly rounded quotient; the host tests check each code against exact
// rational arithmetic, reading these two constants from this file.
constexpr float kRecipHi = 0x1.bb68p-8f;
constexpr float kRecipLo = 0x1.1a16f2p-25f;

__device__ __forceinline__ float code_to_value(float code) {
    return __fmaf_rn(code, kRecipLo, __fmul_rn(code, kRecipHi));
}

// 12-bit window -> fp32 value, bit-exact with code / 147.800537109375.
__device__ __forceinline__ float window_value(uint32_t win) {
    const uint32_t z = win * kHashMul + kHashAdd;
    const float biased = __uint_as_float(__dp4a(z, 0x01010101u, kMagicBits));
    return code_to_value(__fsub_rn(biased, kMagicPlusBias));
}

// Two windows at once: the same steps, the fp32 ones as paired (f32x2)
// instructions, so each issue slot serves two weights.
__device__ __forceinline__ float2 window_value2(uint32_t wa, uint32_t wb) {
    const uint32_t za = wa * kHashMul + kHashAdd;
    const uint32_t zb = wb * kHashMul + kHashAdd;
    const float2 biased = make_float2(__uint_as_float(__dp4a(za, 0x01010101u, kMagicBits)),
                                      __uint_as_float(__dp4a(zb, 0x01010101u, kMagicBits)));
    const float2 code = __fadd2_rn(biased, make_float2(-kMagicPlusBias, -kMagicPlusBias));
    return __ffma2_rn(code, make_float2(kRecipLo, kRecipLo), __fmul2_rn(code, make_float2(kRecipHi, kRecipHi)));
}

// ---- programmatic dependent launch --------------------------------------------
// Wait until the grids this launch depends on have completed and their writes
// are visible (returns at once for an ordinary launch).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next programmatically launched grid on the stream be scheduled.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- quotient table ---------------------------------------------------------
// The value depends on the window only through the byte sum S = code + 510 of
// its hash.  Over the 4096 12-bit windows S only takes values in [62, 964]
// (the host tests enumerate them), so a shared-memory table holds value(S)
// for those 903 sums, once per lane: entry (S, lane) sits at byte
// 128*(S - 62) + 4*lane, and the 32 lanes of a warp always read 32 different
// banks, whatever their S.  dp4a(z, 0x80808080, base) yields base + 128*S
// directly (base = the lane's entry address minus 128*62, in wrapping 32-bit
// arithmetic), so a lookup is one dp4a and one shared load.
constexpr int kSumLo = 62;
constexpr int kSumHi = 964;
constexpr int kTableSums = kSumHi - kSumLo + 1;                  // 903
constexpr int kQuotientTableBytes = kTableSums * 32 * 4;        // 115,584 bytes

__device__ __forceinline__ void build_quotient_table(float* table, int tid, int nthreads) {
    for (int e = tid; e < kTableSums * 8; e += nthreads) {
        const int si = e >> 3, quad = e & 7;
        const float v = code_to_value(static_cast<float>(si + kSumLo - 510));
        *reinterpret_cast<float4*>(table + si * 32 + quad * 4) = make_float4(v, v, v, v);
    }
}

__device__ __forceinline__ uint32_t quotient_table_lane_address(const void* table, int lane) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(table)) + 4u * static_cast<uint32_t>(lane) -
           static_cast<uint32_t>(kSumLo * 128);
}

__device__ __forceinline__ float quotient_lookup(uint32_t win, uint32_t lane_address) {
    const uint32_t z = win * kHashMul + kHashAdd;
    const uint32_t addr = __dp4a(z, 0x80808080u, lane_address);
    float v;
    asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// bf16 round-to-nearest-even of w, returned as the fp32 with the same value
// (the bf16 bits in the upper half, zeros below).
__device__ __forceinline__ float round_bf16_as_f32(float w) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(w), "f"(0.0f));
    return __uint_as_float(r);
}

// Two floats -> packed bf16x2 (lo in the low half, i.e. at the lower address).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// fp32 -> bf16 bits, round to nearest even.
__device__ __forceinline__ uint16_t bf16_bits_rn(float f) {
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Exact unsigned 32-bit division by a runtime constant d >= 1
// (Granlund & Montgomery, "Division by invariant integers using
// multiplication", PLDI 1994): q = (mulhi(n, m) + n) >> l.
struct FastDiv {
    uint32_t d, m, l;
    __host__ __device__ FastDiv() : d(1), m(0), l(0) {}
    __host__ explicit FastDiv(uint32_t divisor) : d(divisor) {
        l = 0;
        while ((1ull << l) < divisor) ++l;
        m = static_cast<uint32_t>((((1ull << l) - divisor) << 32) / divisor + 1);
    }
    __device__ __forceinline__ uint32_t div(uint32_t n) const {
        return static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(n, m)) + n) >> l);
    }
};

}  // namespace trellis
