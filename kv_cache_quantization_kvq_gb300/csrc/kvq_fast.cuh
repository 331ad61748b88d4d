// kvq_fast.cuh -- element pipeline of the bf16 fast paths (sm_103a).
//
// The quantize / dequantize / statistics kernels are HBM-bound only if each
// element costs a handful of issue slots (at the copy roofline an SM must
// retire ~17 elements per clock, i.e. ~7.5 instructions per element).  So:
//  * arithmetic runs on packed float pairs (PTX add/mul/fma .rn.f32x2): one
//    instruction rounds two independent float32 results exactly as two
//    scalar instructions would;
//  * x / s is the exact IEEE quotient computed from the group's reciprocal
//    inv = RN(1/s) with one FMA remainder correction (Markstein's division
//    theorem: with q = RN(x*inv), the remainder r = x - s*q is exact in one
//    FMA and RN(q + r*inv) is the correctly rounded quotient), so no
//    per-element reciprocal instruction is issued.  A unit test checks it
//    bit for bit against __fdiv_rn exhaustively over bf16 operands when
//    |x| and |x / s| are at least 2^-100; below that the remainder or the
//    quotient underflows, but then |x / s| is far below 1/2 and the rounded
//    code -- the only thing used -- is the same (also checked exhaustively);
//    the same method divides a group's range by the integer qmax - qmin;
//  * round-to-nearest-even to an integer is one add of 1.5*2^23: for
//    |y| < 2^22 the sum is exact and its bit pattern is 0x4B400000 + rint(y),
//    so the integer code is read from the bits with no conversion
//    instruction (likewise 0x4B000000 | u reads as 2^23 + u on the way back);
//  * bf16 data is compared in place with min/max.bf16x2.
// Groups whose values do not satisfy the preconditions of the fast quotient
// (scale outside [2^-100, 2^100] or |x / s| >= 2^21) are quantized with
// __fdiv_rn instead; the result is the same, only slower.
#pragma once

#include "kvq_device.cuh"

namespace kvq {

// ---------------------------------------------------------------- float pairs

typedef unsigned long long u64;

__device__ __forceinline__ u64 pk(float lo, float hi) {
    return (u64)__float_as_uint(lo) | ((u64)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float lo_of(u64 v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_of(u64 v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint32_t lo_bits(u64 v) { return (uint32_t)v; }
__device__ __forceinline__ uint32_t hi_bits(u64 v) { return (uint32_t)(v >> 32); }

__device__ __forceinline__ u64 add2(u64 a, u64 b) {
    u64 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ u64 sub2(u64 a, u64 b) {
    u64 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
    u64 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
    u64 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// A bf16x2 word widened to a float pair (exact).
__device__ __forceinline__ u64 widen_bf16x2(uint32_t w) { return pk(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u)); }

// bf16x2 compare in place
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t babs2(uint32_t a) { return a & 0x7FFF7FFFu; }

// ---------------------------------------------------------------- exact quotient

// Per-group constants for the fast quotient: -s and inv = RN(1/s), paired.
struct QuotK { u64 ns, inv; };

__device__ __forceinline__ QuotK quot_consts(float s_lo, float s_hi) {
    QuotK k;
    k.ns = pk(-s_lo, -s_hi);
    k.inv = pk(__frcp_rn(s_lo), __frcp_rn(s_hi));
    return k;
}

// RN(x / s) for both lanes of a pair (one Markstein remainder correction).
__device__ __forceinline__ u64 quot2(u64 x, const QuotK& k) {
    const u64 q = mul2(x, k.inv);
    const u64 r = fma2(k.ns, q, x);
    return fma2(r, k.inv, q);
}

// scalar version (per-group bookkeeping)
__device__ __forceinline__ float quot1(float x, float s, float inv) {
    const float q = __fmul_rn(x, inv);
    const float r = __fmaf_rn(-s, q, x);
    return __fmaf_rn(r, inv, q);
}

// The fast quotient's preconditions for a group with scale s and values of
// magnitude at most amag.
__device__ __forceinline__ bool quot_ok(float s, float inv, float amag) {
    return s >= 0x1p-100f && s <= 0x1p100f && __fmul_rn(amag, inv) < 0x1p21f;
}

constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23
constexpr uint32_t kMagicBits = 0x4B400000u;   // its bit pattern
constexpr uint32_t kTwo23Bits = 0x4B000000u;   // 2^23

// rint(q) as a biased integer: bits(q + 1.5*2^23) = 0x4B400000 + rint(q).
__device__ __forceinline__ u64 rint_bits2(u64 q) { return add2(q, pk(kMagic, kMagic)); }

// ---------------------------------------------------------------- code packing

// Eight clean codes c[j] in [0, 2^BITS) -> one BITS-byte word (element j at bit j*BITS).
template <int BITS>
__device__ __forceinline__ typename CodeWord<BITS>::T pack_clean8(const uint32_t (&c)[8]) {
    if constexpr (BITS == 4) {
        const uint32_t a = c[0] + (c[1] << 4), b = c[2] + (c[3] << 4);
        const uint32_t d = c[4] + (c[5] << 4), e = c[6] + (c[7] << 4);
        return (a + (b << 8)) + ((d + (e << 8)) << 16);
    } else if constexpr (BITS == 2) {
        const uint32_t a = c[0] + (c[1] << 2) + (c[2] << 4) + (c[3] << 6);
        const uint32_t b = c[4] + (c[5] << 2) + (c[6] << 4) + (c[7] << 6);
        return (uint16_t)(a + (b << 8));
    } else {
        uint2 w;
        w.x = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
        w.y = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
        return w;
    }
}

// The eight fields of a code word as "2^23 + field" float bit patterns.
template <int BITS>
__device__ __forceinline__ void unpack_biased8(typename CodeWord<BITS>::T w, uint32_t (&u)[8]) {
    if constexpr (BITS == 4) {
        const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
        u[0] = __byte_perm(lo, kTwo23Bits, 0x7440);
        u[1] = __byte_perm(hi, kTwo23Bits, 0x7440);
        u[2] = __byte_perm(lo, kTwo23Bits, 0x7441);
        u[3] = __byte_perm(hi, kTwo23Bits, 0x7441);
        u[4] = __byte_perm(lo, kTwo23Bits, 0x7442);
        u[5] = __byte_perm(hi, kTwo23Bits, 0x7442);
        u[6] = __byte_perm(lo, kTwo23Bits, 0x7443);
        u[7] = __byte_perm(hi, kTwo23Bits, 0x7443);
    } else if constexpr (BITS == 2) {
        const uint32_t v = (uint32_t)w;
#pragma unroll
        for (int j = 0; j < 8; ++j) u[j] = kTwo23Bits | ((v >> (2 * j)) & 3u);
    } else {
        u[0] = __byte_perm(w.x, kTwo23Bits, 0x7440);
        u[1] = __byte_perm(w.x, kTwo23Bits, 0x7441);
        u[2] = __byte_perm(w.x, kTwo23Bits, 0x7442);
        u[3] = __byte_perm(w.x, kTwo23Bits, 0x7443);
        u[4] = __byte_perm(w.y, kTwo23Bits, 0x7440);
        u[5] = __byte_perm(w.y, kTwo23Bits, 0x7441);
        u[6] = __byte_perm(w.y, kTwo23Bits, 0x7442);
        u[7] = __byte_perm(w.y, kTwo23Bits, 0x7443);
    }
}

// Signed fields are stored two's complement; flipping the sign bit of every
// field turns them into offset binary (field + 2^(BITS-1)), which the biased
// unpack reads directly.
template <int BITS> __device__ __forceinline__ uint32_t sign_flip_mask();
template <> __device__ __forceinline__ uint32_t sign_flip_mask<4>() { return 0x88888888u; }
template <> __device__ __forceinline__ uint32_t sign_flip_mask<2>() { return 0xAAAAu; }
template <> __device__ __forceinline__ uint32_t sign_flip_mask<8>() { return 0x80808080u; }

template <int BITS>
__device__ __forceinline__ typename CodeWord<BITS>::T flip_signs(typename CodeWord<BITS>::T w) {
    if constexpr (BITS == 8) {
        w.x ^= 0x80808080u;
        w.y ^= 0x80808080u;
        return w;
    } else {
        return (typename CodeWord<BITS>::T)((uint32_t)w ^ sign_flip_mask<BITS>());
    }
}

}  // namespace kvq
