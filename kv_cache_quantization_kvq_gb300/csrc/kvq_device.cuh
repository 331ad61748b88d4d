// kvq_device.cuh -- device-side helpers of the kvq CUDA library (sm_103a).
//
// Every float operation on the quantization path is an explicit IEEE
// round-to-nearest intrinsic (__fdiv_rn, __fsub_rn, __fadd_rn, __fmul_rn) so
// that no multiply-add is contracted and the division is the true IEEE
// quotient; the library is also built with -fmad=false.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_internal.h"

namespace kvq {

// ---------------------------------------------------------------- dtype I/O

// Eight consecutive source elements as raw bits (copied bit-exact into the
// residual window) plus their float32 widening (bf16 -> f32 is exact).
template <typename InT> struct Raw8;
template <> struct Raw8<__nv_bfloat16> { uint4 u; };
template <> struct Raw8<float> { uint4 u0, u1; };

__device__ __forceinline__ void load_raw8(const __nv_bfloat16* p, Raw8<__nv_bfloat16>& r) {
    r.u = *reinterpret_cast<const uint4*>(p);
}
__device__ __forceinline__ void load_raw8(const float* p, Raw8<float>& r) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
    r.u0 = q[0];
    r.u1 = q[1];
}
__device__ __forceinline__ void store_raw8(__nv_bfloat16* p, const Raw8<__nv_bfloat16>& r) {
    *reinterpret_cast<uint4*>(p) = r.u;
}
__device__ __forceinline__ void store_raw8(float* p, const Raw8<float>& r) {
    uint4* q = reinterpret_cast<uint4*>(p);
    q[0] = r.u0;
    q[1] = r.u1;
}
__device__ __forceinline__ void zero_raw8(Raw8<__nv_bfloat16>& r) { r.u = make_uint4(0, 0, 0, 0); }
__device__ __forceinline__ void zero_raw8(Raw8<float>& r) {
    r.u0 = make_uint4(0, 0, 0, 0);
    r.u1 = r.u0;
}

__device__ __forceinline__ void widen2(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
}
__device__ __forceinline__ void widen8(const Raw8<__nv_bfloat16>& r, float (&v)[8]) {
    widen2(r.u.x, v[0], v[1]);
    widen2(r.u.y, v[2], v[3]);
    widen2(r.u.z, v[4], v[5]);
    widen2(r.u.w, v[6], v[7]);
}
__device__ __forceinline__ void widen8(const Raw8<float>& r, float (&v)[8]) {
    v[0] = __uint_as_float(r.u0.x); v[1] = __uint_as_float(r.u0.y);
    v[2] = __uint_as_float(r.u0.z); v[3] = __uint_as_float(r.u0.w);
    v[4] = __uint_as_float(r.u1.x); v[5] = __uint_as_float(r.u1.y);
    v[6] = __uint_as_float(r.u1.z); v[7] = __uint_as_float(r.u1.w);
}

// round-to-nearest-even float -> bf16 pair, packed low element first
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float round_to_bf16(float v) {
    return __bfloat162float(__float2bfloat16_rn(v));
}

// store 8 float results in the output dtype (bf16: rounded once)
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = u;
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
    float4* q = reinterpret_cast<float4*>(p);
    q[0] = make_float4(v[0], v[1], v[2], v[3]);
    q[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// x_hat as it lands in OutT (bf16 rounding applied) -- used by the error stats
template <typename OutT> __device__ __forceinline__ float as_output(float v);
template <> __device__ __forceinline__ float as_output<float>(float v) { return v; }
template <> __device__ __forceinline__ float as_output<__nv_bfloat16>(float v) { return round_to_bf16(v); }

// ---------------------------------------------------------------- metadata

// Value of one stored metadata entry, widened to float.
__device__ __forceinline__ float load_meta(const void* buf, int dtype, int64_t i) {
    if (dtype == KVQ_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(buf)[i]);
    if (dtype == KVQ_I8) return (float)reinterpret_cast<const int8_t*>(buf)[i];
    return reinterpret_cast<const float*>(buf)[i];
}

// Round a float to the storage dtype of a scale; returns the value the codes
// are computed with (the stored value, widened back).
__device__ __forceinline__ float scale_as_stored(float s, int dtype) {
    return dtype == KVQ_BF16 ? round_to_bf16(s) : s;
}
__device__ __forceinline__ void store_scale(void* buf, int dtype, int64_t i, float s_use) {
    if (dtype == KVQ_BF16) reinterpret_cast<__nv_bfloat16*>(buf)[i] = __float2bfloat16_rn(s_use);
    else reinterpret_cast<float*>(buf)[i] = s_use;
}
// zero point: rint already applied; int8 saturates, bf16 rounds, f32 keeps.
__device__ __forceinline__ float zero_as_stored(float zp, int dtype) {
    if (dtype == KVQ_I8) return fminf(fmaxf(zp, -128.0f), 127.0f);
    if (dtype == KVQ_BF16) return round_to_bf16(zp);
    return zp;
}
__device__ __forceinline__ void store_zero(void* buf, int dtype, int64_t i, float zp_use) {
    if (dtype == KVQ_I8) reinterpret_cast<int8_t*>(buf)[i] = (int8_t)(int)zp_use;
    else if (dtype == KVQ_BF16) reinterpret_cast<__nv_bfloat16*>(buf)[i] = __float2bfloat16_rn(zp_use);
    else reinterpret_cast<float*>(buf)[i] = zp_use;
}

// Floor of the abs-max / range: the float32 value nearest 1e-8.
__device__ __forceinline__ float range_floor() { return 1e-8f; }

struct Meta { float s, z; };

// Symmetric group parameters from the group abs-max ("KV Compression
// 公式到源码对照" §1.1: scale = max|x| / qmax).
__device__ __forceinline__ Meta meta_sym(float amax, const QSpec& q) {
    float s = __fdiv_rn(fmaxf(amax, range_floor()), (float)q.qmax);
    Meta m;
    m.s = scale_as_stored(s, q.scale_dt);
    m.z = 0.0f;
    return m;
}

// Asymmetric group parameters ("KV Compression 公式到源码对照" §1.2:
// scale = (max - min)/(qmax - qmin), zero_point = round(qmin - min/scale)).
__device__ __forceinline__ Meta meta_asym(float mn, float mx, const QSpec& q) {
    float rng = fmaxf(__fsub_rn(mx, mn), range_floor());
    float s = __fdiv_rn(rng, (float)(q.qmax - q.qmin));
    Meta m;
    m.s = scale_as_stored(s, q.scale_dt);
    float zp = rintf(__fsub_rn((float)q.qmin, __fdiv_rn(mn, m.s)));
    m.z = zero_as_stored(zp, q.zero_dt);
    return m;
}

__device__ __forceinline__ void write_meta(const QArgs& a, int64_t mi, const Meta& m) {
    store_scale(a.scale, a.q.scale_dt, mi, m.s);
    if (a.q.mode == KVQ_ASYM) store_zero(a.zero, a.q.zero_dt, mi, m.z);
}

// One code: clip(rint(x / s) [+ zp], lo, hi), all float32, clipped as an
// integer value (no wrap-around).
template <bool ASYM>
__device__ __forceinline__ int quant_code(float x, const Meta& m, float lo, float hi) {
    float r = rintf(__fdiv_rn(x, m.s));
    float v = ASYM ? __fadd_rn(r, m.z) : r;
    return (int)fminf(fmaxf(v, lo), hi);
}

// x_hat = (q - zp) * s, one float32 subtraction (exact for code-sized ints)
// and one rounded multiply.
__device__ __forceinline__ float dequant_value(int q, const Meta& m) {
    return __fmul_rn(__fsub_rn((float)q, m.z), m.s);
}

// ---------------------------------------------------------------- packing

// Eight codes of one source chunk pack into BITS bytes: element j at bit j*BITS.
template <int BITS> struct CodeWord;
template <> struct CodeWord<8> { using T = uint2; };
template <> struct CodeWord<4> { using T = uint32_t; };
template <> struct CodeWord<2> { using T = uint16_t; };

template <int BITS>
__device__ __forceinline__ typename CodeWord<BITS>::T pack8(const int (&q)[8]) {
    if constexpr (BITS == 8) {
        uint2 w;
        w.x = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) |
              ((uint32_t)(q[2] & 0xFF) << 16) | ((uint32_t)(q[3] & 0xFF) << 24);
        w.y = (uint32_t)(q[4] & 0xFF) | ((uint32_t)(q[5] & 0xFF) << 8) |
              ((uint32_t)(q[6] & 0xFF) << 16) | ((uint32_t)(q[7] & 0xFF) << 24);
        return w;
    } else {
        uint32_t w = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) w |= ((uint32_t)q[j] & ((1u << BITS) - 1u)) << (j * BITS);
        return (typename CodeWord<BITS>::T)w;
    }
}

// Unpack eight codes; SIGNED sign-extends each field.
template <int BITS, bool SIGNED>
__device__ __forceinline__ void unpack8(typename CodeWord<BITS>::T w, int (&q)[8]) {
    if constexpr (BITS == 8) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t fx = (w.x >> (8 * j)) & 0xFFu, fy = (w.y >> (8 * j)) & 0xFFu;
            q[j] = SIGNED ? (int)(int8_t)fx : (int)fx;
            q[j + 4] = SIGNED ? (int)(int8_t)fy : (int)fy;
        }
    } else {
        uint32_t u = (uint32_t)w;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int f = (int)((u >> (j * BITS)) & ((1u << BITS) - 1u));
            q[j] = (SIGNED && f >= (1 << (BITS - 1))) ? f - (1 << BITS) : f;
        }
    }
}

// One code from a packed stream (any element index), for the generic paths.
__device__ __forceinline__ int code_at(const uint8_t* codes, int bits, int64_t ci, bool is_signed) {
    int per = 8 / bits;
    uint32_t f = ((uint32_t)codes[ci / per] >> ((int)(ci % per) * bits)) & ((1u << bits) - 1u);
    int v = (int)f;
    if (is_signed && v >= (1 << (bits - 1))) v -= (1 << bits);
    return v;
}

// ---------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_max_xor(float v, int lanes) {
    for (int o = lanes >> 1; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_min_xor(float v, int lanes) {
    for (int o = lanes >> 1; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Order-preserving map float -> uint32 (for atomic min/max of any float and
// for radix selection): larger float, larger key.  -0 and +0 map apart; the
// callers canonicalise where that matters.
__device__ __forceinline__ uint32_t float_key(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

}  // namespace kvq
