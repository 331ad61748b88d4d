// kvq_elem.cuh -- element-level pieces shared by the bf16 fast kernels
// (fast.cu, staged.cu): group constants, eight-element quantize / dequantize
// steps, statistics accumulators and the per-block partial reduction.
#pragma once

#include "kvq_fast.cuh"

namespace kvq {
namespace elem {

constexpr int kThr = 256;

struct Partial { double s1, s2, mx; };

// ---------------------------------------------------------------- group constants

struct GroupC {
    float s, inv, zp;   // scale and zero point as stored, RN(1/s)
    int32_t zoff;       // clean code = bits(rint(q)+1.5*2^23) + zoff
    bool fast;          // the fast quotient's preconditions hold
    bool lo_ok;         // fast, and no code of the group falls below the clip floor
};

// off = 2^(bits-1) for signed codes (offset binary in registers), else 0.
// The two divisions of the group constants -- range by the integer qmax -
// qmin (or abs-max by qmax) and min by the stored scale -- are the exact
// IEEE quotients, taken by the reciprocal + remainder method when its
// preconditions hold and by __fdiv_rn otherwise.  Codes are monotone in x, so
// the group's lowest code is the code of its minimum: when that one is not
// below the floor no element needs the lower clip.
template <bool ASYM>
__device__ __forceinline__ GroupC make_group(float mn, float mx, const QSpec& q, int off) {
    GroupC g;
    float amag, s;
    if (ASYM) {
        const float rng = fmaxf(__fsub_rn(mx, mn), range_floor());
        const float qr = (float)(q.qmax - q.qmin);
        s = (q.inv_qr > 0.0f && rng <= 0x1p127f) ? quot1(rng, qr, q.inv_qr) : __fdiv_rn(rng, qr);
        amag = fmaxf(fabsf(mn), fabsf(mx));
    } else {
        const float am = fmaxf(mx, range_floor());     // mx carries the abs-max
        s = (q.inv_qr > 0.0f && am <= 0x1p127f) ? quot1(am, (float)q.qmax, q.inv_qr) : __fdiv_rn(am, (float)q.qmax);
        amag = mx;
    }
    g.s = scale_as_stored(s, q.scale_dt);
    g.inv = __frcp_rn(g.s);
    const bool qok = quot_ok(g.s, g.inv, amag);
    if (ASYM) {
        // min / s by the fast quotient only where it is exact (|min| >= 2^-100 or 0)
        const bool mn_ok = qok && (fabsf(mn) >= 0x1p-100f || mn == 0.0f);
        const float a = mn_ok ? quot1(mn, g.s, g.inv) : __fdiv_rn(mn, g.s);
        g.zp = zero_as_stored(rintf(__fsub_rn((float)q.qmin, a)), q.zero_dt);
        g.fast = qok && fabsf(g.zp) < 0x1p21f;
        g.zoff = (int32_t)g.zp + off - (int32_t)kMagicBits;
        g.lo_ok = g.fast && mn_ok && (int32_t)__float_as_uint(__fadd_rn(a, kMagic)) + g.zoff >= q.qmin + off;
    } else {
        g.zp = 0.0f;
        g.fast = qok;
        g.zoff = off - (int32_t)kMagicBits;
        g.lo_ok = qok;
    }
    return g;
}

// Eight elements (one uint4 of bf16) -> eight clean codes, fast quotient.
// kq holds the four pairs' quotient constants; zo[j] the per-element offset.
// LO = false drops the lower clip (valid when every group's lo_ok holds).
template <bool ASYM, bool LO = true>
__device__ __forceinline__ void codes8_fast(const uint4& w, const QuotK (&kq)[4], const int32_t (&zo)[8],
                                            int lo_c, int hi_c, uint32_t (&c)[8]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const u64 r = rint_bits2(quot2(widen_bf16x2(ws[j]), kq[j]));
        if (ASYM && LO) {
            c[2 * j] = (uint32_t)min(__viaddmax_s32((int)lo_bits(r), zo[2 * j], lo_c), hi_c);
            c[2 * j + 1] = (uint32_t)min(__viaddmax_s32((int)hi_bits(r), zo[2 * j + 1], lo_c), hi_c);
        } else if (ASYM) {
            c[2 * j] = (uint32_t)__viaddmin_s32((int)lo_bits(r), zo[2 * j], hi_c);
            c[2 * j + 1] = (uint32_t)__viaddmin_s32((int)hi_bits(r), zo[2 * j + 1], hi_c);
        } else {
            c[2 * j] = lo_bits(r) + (uint32_t)zo[2 * j];
            c[2 * j + 1] = hi_bits(r) + (uint32_t)zo[2 * j + 1];
        }
    }
}

// Same codes through the IEEE division (groups outside the fast domain).
template <bool ASYM>
__device__ __forceinline__ void codes8_slow(const uint4& w, const float (&s)[8], const float (&zp)[8],
                                            const QSpec& q, int off, uint32_t (&c)[8]) {
    float v[8];
    Raw8<__nv_bfloat16> raw;
    raw.u = w;
    widen8(raw, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        Meta m;
        m.s = s[j];
        m.z = zp[j];
        c[j] = (uint32_t)(quant_code<ASYM>(v[j], m, q.lo, q.hi) + off);
    }
}

template <int BITS>
__device__ __forceinline__ typename CodeWord<BITS>::T finish_word(const uint32_t (&c)[8], bool is_signed) {
    typename CodeWord<BITS>::T w = pack_clean8<BITS>(c);
    return is_signed ? flip_signs<BITS>(w) : w;
}

template <int BITS>
__device__ __forceinline__ void store_codes(uint8_t* p, typename CodeWord<BITS>::T w) {
    *reinterpret_cast<typename CodeWord<BITS>::T*>(p) = w;
}

// bf16x2 min/max folding of 4 words
__device__ __forceinline__ void fold_minmax(const uint4& w, uint32_t& mn, uint32_t& mx) {
    mn = bmin2(bmin2(mn, w.x), bmin2(w.y, bmin2(w.z, w.w)));
    mx = bmax2(bmax2(mx, w.x), bmax2(w.y, bmax2(w.z, w.w)));
}
__device__ __forceinline__ void fold_absmax(const uint4& w, uint32_t& mx) {
    mx = bmax2(bmax2(mx, babs2(w.x)), bmax2(babs2(w.y), bmax2(babs2(w.z), babs2(w.w))));
}
__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

constexpr uint32_t kBfPosInf2 = 0x7F807F80u, kBfNegInf2 = 0xFF80FF80u;

// Per-tile sums of |d| and d^2 on float pairs, one accumulator per pair of
// a lane's eight channels, so consecutive rows do not chain on one register.
struct TileAcc {
    u64 a1[4] = {0, 0, 0, 0}, a2[4] = {0, 0, 0, 0};
};

// Kahan-compensated float32 accumulators of the tile sums, one max as float bits.
struct Acc2 {
    float s1 = 0.0f, e1 = 0.0f, s2 = 0.0f, e2 = 0.0f;
    uint32_t mxb = 0;
    __device__ __forceinline__ static void kahan(float& s, float& e, float v) {
        const float y = __fsub_rn(v, e);
        const float t = __fadd_rn(s, y);
        e = __fsub_rn(__fsub_rn(t, s), y);
        s = t;
    }
    __device__ __forceinline__ void fold(const TileAcc& t) {   // a tile's pair sums
        const u64 p1 = add2(add2(t.a1[0], t.a1[1]), add2(t.a1[2], t.a1[3]));
        const u64 p2 = add2(add2(t.a2[0], t.a2[1]), add2(t.a2[2], t.a2[3]));
        kahan(s1, e1, __fadd_rn(lo_of(p1), hi_of(p1)));
        kahan(s2, e2, __fadd_rn(lo_of(p2), hi_of(p2)));
    }
};

// The statistics of eight differences (four float pairs): sums into the
// tile accumulators, the max of |d| (as float bits, |d| >= 0) into mxb.
__device__ __forceinline__ void acc8(const u64 (&d)[4], TileAcc& t, uint32_t& mxb) {
    uint32_t ab[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        ab[2 * j] = lo_bits(d[j]) & 0x7FFFFFFFu;
        ab[2 * j + 1] = hi_bits(d[j]) & 0x7FFFFFFFu;
        t.a1[j] = add2(t.a1[j], pk(__uint_as_float(ab[2 * j]), __uint_as_float(ab[2 * j + 1])));
        t.a2[j] = fma2(d[j], d[j], t.a2[j]);
    }
    const int m0 = __vimax3_s32((int)ab[0], (int)ab[1], (int)ab[2]);
    const int m1 = __vimax3_s32((int)ab[3], (int)ab[4], (int)ab[5]);
    const int m2 = __vimax3_s32((int)ab[6], (int)ab[7], (int)mxb);
    mxb = (uint32_t)__vimax3_s32(m0, m1, m2);
}

// x_hat of eight codes (biased fields u) -> bf16x8; with STATS the
// differences against the source word xw are accumulated instead.
template <bool STATS>
__device__ __forceinline__ uint4 dq8(const uint32_t (&u)[8], const u64 (&cp)[4], const u64 (&sp)[4],
                                    const uint4& xw, TileAcc& t, uint32_t& mxb) {
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const u64 v = mul2(sub2(pk(__uint_as_float(u[2 * j]), __uint_as_float(u[2 * j + 1])), cp[j]), sp[j]);
        o[j] = pack_bf16x2(lo_of(v), hi_of(v));
    }
    if (STATS) {
        const uint32_t xs[4] = {xw.x, xw.y, xw.z, xw.w};
        u64 d[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) d[j] = sub2(widen_bf16x2(xs[j]), widen_bf16x2(o[j]));
        acc8(d, t, mxb);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// exact slow path for groups whose zero point is too large for the biased
// form: q = field - off, then ((float)q - zp) * s exactly as the reference
template <bool STATS>
__device__ __forceinline__ uint4 dq8_slow(const uint32_t (&u)[8], int off, const float (&zp)[8], const float (&s)[8],
                                         const uint4& xw, TileAcc& t, uint32_t& mxb) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        Meta m;
        m.s = s[j];
        m.z = zp[j];
        v[j] = dequant_value((int)(u[j] - kTwo23Bits) - off, m);
    }
    uint4 out;
    out.x = pack_bf16x2(v[0], v[1]);
    out.y = pack_bf16x2(v[2], v[3]);
    out.z = pack_bf16x2(v[4], v[5]);
    out.w = pack_bf16x2(v[6], v[7]);
    if (STATS) {
        const uint32_t xs[4] = {xw.x, xw.y, xw.z, xw.w}, os[4] = {out.x, out.y, out.z, out.w};
        u64 d[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) d[j] = sub2(widen_bf16x2(xs[j]), widen_bf16x2(os[j]));
        acc8(d, t, mxb);
    }
    return out;
}

// A thread's statistics, reduced over its warp in float32 (a fixed shuffle
// tree: 5 roundings, ~3e-7 relative, far inside the 1e-5 bar) and widened to
// double; the max is exact.  Lane 0 holds the warp's values.
__device__ __forceinline__ void warp_partial(const Acc2& A, double& s1, double& s2, double& mx) {
    float f1 = __fsub_rn(A.s1, A.e1), f2 = __fsub_rn(A.s2, A.e2), fm = __uint_as_float(A.mxb);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        f1 = __fadd_rn(f1, __shfl_xor_sync(0xFFFFFFFFu, f1, o));
        f2 = __fadd_rn(f2, __shfl_xor_sync(0xFFFFFFFFu, f2, o));
        fm = fmaxf(fm, __shfl_xor_sync(0xFFFFFFFFu, fm, o));
    }
    s1 = (double)f1;
    s2 = (double)f2;
    mx = (double)fm;
}

__device__ __forceinline__ void block_reduce_partial(const Acc2& A, Partial* partials)
{
    __shared__ double sh1[kThr / 32], sh2[kThr / 32], shm[kThr / 32];
    double s1, s2, mx;
    warp_partial(A, s1, s2, mx);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) { sh1[w] = s1; sh2[w] = s2; shm[w] = mx; }
    __syncthreads();
    if (threadIdx.x == 0) {
        Partial p = {0.0, 0.0, 0.0};
        for (int i = 0; i < kThr / 32; ++i) { p.s1 += sh1[i]; p.s2 += sh2[i]; p.mx = fmax(p.mx, shm[i]); }
        partials[(int64_t)blockIdx.y * gridDim.x + blockIdx.x] = p;
    }
}

// Per-group dequant constants: biased subtrahend 2^23 + off + zp and the scale.
__device__ __forceinline__ void dq_consts(float s, float zp, int off, u64& cp_half, u64& sp_half, bool& fast) {
    fast = fabsf(zp) < 0x1p21f;
    const float c = __fadd_rn(8388608.0f + (float)off, zp);     // exact when |zp| < 2^21
    cp_half = pk(c, c);
    sp_half = pk(s, s);
}


}  // namespace elem
}  // namespace kvq
