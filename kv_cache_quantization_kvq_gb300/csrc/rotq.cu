// rotq.cu -- the randomized Hadamard rotation fused into per-token
// quantization (groups along C) and into dequantization, bf16 tensors.
//
// Method: KV-COBRA notes (papernotes.org), "关键设计" item 4: the orthogonal
// Walsh-Hadamard rotation with fixed random sign flips is absorbed into the
// quantize path, so the rotated tensor never goes to memory; the quantizer is
// "KV Compression 公式到源码对照" §1.1 / §1.2 with groups of g channels of one
// token ("KV cache 压缩：把历史装得更小", value cache grouped per token).
//     rotate + quantize:   y = RN_bf16((1/sqrt(C)) H_C (signs .* x)), codes of y
//     dequantize + rotate: x = RN_bf16(signs .* ((1/sqrt(C)) H_C RN_bf16(x_hat(y))))
// Each result is the one the two separate calls give (kvq_rotate into a bf16
// tensor, then kvq_quantize; kvq_dequantize into bf16, then the inverse
// kvq_rotate), bit for bit: the butterfly stages run in the same order
// (channel bit 1, 2, 4, ...), each output pair formed by the same IEEE
// float32 addition and subtraction, the same multiply by RN(1/sqrt(C)), and
// the quantize / dequantize steps are the same element functions.
//
// Layout: a row (one token, C channels) is held by L = C/32 lanes with 32
// consecutive channels each (four 16-byte loads and stores per lane); the
// five butterfly stages inside a lane run on registers (paired float32
// arithmetic from the second stage on), the log2(L) stages across lanes
// exchange partner values with shuffles.  Groups are 32..C channels, so a
// group is one lane or a few neighbouring lanes of its row: the group min /
// max is a fold of the lane's bf16 pairs and at most log2(L) shuffles.  One
// read and one write of the tensor; no shared memory.
#include <algorithm>
#include <cmath>

#include "kvq_div.cuh"
#include "kvq_elem.cuh"

namespace kvq {

namespace {

using namespace elem;

constexpr int kRQThreads = 256;
constexpr int kLaneCh = 32;                     // channels per lane

// One 16-byte global load that bypasses L1 (the rows are read once).
__device__ __forceinline__ uint4 ld_once16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Sign masks of the C/2 bf16 pairs of a row in shared memory (bit 15 / 31
// set where the channel flips); a lane reads its 16 with four 16-byte loads.
template <int C>
__device__ __forceinline__ void sign_masks(const int8_t* signs, uint32_t* sm) {
    for (int k = threadIdx.x; k < C / 2; k += blockDim.x)
        sm[k] = (signs[2 * k] < 0 ? 0x8000u : 0u) | (signs[2 * k + 1] < 0 ? 0x80000000u : 0u);
    __syncthreads();
}
__device__ __forceinline__ uint4 lane_masks(const uint32_t* sm, int c0, int k) {
    return *reinterpret_cast<const uint4*>(sm + c0 / 2 + 4 * k);
}

// Butterflies of channel bits 1 .. 16 inside the lane: V[k] holds channels
// (2k, 2k+1).  Stage h pairs channel e with e + h (bit h of e clear) into
// (v_e + v_{e+h}, v_e - v_{e+h}).
__device__ __forceinline__ void fwht_in_lane(u64 (&V)[16]) {
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float a = lo_of(V[k]), b = hi_of(V[k]);
        V[k] = pk(__fadd_rn(a, b), __fsub_rn(a, b));
    }
#pragma unroll
    for (int hw = 1; hw < 16; hw <<= 1) {       // channel bit 2*hw is word bit hw
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if ((k & hw) == 0) {
                const u64 a = V[k], b = V[k + hw];
                V[k] = add2(a, b);
                V[k + hw] = sub2(a, b);
            }
        }
    }
}

// Butterflies of channel bits 32, 64, ... across the L lanes of a row
// (channel bit 32*m is lane bit m).  The lane with the bit clear keeps
// own + partner, the other partner - own: fma(+-1, own, partner) rounds once,
// so each equals the IEEE sum or difference.
template <int L>
__device__ __forceinline__ void fwht_across(u64 (&V)[16], int p) {
#pragma unroll
    for (int m = 1; m < L; m <<= 1) {
        const float sg = (p & m) ? -1.0f : 1.0f;
        const u64 S = pk(sg, sg);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, lo_bits(V[k]), m);
            const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, hi_bits(V[k]), m);
            V[k] = fma2(V[k], S, pk(__uint_as_float(lo), __uint_as_float(hi)));
        }
    }
}

template <int L>
__device__ __forceinline__ void fwht_row(u64 (&V)[16], int p, float rscale) {
    fwht_in_lane(V);
    fwht_across<L>(V, p);
    const u64 R = pk(rscale, rscale);
#pragma unroll
    for (int k = 0; k < 16; ++k) V[k] = mul2(V[k], R);
}

// ---------------------------------------------------------------- rotate + quantize

// Codes of the lane's 32 bf16 values (16 words) with one group's constants,
// stored at dst (BITS * 4 bytes).
template <int BITS, bool ASYM>
__device__ __forceinline__ void store_lane_codes(const uint32_t (&yb)[16], const GroupC& gc, const QSpec& q, int off,
                                                 uint8_t* dst) {
    const int lo_c = q.qmin + off, hi_c = q.qmax + off;
    typename CodeWord<BITS>::T cw[4];
    if (gc.fast) {
        QuotK kq[4];
        int32_t zo[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) { kq[j].ns = pk(-gc.s, -gc.s); kq[j].inv = pk(gc.inv, gc.inv); }
#pragma unroll
        for (int j = 0; j < 8; ++j) zo[j] = gc.zoff;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 w = make_uint4(yb[4 * k], yb[4 * k + 1], yb[4 * k + 2], yb[4 * k + 3]);
            uint32_t cc[8];
            if (!ASYM || gc.lo_ok) codes8_fast<ASYM, false>(w, kq, zo, lo_c, hi_c, cc);
            else codes8_fast<ASYM, true>(w, kq, zo, lo_c, hi_c, cc);
            cw[k] = finish_word<BITS>(cc, q.is_signed);
        }
    } else {
        float s8[8], z8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) { s8[j] = gc.s; z8[j] = gc.zp; }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 w = make_uint4(yb[4 * k], yb[4 * k + 1], yb[4 * k + 2], yb[4 * k + 3]);
            uint32_t cc[8];
            codes8_slow<ASYM>(w, s8, z8, q, off, cc);
            cw[k] = finish_word<BITS>(cc, q.is_signed);
        }
    }
    if constexpr (BITS == 8) {
        uint4* d = reinterpret_cast<uint4*>(dst);
        d[0] = make_uint4(cw[0].x, cw[0].y, cw[1].x, cw[1].y);
        d[1] = make_uint4(cw[2].x, cw[2].y, cw[3].x, cw[3].y);
    } else if constexpr (BITS == 4) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    } else {
        *reinterpret_cast<uint2*>(dst) = make_uint2((uint32_t)cw[0] | ((uint32_t)cw[1] << 16),
                                                    (uint32_t)cw[2] | ((uint32_t)cw[3] << 16));
    }
}

template <int BITS, bool ASYM, int C>
__global__ void __launch_bounds__(kRQThreads, 4)
rot_quant_kernel(const QArgs a, const int8_t* signs, float rscale, DivU32 tdiv)
{
    constexpr int L = C / kLaneCh;              // lanes per row
    constexpr int RPW = 32 / L;                 // rows per warp
    const QSpec& q = a.q;
    const int lane = threadIdx.x & 31, p = lane % L;
    const int c0 = p * kLaneCh;
    const int gl = (int)(q.g / kLaneCh);        // lanes per group: 1 .. L
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const uint64_t T = (uint64_t)q.T, Tq = (uint64_t)q.Tq, rows = (uint64_t)q.outer * T;
    const uint64_t ng = (uint64_t)q.ngroups;
    __shared__ __align__(16) uint32_t sm[C / 2];
    sign_masks<C>(signs, sm);

    const uint64_t nwarps = (uint64_t)gridDim.x * (kRQThreads / 32);
    for (uint64_t w = (uint64_t)blockIdx.x * (kRQThreads / 32) + (threadIdx.x >> 5); w * RPW < rows; w += nwarps) {
        const uint64_t row = w * RPW + (uint64_t)(lane / L);
        const bool live = row < rows;
        uint4 xw[4];
        const unsigned char* src = static_cast<const unsigned char*>(a.x) + (row * C + c0) * 2;
#pragma unroll
        for (int k = 0; k < 4; ++k) xw[k] = live ? ld_once16(src + 16 * k) : make_uint4(0u, 0u, 0u, 0u);
        u64 V[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 mk = lane_masks(sm, c0, k);
            V[4 * k] = widen_bf16x2(xw[k].x ^ mk.x);
            V[4 * k + 1] = widen_bf16x2(xw[k].y ^ mk.y);
            V[4 * k + 2] = widen_bf16x2(xw[k].z ^ mk.z);
            V[4 * k + 3] = widen_bf16x2(xw[k].w ^ mk.w);
        }
        fwht_row<L>(V, p, rscale);
        uint32_t yb[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) yb[k] = pack_bf16x2(lo_of(V[k]), hi_of(V[k]));

        const uint64_t o = div_u32((uint32_t)row, tdiv), t = row - o * T;   // rows < 2^32
        const bool res = t >= Tq;
        // group min / max (abs-max when symmetric) of the bf16 values
        uint32_t mn = kBfPosInf2, mx = ASYM ? kBfNegInf2 : 0u;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (ASYM) { mn = bmin2(mn, yb[k]); mx = bmax2(mx, yb[k]); }
            else mx = bmax2(mx, babs2(yb[k]));
        }
        float fmn = fminf(lo_f(mn), hi_f(mn)), fmx = fmaxf(lo_f(mx), hi_f(mx));
        for (int m = 1; m < gl; m <<= 1) {
            if (ASYM) fmn = fminf(fmn, __shfl_xor_sync(0xFFFFFFFFu, fmn, m));
            fmx = fmaxf(fmx, __shfl_xor_sync(0xFFFFFFFFu, fmx, m));
        }
        if (!live) continue;
        if (res) {
            uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.resid) +
                                                ((o * (uint64_t)q.R + (t - Tq)) * C + c0));
#pragma unroll
            for (int k = 0; k < 4; ++k) d[k] = make_uint4(yb[4 * k], yb[4 * k + 1], yb[4 * k + 2], yb[4 * k + 3]);
            continue;
        }
        const GroupC gc = make_group<ASYM>(fmn, fmx, q, off);
        if (p % gl == 0) {
            Meta mt;
            mt.s = gc.s;
            mt.z = gc.zp;
            write_meta(a, (int64_t)((o * Tq + t) * ng + (uint64_t)(c0 / q.g)), mt);
        }
        uint8_t* dst = static_cast<uint8_t*>(a.codes) + (o * Tq + t) * ((uint64_t)C * BITS / 8) + (uint64_t)c0 * BITS / 8;
        store_lane_codes<BITS, ASYM>(yb, gc, q, off, dst);
    }
}

// ---------------------------------------------------------------- dequantize + inverse rotation

template <int BITS, bool ASYM, int C>
__global__ void __launch_bounds__(kRQThreads, 4)
dequant_rot_kernel(const QArgs a, const int8_t* signs, float rscale, DivU32 tdiv)
{
    constexpr int L = C / kLaneCh;
    constexpr int RPW = 32 / L;
    using W = typename CodeWord<BITS>::T;
    const QSpec& q = a.q;
    const int lane = threadIdx.x & 31, p = lane % L;
    const int c0 = p * kLaneCh;
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const uint64_t T = (uint64_t)q.T, Tq = (uint64_t)q.Tq, rows = (uint64_t)q.outer * T;
    const uint64_t ng = (uint64_t)q.ngroups;
    __shared__ __align__(16) uint32_t sm[C / 2];
    sign_masks<C>(signs, sm);

    const uint64_t nwarps = (uint64_t)gridDim.x * (kRQThreads / 32);
    for (uint64_t w = (uint64_t)blockIdx.x * (kRQThreads / 32) + (threadIdx.x >> 5); w * RPW < rows; w += nwarps) {
        const uint64_t row = w * RPW + (uint64_t)(lane / L);
        const bool live = row < rows;
        const uint64_t o = live ? div_u32((uint32_t)row, tdiv) : 0, t = live ? row - o * T : 0;   // rows < 2^32
        uint32_t yb[16];
        if (!live) {
#pragma unroll
            for (int k = 0; k < 16; ++k) yb[k] = 0u;
        } else if (t >= Tq) {
            const unsigned char* src = reinterpret_cast<const unsigned char*>(
                static_cast<const __nv_bfloat16*>(a.resid) + ((o * (uint64_t)q.R + (t - Tq)) * C + c0));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 v = ld_once16(src + 16 * k);
                yb[4 * k] = v.x; yb[4 * k + 1] = v.y; yb[4 * k + 2] = v.z; yb[4 * k + 3] = v.w;
            }
        } else {
            const unsigned char* cs = static_cast<const unsigned char*>(a.codes) + (o * Tq + t) * ((uint64_t)C * BITS / 8) +
                                      (uint64_t)c0 * BITS / 8;
            W cw[4];
            if constexpr (BITS == 8) {
                const uint4 v0 = ld_once16(cs), v1 = ld_once16(cs + 16);
                cw[0] = make_uint2(v0.x, v0.y); cw[1] = make_uint2(v0.z, v0.w);
                cw[2] = make_uint2(v1.x, v1.y); cw[3] = make_uint2(v1.z, v1.w);
            } else if constexpr (BITS == 4) {
                const uint4 v = ld_once16(cs);
                cw[0] = v.x; cw[1] = v.y; cw[2] = v.z; cw[3] = v.w;
            } else {
                const uint2 v = *reinterpret_cast<const uint2*>(cs);
                cw[0] = (uint16_t)v.x; cw[1] = (uint16_t)(v.x >> 16); cw[2] = (uint16_t)v.y; cw[3] = (uint16_t)(v.y >> 16);
            }
            const int64_t mi = (int64_t)((o * Tq + t) * ng + (uint64_t)(c0 / q.g));
            const float s = load_meta(a.scale, q.scale_dt, mi);
            const float z = ASYM ? load_meta(a.zero, q.zero_dt, mi) : 0.0f;
            u64 cp, sp;
            bool fast;
            dq_consts(s, z, off, cp, sp, fast);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t u[8];
                unpack_biased8<BITS>(q.is_signed ? flip_signs<BITS>(cw[k]) : cw[k], u);
                if (fast) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const u64 v = mul2(sub2(pk(__uint_as_float(u[2 * j]), __uint_as_float(u[2 * j + 1])), cp), sp);
                        yb[4 * k + j] = pack_bf16x2(lo_of(v), hi_of(v));
                    }
                } else {
                    Meta m;
                    m.s = s;
                    m.z = z;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        yb[4 * k + j] = pack_bf16x2(dequant_value((int)(u[2 * j] - kTwo23Bits) - off, m),
                                                    dequant_value((int)(u[2 * j + 1] - kTwo23Bits) - off, m));
                }
            }
        }
        u64 V[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) V[k] = widen_bf16x2(yb[k]);
        fwht_row<L>(V, p, rscale);
        if (!live) continue;
        uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + (row * C + c0));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 mk = lane_masks(sm, c0, k);
            d[k] = make_uint4(pack_bf16x2(lo_of(V[4 * k]), hi_of(V[4 * k])) ^ mk.x,
                              pack_bf16x2(lo_of(V[4 * k + 1]), hi_of(V[4 * k + 1])) ^ mk.y,
                              pack_bf16x2(lo_of(V[4 * k + 2]), hi_of(V[4 * k + 2])) ^ mk.z,
                              pack_bf16x2(lo_of(V[4 * k + 3]), hi_of(V[4 * k + 3])) ^ mk.w);
        }
    }
}

template <typename K>
cudaError_t rq_launch(K kernel, const QArgs& a, const int8_t* signs, int64_t C, cudaStream_t st)
{
    const uint64_t rows = (uint64_t)a.q.outer * (uint64_t)a.q.T;
    if (rows == 0) return cudaSuccess;
    const uint64_t rpw = 32 / (uint64_t)(C / kLaneCh);
    const uint64_t warps = (rows + rpw - 1) / rpw;
    const uint64_t blocks = std::max<uint64_t>(1, std::min<uint64_t>((warps + 7) / 8, (uint64_t)sm_count() * 8));
    const float rscale = (float)(1.0 / std::sqrt((double)C));
    kernel<<<(unsigned)blocks, kRQThreads, 0, st>>>(a, signs, rscale, make_div((uint32_t)a.q.T));
    return cudaGetLastError();
}

template <int BITS, bool ASYM>
cudaError_t rq_dispatch(const QArgs& a, const int8_t* signs, bool dequant, cudaStream_t st)
{
    switch (a.q.C) {
    case 32: return dequant ? rq_launch(dequant_rot_kernel<BITS, ASYM, 32>, a, signs, 32, st)
                            : rq_launch(rot_quant_kernel<BITS, ASYM, 32>, a, signs, 32, st);
    case 64: return dequant ? rq_launch(dequant_rot_kernel<BITS, ASYM, 64>, a, signs, 64, st)
                            : rq_launch(rot_quant_kernel<BITS, ASYM, 64>, a, signs, 64, st);
    case 128: return dequant ? rq_launch(dequant_rot_kernel<BITS, ASYM, 128>, a, signs, 128, st)
                             : rq_launch(rot_quant_kernel<BITS, ASYM, 128>, a, signs, 128, st);
    default: return dequant ? rq_launch(dequant_rot_kernel<BITS, ASYM, 256>, a, signs, 256, st)
                            : rq_launch(rot_quant_kernel<BITS, ASYM, 256>, a, signs, 256, st);
    }
}

cudaError_t rq_run(const QArgs& a, const int8_t* signs, bool dequant, cudaStream_t st)
{
    const bool asym = a.q.mode == KVQ_ASYM;
    switch (a.q.bits) {
    case 8: return asym ? rq_dispatch<8, true>(a, signs, dequant, st) : rq_dispatch<8, false>(a, signs, dequant, st);
    case 4: return asym ? rq_dispatch<4, true>(a, signs, dequant, st) : rq_dispatch<4, false>(a, signs, dequant, st);
    default: return asym ? rq_dispatch<2, true>(a, signs, dequant, st) : rq_dispatch<2, false>(a, signs, dequant, st);
    }
}

}  // namespace

bool rotq_supported(const QSpec& q)
{
    return q.axis == KVQ_GROUP_ALONG_C && q.outer * q.T < (int64_t(1) << 32) && q.x_dt == KVQ_BF16 &&
           (q.C == 32 || q.C == 64 || q.C == 128 || q.C == 256) && q.g >= kLaneCh && q.g <= q.C && q.C % q.g == 0 &&
           (q.g & (q.g - 1)) == 0;
}

cudaError_t launch_rotate_quantize(const QArgs& a, const int8_t* signs, cudaStream_t st)
{
    return rq_run(a, signs, false, st);
}

cudaError_t launch_dequantize_rotate(const QArgs& a, const int8_t* signs, cudaStream_t st)
{
    return rq_run(a, signs, true, st);
}

}  // namespace kvq
