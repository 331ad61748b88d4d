// mixed.cu -- per-token mixed precision: each token of the cache is stored at
// the precision its tag selects (2, 4, 8 or 16 bits).
//
// Method: "大模型KV缓存自适应量化实战" (adaptive KV-cache quantization), §2.1
// (four levels, 2/4/8/16 bits, chosen per token), §3.1 (per-token dynamic
// quantization; symmetric for 2 and 4 bits, asymmetric for 8 bits, 16 bits
// stored as is), §3.2 (same-precision data kept together; 2-bit precision tags
// 00/01/10/11 for 2/4/8/16 bits).  The controller that chooses the levels is
// not part of this path: the caller passes the tags.
//
// Layout of one slice (outer index o) of a [outer, T, C] cache:
//  - records: token t's record starts at byte off[o][t] of the slice's stream
//    (streams are T * 2C bytes apart, the size of an all-16-bit slice); a record
//    is the packed codes followed by the bf16 scale (and, for 8 bits, the bf16
//    zero point), or the C bf16 values for 16 bits;
//  - off[o][0..T]: exclusive prefix sums of the record sizes (off[o][T] = the
//    bytes the slice uses);
//  - tags2[o][ceil(T/4)]: the 2-bit tags, token t at bit 2*(t%4) of byte t/4.
// The codes of a 2/4/8-bit record follow the packing of the uniform formats
// (channel c at bit (c mod 8/bits)*bits of byte c*bits/8, two's complement).
#include <algorithm>

#include "kvq_elem.cuh"

namespace kvq {

namespace {

using namespace elem;

constexpr int kMThreads = 256;

// record bytes of a token with tag g (0..3 -> 2/4/8/16 bits) and C channels
__host__ __device__ __forceinline__ int64_t record_bytes(int g, int64_t C) {
    return g == 0 ? C / 4 + 2 : g == 1 ? C / 2 + 2 : g == 2 ? C + 4 : 2 * C;
}

// One CTA per slice.  Thread i owns the tokens [i*K, (i+1)*K), K = ceil(T /
// 256) rounded up to a multiple of 4: it sums its records' sizes, the block
// scans the 256 sums, and each thread then writes its tokens' offsets and the
// bytes of packed tags that cover them (no byte is shared by two threads).
__global__ void __launch_bounds__(kMThreads)
mixed_plan_kernel(const uint8_t* tags, int64_t T, int64_t C, int64_t* off, uint8_t* tags2)
{
    __shared__ int64_t warp_sums[kMThreads / 32];
    const int64_t o = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint8_t* tg = tags + o * T;
    int64_t* of = off + o * (T + 1);
    uint8_t* t2 = tags2 + o * ((T + 3) / 4);
    const int64_t K = ((T + kMThreads - 1) / kMThreads + 3) / 4 * 4;
    const int64_t t0 = std::min<int64_t>(T, (int64_t)tid * K), t1 = std::min<int64_t>(T, t0 + K);
    int64_t sum = 0;
#pragma unroll 8
    for (int64_t t = t0; t < t1; ++t) sum += record_bytes(tg[t] & 3, C);
    int64_t v = sum;                                               // inclusive scan within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t u = __shfl_up_sync(0xFFFFFFFFu, v, d);
        if (lane >= d) v += u;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    int64_t before = 0;
    for (int w = 0; w < warp; ++w) before += warp_sums[w];
    int64_t run = before + v - sum;                                // offset of token t0
    for (int64_t t = t0; t < t1; t += 4) {
        uint32_t b = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (t + j < t1) {
                const int g = tg[t + j] & 3;
                of[t + j] = run;
                run += record_bytes(g, C);
                b |= (uint32_t)g << (2 * j);
            }
        }
        t2[t / 4] = (uint8_t)b;
    }
    if (tid == kMThreads - 1) of[T] = before + v;                  // the slice's total
}

struct MixedFormats { QSpec f2, f4, f8; };                         // per-token formats of tags 0, 1, 2

__device__ __forceinline__ void put_bf16(uint8_t* p, float v) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    *reinterpret_cast<__nv_bfloat16*>(p) = h;                      // records start at even offsets
}
__device__ __forceinline__ float get_bf16(const uint8_t* p) { return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p)); }

// 2-byte stores of a code word (records start at even offsets only)
template <int BITS>
__device__ __forceinline__ void store_word_u16(uint8_t* p, typename CodeWord<BITS>::T w) {
    uint16_t* d = reinterpret_cast<uint16_t*>(p);
    if constexpr (BITS == 2) {
        d[0] = w;
    } else if constexpr (BITS == 4) {
        d[0] = (uint16_t)w;
        d[1] = (uint16_t)(w >> 16);
    } else {
        d[0] = (uint16_t)w.x;
        d[1] = (uint16_t)(w.x >> 16);
        d[2] = (uint16_t)w.y;
        d[3] = (uint16_t)(w.y >> 16);
    }
}
template <int BITS>
__device__ __forceinline__ typename CodeWord<BITS>::T load_word_u16(const uint8_t* p) {
    const uint16_t* s = reinterpret_cast<const uint16_t*>(p);
    if constexpr (BITS == 2) {
        return s[0];
    } else if constexpr (BITS == 4) {
        return (uint32_t)s[0] | ((uint32_t)s[1] << 16);
    } else {
        return make_uint2((uint32_t)s[0] | ((uint32_t)s[1] << 16), (uint32_t)s[2] | ((uint32_t)s[3] << 16));
    }
}

// Codes of one lane's 8 channels in the record's format, by the exact fast
// quotient when the group allows it (the same constants and steps as the
// uniform per-token kernels), else by the IEEE division.
template <int BITS, bool ASYM>
__device__ __forceinline__ void record_codes(const uint4& w, const GroupC& gc, const QSpec& q, uint8_t* pay) {
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    uint32_t cc[8];
    if (gc.fast) {
        QuotK kq[4];
        kq[0].ns = pk(-gc.s, -gc.s);
        kq[0].inv = pk(gc.inv, gc.inv);
        kq[1] = kq[2] = kq[3] = kq[0];
        int32_t zo[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) zo[j] = gc.zoff;
        if (!ASYM || gc.lo_ok) codes8_fast<ASYM, false>(w, kq, zo, q.qmin + off, q.qmax + off, cc);
        else codes8_fast<ASYM, true>(w, kq, zo, q.qmin + off, q.qmax + off, cc);
    } else {
        float s8[8], z8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) { s8[j] = gc.s; z8[j] = gc.zp; }
        codes8_slow<ASYM>(w, s8, z8, q, off, cc);
    }
    store_word_u16<BITS>(pay, finish_word<BITS>(cc, q.is_signed));
}

// LT = C/8 lanes per token, 8 channels (one 16-byte load) per lane; 32/LT
// tokens per warp.  The token's min / max / abs-max are folded as bf16 pairs
// and reduced over its LT lanes; the tag then selects the format.
template <int LT>
__global__ void __launch_bounds__(kMThreads)
mixed_quant_kernel(const __nv_bfloat16* x, const uint8_t* tags, int64_t outer, int64_t T, const int64_t* off,
                   uint8_t* stream, const MixedFormats F)
{
    constexpr int C = 8 * LT, TPW = 32 / LT;
    const int lane = threadIdx.x & 31, sub = lane % LT;
    const uint64_t ntok = (uint64_t)outer * T;
    const uint64_t warps = (uint64_t)gridDim.x * (kMThreads / 32);
    for (uint64_t w0 = ((uint64_t)blockIdx.x * (kMThreads / 32) + (threadIdx.x >> 5)) * TPW; w0 < ntok;
         w0 += warps * TPW) {
        const uint64_t tok = w0 + lane / LT;
        const bool live = tok < ntok;
        const uint4 v = live ? *reinterpret_cast<const uint4*>(x + tok * C + sub * 8) : make_uint4(0, 0, 0, 0);
        uint32_t mn = kBfPosInf2, mx = kBfNegInf2, am = 0u;
        fold_minmax(v, mn, mx);
        fold_absmax(v, am);
#pragma unroll
        for (int d = 1; d < LT; d <<= 1) {
            mn = bmin2(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, d));
            mx = bmax2(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, d));
            am = bmax2(am, __shfl_xor_sync(0xFFFFFFFFu, am, d));
        }
        if (!live) continue;
        const uint64_t o = tok / T, t = tok - o * T;
        const int g = tags[tok] & 3;
        uint8_t* rec = stream + o * (uint64_t)T * 2 * C + off[o * (T + 1) + t];
        if (g == 3) {                                              // 16 bits: the values as stored
            uint16_t* d = reinterpret_cast<uint16_t*>(rec) + sub * 8;
            const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) { d[2 * k] = (uint16_t)ws[k]; d[2 * k + 1] = (uint16_t)(ws[k] >> 16); }
            continue;
        }
        const float fmn = fminf(lo_f(mn), hi_f(mn)), fmx = fmaxf(lo_f(mx), hi_f(mx)), fam = fmaxf(lo_f(am), hi_f(am));
        GroupC gc;
        int bits;
        if (g == 2) {
            gc = make_group<true>(fmn, fmx, F.f8, 0);
            record_codes<8, true>(v, gc, F.f8, rec + sub * 8);
            bits = 8;
        } else if (g == 1) {
            gc = make_group<false>(0.0f, fam, F.f4, 8);
            record_codes<4, false>(v, gc, F.f4, rec + sub * 4);
            bits = 4;
        } else {
            gc = make_group<false>(0.0f, fam, F.f2, 2);
            record_codes<2, false>(v, gc, F.f2, rec + sub * 2);
            bits = 2;
        }
        if (sub == 0) {
            const int64_t pb = (int64_t)C * bits / 8;
            put_bf16(rec + pb, gc.s);
            if (g == 2) put_bf16(rec + pb + 2, gc.zp);
        }
    }
}

// LT lanes per token, 8 channels per lane, one 16-byte store each.
template <int LT>
__global__ void __launch_bounds__(kMThreads)
mixed_dequant_kernel(const uint8_t* stream, const uint8_t* tags2, int64_t outer, int64_t T, const int64_t* off,
                     __nv_bfloat16* out)
{
    constexpr int C = 8 * LT, TPW = 32 / LT;
    const int lane = threadIdx.x & 31, sub = lane % LT;
    const uint64_t ntok = (uint64_t)outer * T;
    const uint64_t warps = (uint64_t)gridDim.x * (kMThreads / 32);
    const int64_t tb = (T + 3) / 4;
    for (uint64_t w0 = ((uint64_t)blockIdx.x * (kMThreads / 32) + (threadIdx.x >> 5)) * TPW; w0 < ntok;
         w0 += warps * TPW) {
        const uint64_t tok = w0 + lane / LT;
        if (tok >= ntok) continue;
        const uint64_t o = tok / T, t = tok - o * T;
        const int g = (tags2[o * tb + t / 4] >> (2 * (t % 4))) & 3;
        const uint8_t* rec = stream + o * (uint64_t)T * 2 * C + off[o * (T + 1) + t];
        uint4 r;
        if (g == 3) {
            const uint16_t* sv = reinterpret_cast<const uint16_t*>(rec) + sub * 8;
            r = make_uint4((uint32_t)sv[0] | ((uint32_t)sv[1] << 16), (uint32_t)sv[2] | ((uint32_t)sv[3] << 16),
                           (uint32_t)sv[4] | ((uint32_t)sv[5] << 16), (uint32_t)sv[6] | ((uint32_t)sv[7] << 16));
        } else {
            const int bits = g == 0 ? 2 : (g == 1 ? 4 : 8);
            const int64_t pb = (int64_t)C * bits / 8;
            Meta m;
            m.s = get_bf16(rec + pb);
            m.z = g == 2 ? get_bf16(rec + pb + 2) : 0.0f;
            uint32_t u[8];
            if (g == 2) unpack_biased8<8>(load_word_u16<8>(rec + sub * 8), u);
            else if (g == 1) unpack_biased8<4>(flip_signs<4>(load_word_u16<4>(rec + sub * 4)), u);
            else unpack_biased8<2>(flip_signs<2>(load_word_u16<2>(rec + sub * 2)), u);
            const int offb = g == 2 ? 0 : (1 << (bits - 1));   // offset binary of the symmetric codes
            u64 cp[4], sp[4];
            bool fast;
            u64 cph, sph;
            dq_consts(m.s, m.z, offb, cph, sph, fast);
#pragma unroll
            for (int k = 0; k < 4; ++k) { cp[k] = cph; sp[k] = sph; }
            TileAcc ta;
            uint32_t mxb = 0;
            if (fast) {
                r = dq8<false>(u, cp, sp, make_uint4(0, 0, 0, 0), ta, mxb);
            } else {
                float zs[8], ss[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) { zs[j] = m.z; ss[j] = m.s; }
                r = dq8_slow<false>(u, offb, zs, ss, make_uint4(0, 0, 0, 0), ta, mxb);
            }
        }
        *reinterpret_cast<uint4*>(out + tok * C + sub * 8) = r;
    }
}

unsigned warps_grid(uint64_t ntok)
{
    const uint64_t blocks = (ntok + kMThreads / 32 - 1) / (kMThreads / 32);
    return (unsigned)std::max<uint64_t>(1, std::min<uint64_t>(blocks, (uint64_t)sm_count() * 16));
}

}  // namespace

int64_t mixed_record_bytes(int tag, int64_t C) { return record_bytes(tag & 3, C); }

cudaError_t launch_mixed_quantize(const void* x, const uint8_t* tags, int64_t outer, int64_t T, int64_t C,
                                  void* stream_buf, int64_t* off, uint8_t* tags2, const QSpec& f2, const QSpec& f4,
                                  const QSpec& f8, cudaStream_t st)
{
    if (outer == 0 || T == 0) return cudaSuccess;
    mixed_plan_kernel<<<(unsigned)outer, kMThreads, 0, st>>>(tags, T, C, off, tags2);
    const MixedFormats F = {f2, f4, f8};
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    uint8_t* sb = static_cast<uint8_t*>(stream_buf);
    const unsigned grid = warps_grid((uint64_t)outer * T);
    switch (C) {
    case 64: mixed_quant_kernel<8><<<grid, kMThreads, 0, st>>>(xb, tags, outer, T, off, sb, F); break;
    case 128: mixed_quant_kernel<16><<<grid, kMThreads, 0, st>>>(xb, tags, outer, T, off, sb, F); break;
    default: mixed_quant_kernel<32><<<grid, kMThreads, 0, st>>>(xb, tags, outer, T, off, sb, F); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_mixed_dequantize(const void* stream_buf, const int64_t* off, const uint8_t* tags2, int64_t outer,
                                    int64_t T, int64_t C, void* out, cudaStream_t st)
{
    if (outer == 0 || T == 0) return cudaSuccess;
    const uint8_t* sb = static_cast<const uint8_t*>(stream_buf);
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
    const unsigned grid = warps_grid((uint64_t)outer * T);
    switch (C) {
    case 64: mixed_dequant_kernel<8><<<grid, kMThreads, 0, st>>>(sb, tags2, outer, T, off, ob); break;
    case 128: mixed_dequant_kernel<16><<<grid, kMThreads, 0, st>>>(sb, tags2, outer, T, off, ob); break;
    default: mixed_dequant_kernel<32><<<grid, kMThreads, 0, st>>>(sb, tags2, outer, T, off, ob); break;
    }
    return cudaGetLastError();
}

}  // namespace kvq
