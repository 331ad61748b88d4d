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

#include "kvq_device.cuh"

namespace kvq {

namespace {

constexpr int kMThreads = 256;

// record bytes of a token with tag g (0..3 -> 2/4/8/16 bits) and C channels
__host__ __device__ __forceinline__ int64_t record_bytes(int g, int64_t C) {
    return g == 0 ? C / 4 + 2 : g == 1 ? C / 2 + 2 : g == 2 ? C + 4 : 2 * C;
}

// One CTA per slice: record offsets by a block-wide exclusive scan over the
// tokens (chunks of kMThreads), and the packed 2-bit tags.
__global__ void __launch_bounds__(kMThreads)
mixed_plan_kernel(const uint8_t* tags, int64_t T, int64_t C, int64_t* off, uint8_t* tags2)
{
    __shared__ int64_t warp_sums[kMThreads / 32];
    __shared__ int64_t carry;
    const int64_t o = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint8_t* tg = tags + o * T;
    int64_t* of = off + o * (T + 1);
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int64_t base = 0; base < T; base += kMThreads) {
        const int64_t t = base + tid;
        const int64_t sz = t < T ? record_bytes(tg[t] & 3, C) : 0;
        int64_t v = sz;                                            // inclusive scan within the warp
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t u = __shfl_up_sync(0xFFFFFFFFu, v, d);
            if (lane >= d) v += u;
        }
        if (lane == 31) warp_sums[warp] = v;
        __syncthreads();
        int64_t before = carry;
        for (int w = 0; w < warp; ++w) before += warp_sums[w];
        if (t < T) of[t] = before + v - sz;
        __syncthreads();
        if (tid == kMThreads - 1) carry = before + v;             // the chunk's total
        __syncthreads();
    }
    if (tid == 0) of[T] = carry;
    // packed tags: thread handles one byte (4 tokens)
    for (int64_t k = tid; k < (T + 3) / 4; k += kMThreads) {
        uint32_t b = 0;
        for (int j = 0; j < 4; ++j)
            if (k * 4 + j < T) b |= (uint32_t)(tg[k * 4 + j] & 3) << (2 * j);
        tags2[o * ((T + 3) / 4) + k] = (uint8_t)b;
    }
}

struct MixedFormats { QSpec f2, f4, f8; };                         // per-token formats of tags 0, 1, 2

__device__ __forceinline__ void put_bf16(uint8_t* p, float v) {
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    *reinterpret_cast<__nv_bfloat16*>(p) = h;                      // records start at even offsets
}
__device__ __forceinline__ float get_bf16(const uint8_t* p) { return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p)); }

// Warp per token: E = C/32 consecutive channels per lane.
template <int E>
__global__ void __launch_bounds__(kMThreads)
mixed_quant_kernel(const __nv_bfloat16* x, const uint8_t* tags, int64_t outer, int64_t T, const int64_t* off,
                   uint8_t* stream, const MixedFormats F)
{
    constexpr int C = 32 * E;
    const int lane = threadIdx.x & 31;
    const uint64_t ntok = (uint64_t)outer * T;
    const uint64_t warps = (uint64_t)gridDim.x * (kMThreads / 32);
    for (uint64_t w = (uint64_t)blockIdx.x * (kMThreads / 32) + (threadIdx.x >> 5); w < ntok; w += warps) {
        const uint64_t o = w / T, t = w - o * T;
        const int g = tags[w] & 3;
        uint8_t* rec = stream + o * (uint64_t)T * 2 * C + off[o * (T + 1) + t];
        float v[E];
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = __bfloat162float(x[w * C + lane * E + e]);
        if (g == 3) {                                              // 16 bits: the values as stored
#pragma unroll
            for (int e = 0; e < E; ++e) put_bf16(rec + 2 * (lane * E + e), v[e]);
            continue;
        }
        const QSpec& q = g == 0 ? F.f2 : (g == 1 ? F.f4 : F.f8);
        const int bits = g == 0 ? 2 : (g == 1 ? 4 : 8);
        float mn = v[0], mx = v[0], am = fabsf(v[0]);
#pragma unroll
        for (int e = 1; e < E; ++e) { mn = fminf(mn, v[e]); mx = fmaxf(mx, v[e]); am = fmaxf(am, fabsf(v[e])); }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, d));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, d));
            am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, d));
        }
        const bool asym = g == 2;
        const Meta m = asym ? meta_asym(mn, mx, q) : meta_sym(am, q);
        const uint32_t mask = (1u << bits) - 1u;
        // this lane's E codes occupy E*bits bits starting at bit lane*E*bits
        uint32_t acc = 0;
        int nb = 0;
        uint8_t* pay = rec + (lane * E * bits) / 8;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int c = asym ? quant_code<true>(v[e], m, q.lo, q.hi) : quant_code<false>(v[e], m, q.lo, q.hi);
            acc |= ((uint32_t)c & mask) << nb;
            nb += bits;
            if (nb == 8) { *pay++ = (uint8_t)acc; acc = 0; nb = 0; }
        }
        if (nb) {                                                  // 2-bit codes of fewer than 4 channels
            // the lane's bits share a byte with the next lane's: combine within the warp
            const uint32_t mine = acc;
            const int lanes_per_byte = 8 / (E * bits);
            uint32_t b = 0;
            const int first = lane - lane % lanes_per_byte;
            for (int j = 0; j < lanes_per_byte; ++j)
                b |= __shfl_sync(0xFFFFFFFFu, mine, first + j) << (j * E * bits);
            if (lane % lanes_per_byte == 0) *pay = (uint8_t)b;
        }
        if (lane == 0) {
            const int64_t pb = (int64_t)C * bits / 8;
            put_bf16(rec + pb, m.s);
            if (asym) put_bf16(rec + pb + 2, m.z);
        }
    }
}

template <int E>
__global__ void __launch_bounds__(kMThreads)
mixed_dequant_kernel(const uint8_t* stream, const uint8_t* tags2, int64_t outer, int64_t T, const int64_t* off,
                     __nv_bfloat16* out)
{
    constexpr int C = 32 * E;
    const int lane = threadIdx.x & 31;
    const uint64_t ntok = (uint64_t)outer * T;
    const uint64_t warps = (uint64_t)gridDim.x * (kMThreads / 32);
    const int64_t tb = (T + 3) / 4;
    for (uint64_t w = (uint64_t)blockIdx.x * (kMThreads / 32) + (threadIdx.x >> 5); w < ntok; w += warps) {
        const uint64_t o = w / T, t = w - o * T;
        const int g = (tags2[o * tb + t / 4] >> (2 * (t % 4))) & 3;
        const uint8_t* rec = stream + o * (uint64_t)T * 2 * C + off[o * (T + 1) + t];
        __nv_bfloat16* dst = out + w * C + lane * E;
        if (g == 3) {
#pragma unroll
            for (int e = 0; e < E; ++e) dst[e] = __float2bfloat16_rn(get_bf16(rec + 2 * (lane * E + e)));
            continue;
        }
        const int bits = g == 0 ? 2 : (g == 1 ? 4 : 8);
        const int64_t pb = (int64_t)C * bits / 8;
        Meta m;
        m.s = get_bf16(rec + pb);
        m.z = g == 2 ? get_bf16(rec + pb + 2) : 0.0f;
        const uint32_t mask = (1u << bits) - 1u;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int c = lane * E + e;
            const uint32_t byte = rec[(c * bits) / 8];
            uint32_t f = (byte >> ((c * bits) % 8)) & mask;
            int qv = (int)f;
            if (g != 2 && (f >> (bits - 1))) qv -= (1 << bits);    // symmetric: two's complement
            dst[e] = __float2bfloat16_rn(dequant_value(qv, m));
        }
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
    case 64: mixed_quant_kernel<2><<<grid, kMThreads, 0, st>>>(xb, tags, outer, T, off, sb, F); break;
    case 128: mixed_quant_kernel<4><<<grid, kMThreads, 0, st>>>(xb, tags, outer, T, off, sb, F); break;
    default: mixed_quant_kernel<8><<<grid, kMThreads, 0, st>>>(xb, tags, outer, T, off, sb, F); break;
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
    case 64: mixed_dequant_kernel<2><<<grid, kMThreads, 0, st>>>(sb, tags2, outer, T, off, ob); break;
    case 128: mixed_dequant_kernel<4><<<grid, kMThreads, 0, st>>>(sb, tags2, outer, T, off, ob); break;
    default: mixed_dequant_kernel<8><<<grid, kMThreads, 0, st>>>(sb, tags2, outer, T, off, ob); break;
    }
    return cudaGetLastError();
}

}  // namespace kvq
