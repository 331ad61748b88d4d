// rotate.cu -- data-free randomized Hadamard rotation of every row (the C
// channels of one token) of a [outer, T, C] tensor.
//
// Method: KV-COBRA notes (papernotes.org), "关键设计" item 4: an orthogonal
// Walsh-Hadamard matrix with fixed random sign flips mixes the coordinates so
// that each gets the mean variance before scalar quantization; used here
// without the calibrated projection.
//     forward  y = (1/sqrt(C)) H_C (signs .* x)
//     inverse  x = signs .* ((1/sqrt(C)) H_C y)
// H_C is the Sylvester Hadamard matrix, H_2n = [[H_n, H_n], [H_n, -H_n]].
//
// Fast transform in registers: a row is held by L = min(32, C/8) lanes with
// E = C/L consecutive channels each (16-byte vector loads and stores); the
// log2(E) butterfly stages inside a lane run on registers, the log2(L) stages
// across lanes exchange partner values with shuffles (channel bit h = m*E is
// lane bit m).  One read and one write of the tensor.
#include <algorithm>
#include <cmath>

#include "kvq_device.cuh"

namespace kvq {

namespace {

constexpr int kRThreads = 256;

template <int C, int XDT, int ODT>
__global__ void __launch_bounds__(kRThreads)
rotate_kernel(const void* x, void* out, const int8_t* signs, uint64_t rows, int inverse, float scale)
{
    constexpr int L = C / 8 < 32 ? C / 8 : 32;   // lanes per row
    constexpr int E = C / L;                     // channels per lane
    constexpr int RPW = 32 / L;                  // rows per warp
    constexpr int XB = XDT == KVQ_BF16 ? 2 : 4, OB = ODT == KVQ_BF16 ? 2 : 4;
    const int lane = threadIdx.x & 31;
    const int p = lane % L;                      // position of the lane within its row
    const int c0 = p * E;
    uint32_t neg = 0;                            // channels c0 + e flipped by the signs
#pragma unroll
    for (int e = 0; e < E; ++e) neg |= (signs[c0 + e] < 0 ? 1u : 0u) << e;

    const uint64_t warps = (uint64_t)gridDim.x * (kRThreads / 32);
    for (uint64_t w = (uint64_t)blockIdx.x * (kRThreads / 32) + (threadIdx.x >> 5); w * RPW < rows; w += warps) {
        const uint64_t row = w * RPW + (uint64_t)(lane / L);
        const bool live = row < rows;
        float v[E];
        if (live) {
            const unsigned char* src = static_cast<const unsigned char*>(x) + (row * C + c0) * XB;
#pragma unroll
            for (int k = 0; k < E * XB / 16; ++k) {
                const uint4 q = *reinterpret_cast<const uint4*>(src + 16 * k);
                const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
                if constexpr (XDT == KVQ_BF16) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        v[8 * k + 2 * i] = __uint_as_float(wv[i] << 16);
                        v[8 * k + 2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[4 * k + i] = __uint_as_float(wv[i]);
                }
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) v[e] = 0.0f;
        }
        if (!inverse) {
#pragma unroll
            for (int e = 0; e < E; ++e) if (neg & (1u << e)) v[e] = -v[e];
        }
        // butterflies inside the lane: channel bit h < E
#pragma unroll
        for (int h = 1; h < E; h <<= 1) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                if ((e & h) == 0) {
                    const float a = v[e], b = v[e + h];
                    v[e] = __fadd_rn(a, b);
                    v[e + h] = __fsub_rn(a, b);
                }
            }
        }
        // butterflies across the row's lanes: channel bit m*E is lane bit m
#pragma unroll
        for (int m = 1; m < L; m <<= 1) {
            const bool upper = (p & m) != 0;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float o = __shfl_xor_sync(0xFFFFFFFFu, v[e], m);
                v[e] = upper ? __fsub_rn(o, v[e]) : __fadd_rn(v[e], o);
            }
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
            v[e] = __fmul_rn(v[e], scale);
            if (inverse && (neg & (1u << e))) v[e] = -v[e];
        }
        if (live) {
            unsigned char* dst = static_cast<unsigned char*>(out) + (row * C + c0) * OB;
#pragma unroll
            for (int k = 0; k < E * OB / 16; ++k) {
                uint4 q;
                if constexpr (ODT == KVQ_BF16) {
                    q.x = pack_bf16x2(v[8 * k], v[8 * k + 1]);
                    q.y = pack_bf16x2(v[8 * k + 2], v[8 * k + 3]);
                    q.z = pack_bf16x2(v[8 * k + 4], v[8 * k + 5]);
                    q.w = pack_bf16x2(v[8 * k + 6], v[8 * k + 7]);
                } else {
                    q = make_uint4(__float_as_uint(v[4 * k]), __float_as_uint(v[4 * k + 1]),
                                   __float_as_uint(v[4 * k + 2]), __float_as_uint(v[4 * k + 3]));
                }
                *reinterpret_cast<uint4*>(dst + 16 * k) = q;
            }
        }
    }
}

template <int C, int XDT, int ODT>
void rotate_launch(const void* x, void* out, const int8_t* signs, uint64_t rows, int inverse, cudaStream_t st)
{
    constexpr int L = C / 8 < 32 ? C / 8 : 32;
    constexpr int RPW = 32 / L;
    const uint64_t warps = (rows + RPW - 1) / RPW;
    const uint64_t blocks = std::max<uint64_t>(1, std::min<uint64_t>((warps + 7) / 8, (uint64_t)sm_count() * 8));
    const float scale = (float)(1.0 / std::sqrt((double)C));
    rotate_kernel<C, XDT, ODT><<<(unsigned)blocks, kRThreads, 0, st>>>(x, out, signs, rows, inverse, scale);
}

template <int C>
void rotate_dtypes(const void* x, int xdt, void* out, int odt, const int8_t* signs, uint64_t rows, int inverse,
                   cudaStream_t st)
{
    if (xdt == KVQ_BF16) {
        if (odt == KVQ_BF16) rotate_launch<C, KVQ_BF16, KVQ_BF16>(x, out, signs, rows, inverse, st);
        else rotate_launch<C, KVQ_BF16, KVQ_F32>(x, out, signs, rows, inverse, st);
    } else {
        if (odt == KVQ_BF16) rotate_launch<C, KVQ_F32, KVQ_BF16>(x, out, signs, rows, inverse, st);
        else rotate_launch<C, KVQ_F32, KVQ_F32>(x, out, signs, rows, inverse, st);
    }
}

}  // namespace

cudaError_t launch_rotate(const void* x, int x_dt, void* out, int out_dt, const int8_t* signs, uint64_t rows,
                          int64_t C, int inverse, cudaStream_t st)
{
    if (rows == 0) return cudaSuccess;
    switch (C) {
    case 32: rotate_dtypes<32>(x, x_dt, out, out_dt, signs, rows, inverse, st); break;
    case 64: rotate_dtypes<64>(x, x_dt, out, out_dt, signs, rows, inverse, st); break;
    case 128: rotate_dtypes<128>(x, x_dt, out, out_dt, signs, rows, inverse, st); break;
    case 256: rotate_dtypes<256>(x, x_dt, out, out_dt, signs, rows, inverse, st); break;
    case 512: rotate_dtypes<512>(x, x_dt, out, out_dt, signs, rows, inverse, st); break;
    default: rotate_dtypes<1024>(x, x_dt, out, out_dt, signs, rows, inverse, st); break;
    }
    return cudaGetLastError();
}

}  // namespace kvq
