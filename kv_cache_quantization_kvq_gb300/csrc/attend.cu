// attend.cu -- decode attention over a quantized KV cache with the
// dequantization fused into the attention read.
//
// Method: "KV cache 压缩：把历史装得更小" §"量化：位置都留着，每个数更短" (the
// attention kernel reads the group-quantized cache, x ~ s * (q - z), and
// dequantizes it; K grouped per channel, V per token), §"让 kernel 接住收益"
// (the byte savings only materialise when the dequantization is fused into the
// attention kernel) and §"K 的误差会改变权重，V 的误差会改变内容" (logit_t =
// q^T k_t / sqrt(d); y = sum_t a_t v_t with a = softmax(logits)).
//
// Work split (one launch plus a small merge): CTA (split, slice o) takes
// kAChunk consecutive tokens of KV slice o and all `G` query heads reading it.
// Each of its warps walks 64 tokens in batches of 32:
//  * scores, lane = token: the K scale of the batch's group (per channel) is
//    folded into the query once per group, A[j][c] = q[j][c] * s[c], and the
//    zero point into the integer-to-float step: the code field read as the
//    float 2^23 + field, minus 2^23 + zeff[c], is code - zp exactly; a token's
//    logit is sum_c A[j][c] * (code[c] - zp[c]) / sqrt(C), one FMA per code
//    and query head;
//  * online softmax in base 2 (running max and rescaled sums);
//  * values, half-warp = token, lane = 8 channels: the batch's V codes and
//    per-token (scale, 2^23 + zeff) are staged in shared memory; each step
//    takes two tokens (one per half-warp), a lane unpacks one packed code
//    word of 8 channels and adds (p_j * s) * (code - zp); the halves are
//    summed at the end.
// The residual tokens (t >= Tq) are read as bf16 rows.  The CTA merges its
// warps and writes (max, sum, unnormalised output) per query head; the merge
// kernel combines the splits of T.
#include <algorithm>

#include "kvq_elem.cuh"

namespace kvq {

namespace {

using namespace elem;

constexpr int kAC = 128;                         // head_dim
constexpr int kAWarps = 4;
constexpr int kAThreads = kAWarps * 32;
constexpr int kATokWarp = 64;                    // tokens per warp and split
constexpr int kAChunk = kAWarps * kATokWarp;     // tokens per split of T
constexpr int kAMaxVG = kAC / 32;                // V groups per row (g >= 32)
constexpr float kTwo23 = 8388608.0f;

struct AttnArgs {
    const float* q;                              // [outer][G][C]
    const uint8_t* kc;                           // [outer][Tq][C*bits/8]
    const void* ks;                              // [outer][ngk][C]
    const void* kz;
    const __nv_bfloat16* kr;                     // [outer][R][C]
    const uint8_t* vc;
    const void* vs;                              // [outer][Tq][ngv]
    const void* vz;
    const __nv_bfloat16* vr;
    int32_t ks_dt, kz_dt, vs_dt, vz_dt;          // zero dtype KVQ_NONE: symmetric
    int32_t k_off, v_off;                        // 2^(bits-1) for two's complement codes, else 0
    int32_t k_signed, v_signed;
    int64_t outer, T, Tq, R;
    int32_t gk, ngk;                             // K: group length along T, groups per slice
    int32_t gv, ngv;                             // V: group length along C, groups per row
    int32_t nsplit;
    float scale2;                                // log2(e) / sqrt(C)
    float* part;                                 // [outer][G][nsplit][2 + C]
};

// The k-th BITS-bit code word (8 codes) of a row held as 16-byte vectors.
template <int BITS>
__device__ __forceinline__ typename CodeWord<BITS>::T word_at(const uint4* v, int k) {
    if constexpr (BITS == 4) {
        const uint4 x = v[k >> 2];
        const int i = k & 3;
        return i == 0 ? x.x : i == 1 ? x.y : i == 2 ? x.z : x.w;
    } else if constexpr (BITS == 8) {
        const uint4 x = v[k >> 1];
        return (k & 1) ? make_uint2(x.z, x.w) : make_uint2(x.x, x.y);
    } else {
        const uint4 x = v[k >> 3];
        const int i = (k & 7) >> 1;
        const uint32_t w = i == 0 ? x.x : i == 1 ? x.y : i == 2 ? x.z : x.w;
        return (uint16_t)((k & 1) ? (w >> 16) : (w & 0xFFFFu));
    }
}

// 16 bytes global -> shared without passing through registers (sm_80+).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

template <int BITS, int G>
__global__ void __launch_bounds__(kAThreads)
attend_split_kernel(const AttnArgs a)
{
    constexpr int kRowB = kAC * BITS / 8;        // packed bytes per token row
    constexpr int kNV = kRowB / 16;              // 16-byte vectors per row
    using W = typename CodeWord<BITS>::T;
    __shared__ __align__(16) float qs[G][kAC];
    // per warp: the queries with the K scales folded in; after the token loop
    // the same warp's unnormalised output (the buffers are never live together)
    __shared__ __align__(16) float A[kAWarps][G][kAC];
    __shared__ __align__(16) float CZ[kAWarps][kAC];                 // 2^23 + zeff of the K group
    __shared__ __align__(16) unsigned char vst[kAWarps][32][kRowB];
    __shared__ __align__(8) float2 vmeta[kAWarps][32][kAMaxVG];    // (scale, 2^23 + zeff) per token and V group
    __shared__ float wm[kAWarps][G], wl[kAWarps][G];
    float (*wo)[G][kAC] = A;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t o = blockIdx.y;
    const int split = blockIdx.x;
    const int64_t T = a.T, Tq = a.Tq;
    for (int i = tid; i < G * kAC; i += kAThreads) qs[i / kAC][i % kAC] = a.q[(o * G) * kAC + i];
    __syncthreads();

    float m[G], ell[G];
    u64 acc_o[G][4];                             // channels c8 .. c8+7 over this half-warp's tokens
#pragma unroll
    for (int j = 0; j < G; ++j) {
        m[j] = -INFINITY;
        ell[j] = 0.0f;
        acc_o[j][0] = acc_o[j][1] = acc_o[j][2] = acc_o[j][3] = 0;
    }
    int cur_gk = -1;
    const int half = lane >> 4;                  // value side: which token of a step
    const int c8 = (lane & 15) * 8;              // this lane's first value channel
    const int vgrp = c8 / a.gv;                  // its V group within a row

    for (int b = 0; b < kATokWarp / 32; ++b) {
        const int64_t t0 = (int64_t)split * kAChunk + warp * kATokWarp + b * 32;
        if (t0 >= T) break;                      // warp-uniform
        const int64_t t = t0 + lane;

        // ---- this batch's V codes: an asynchronous copy to shared memory, in
        // flight while the scores are computed
        const int64_t nq64 = Tq - t0;
        const int nq = nq64 <= 0 ? 0 : (nq64 >= 32 ? 32 : (int)nq64);     // quantized tokens of the batch
        if (nq > 0) {
            const uint4* src = reinterpret_cast<const uint4*>(a.vc + ((uint64_t)o * Tq + t0) * kRowB);
            uint4* dst = reinterpret_cast<uint4*>(&vst[warp][0][0]);
            for (int k = lane; k < nq * kNV; k += 32) cp_async16(dst + k, src + k);
            cp_async_commit();
        }

        // ---- K group constants folded into the queries (once per group)
        if (t0 < Tq) {
            const int gk = (int)(t0 / a.gk);
            if (gk != cur_gk) {
                cur_gk = gk;
#pragma unroll
                for (int mm = 0; mm < kAC / 32; ++mm) {
                    const int c = lane + 32 * mm;
                    const int64_t mi = (o * a.ngk + gk) * kAC + c;
                    const float s = load_meta(a.ks, a.ks_dt, mi);
                    const float z = a.kz_dt == KVQ_NONE ? 0.0f : load_meta(a.kz, a.kz_dt, mi);
                    CZ[warp][c] = __fadd_rn(kTwo23, __fadd_rn((float)a.k_off, z));
#pragma unroll
                    for (int j = 0; j < G; ++j) A[warp][j][c] = __fmul_rn(qs[j][c], s);
                }
                __syncwarp();
            }
        }

        // ---- logits (base 2), lane = token
        float lg[G];
        if (t < Tq) {
            const uint4* crow = reinterpret_cast<const uint4*>(a.kc + ((uint64_t)o * Tq + t) * kRowB);
            uint4 cv[kNV];
#pragma unroll
            for (int k = 0; k < kNV; ++k) cv[k] = __ldcs(crow + k);
            u64 acc[G];
#pragma unroll
            for (int j = 0; j < G; ++j) acc[j] = 0;
#pragma unroll
            for (int w8 = 0; w8 < kAC / 8; ++w8) {
                W cw = word_at<BITS>(cv, w8);
                uint32_t u[8];
                unpack_biased8<BITS>(a.k_signed ? flip_signs<BITS>(cw) : cw, u);
                const float4 z0 = *reinterpret_cast<const float4*>(&CZ[warp][w8 * 8]);
                const float4 z1 = *reinterpret_cast<const float4*>(&CZ[warp][w8 * 8 + 4]);
                const u64 cz[4] = {pk(z0.x, z0.y), pk(z0.z, z0.w), pk(z1.x, z1.y), pk(z1.z, z1.w)};
                u64 f[4];                                     // code - zp, exact
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    f[p] = sub2(pk(__uint_as_float(u[2 * p]), __uint_as_float(u[2 * p + 1])), cz[p]);
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const float4 a0 = *reinterpret_cast<const float4*>(&A[warp][j][w8 * 8]);
                    const float4 a1 = *reinterpret_cast<const float4*>(&A[warp][j][w8 * 8 + 4]);
                    acc[j] = fma2(pk(a0.x, a0.y), f[0], acc[j]);
                    acc[j] = fma2(pk(a0.z, a0.w), f[1], acc[j]);
                    acc[j] = fma2(pk(a1.x, a1.y), f[2], acc[j]);
                    acc[j] = fma2(pk(a1.z, a1.w), f[3], acc[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < G; ++j) lg[j] = __fmul_rn(__fadd_rn(lo_of(acc[j]), hi_of(acc[j])), a.scale2);
        } else if (t < T) {
            const uint4* rrow = reinterpret_cast<const uint4*>(a.kr + ((uint64_t)o * a.R + (t - Tq)) * kAC);
            u64 acc[G];
#pragma unroll
            for (int j = 0; j < G; ++j) acc[j] = 0;
#pragma unroll 4
            for (int k = 0; k < kAC / 8; ++k) {
                const uint4 rv = __ldcs(rrow + k);
                const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const u64 r2 = widen_bf16x2(rw[p]);
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        const float2 q2 = *reinterpret_cast<const float2*>(&qs[j][k * 8 + 2 * p]);
                        acc[j] = fma2(pk(q2.x, q2.y), r2, acc[j]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < G; ++j) lg[j] = __fmul_rn(__fadd_rn(lo_of(acc[j]), hi_of(acc[j])), a.scale2);
        } else {
#pragma unroll
            for (int j = 0; j < G; ++j) lg[j] = -INFINITY;
        }

        // ---- online softmax
        float p[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const float mn = fmaxf(m[j], warp_max(lg[j]));
            float alpha = 1.0f;
            if (mn == -INFINITY) {
                p[j] = 0.0f;
            } else {
                alpha = exp2f(m[j] - mn);                // 0 while nothing was seen
                p[j] = exp2f(lg[j] - mn);                // 0 for masked tokens
            }
            m[j] = mn;
            ell[j] = __fmaf_rn(ell[j], alpha, p[j]);
            const u64 al2 = pk(alpha, alpha);
#pragma unroll
            for (int k = 0; k < 4; ++k) acc_o[j][k] = mul2(acc_o[j][k], al2);
        }

        // ---- per-token V constants to shared memory; the staged codes have landed
        if (nq > 0) {
            if (lane < nq) {
                for (int g = 0; g < a.ngv; ++g) {
                    const int64_t mi = (o * Tq + t) * a.ngv + g;
                    const float sv = load_meta(a.vs, a.vs_dt, mi);
                    const float zv = a.vz_dt == KVQ_NONE ? 0.0f : load_meta(a.vz, a.vz_dt, mi);
                    vmeta[warp][lane][g] = make_float2(sv, __fadd_rn(kTwo23, __fadd_rn((float)a.v_off, zv)));
                }
            }
            cp_async_wait_all();
        }
        __syncwarp();

        // ---- values: step i takes token 2i + half, lane = 8 channels
        const int nt = T - t0 >= 32 ? 32 : (int)(T - t0);
        for (int i = 0; i < (nt + 1) / 2; ++i) {
            const int ti = 2 * i + half;
            float pi[G];
#pragma unroll
            for (int j = 0; j < G; ++j) pi[j] = __shfl_sync(0xFFFFFFFFu, p[j], ti & 31);
            if (ti < nq) {
                W cw = *reinterpret_cast<const W*>(&vst[warp][ti][c8 * BITS / 8]);
                uint32_t u[8];
                unpack_biased8<BITS>(a.v_signed ? flip_signs<BITS>(cw) : cw, u);
                const float2 sm = vmeta[warp][ti][vgrp];
                const u64 cz = pk(sm.y, sm.y);
                u64 f[4];                                     // code - zp, exact
#pragma unroll
                for (int k = 0; k < 4; ++k) f[k] = sub2(pk(__uint_as_float(u[2 * k]), __uint_as_float(u[2 * k + 1])), cz);
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const float w = __fmul_rn(pi[j], sm.x);
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc_o[j][k] = fma2(f[k], pk(w, w), acc_o[j][k]);
                }
            } else if (ti < nt) {
                const uint4 rv = __ldcs(reinterpret_cast<const uint4*>(a.vr + ((uint64_t)o * a.R + (t0 + ti - Tq)) * kAC + c8));
                const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                for (int j = 0; j < G; ++j) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc_o[j][k] = fma2(widen_bf16x2(rw[k]), pk(pi[j], pi[j]), acc_o[j][k]);
                }
            }
        }
        __syncwarp();
    }

    // ---- merge the warps of the CTA, write this split's partial
    __syncwarp();
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const float l = warp_sum(ell[j]);
        if (lane == 0) { wm[warp][j] = m[j]; wl[warp][j] = l; }
#pragma unroll
        for (int k = 0; k < 4; ++k)                   // the two half-warps' tokens
            acc_o[j][k] = add2(acc_o[j][k], __shfl_xor_sync(0xFFFFFFFFu, acc_o[j][k], 16));
        if (half == 0) {
            *reinterpret_cast<float4*>(&wo[warp][j][c8]) =
                make_float4(lo_of(acc_o[j][0]), hi_of(acc_o[j][0]), lo_of(acc_o[j][1]), hi_of(acc_o[j][1]));
            *reinterpret_cast<float4*>(&wo[warp][j][c8 + 4]) =
                make_float4(lo_of(acc_o[j][2]), hi_of(acc_o[j][2]), lo_of(acc_o[j][3]), hi_of(acc_o[j][3]));
        }
    }
    __syncthreads();
    for (int j = 0; j < G; ++j) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAWarps; ++w) M = fmaxf(M, wm[w][j]);
        float L = 0.0f, y = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kAWarps; ++w) {
                const float e = exp2f(wm[w][j] - M);
                L = __fmaf_rn(wl[w][j], e, L);
                y = __fmaf_rn(wo[w][j][tid], e, y);
            }
        }
        float* dst = a.part + ((o * G + j) * a.nsplit + split) * (2 + kAC);
        if (tid == 0) { dst[0] = M; dst[1] = L; }
        dst[2 + tid] = y;
    }
}

// out[o][j][c] = sum_s y_s[c] 2^(m_s - M) / sum_s l_s 2^(m_s - M)
__global__ void __launch_bounds__(kAC)
attend_merge_kernel(const float* part, int nsplit, float* out)
{
    const int64_t oj = blockIdx.x;
    const int c = threadIdx.x;
    const float* p = part + oj * nsplit * (2 + kAC);
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, p[s * (2 + kAC)]);
    float L = 0.0f, y = 0.0f;
    if (M != -INFINITY) {
        for (int s = 0; s < nsplit; ++s) {
            const float* q = p + s * (2 + kAC);
            const float e = exp2f(q[0] - M);
            L = __fmaf_rn(q[1], e, L);
            y = __fmaf_rn(q[2 + c], e, y);
        }
    }
    out[oj * kAC + c] = L > 0.0f ? __fdiv_rn(y, L) : 0.0f;
}

template <int BITS>
void attend_typed(const AttnArgs& a, int G, float* out, cudaStream_t st)
{
    const dim3 grid((unsigned)a.nsplit, (unsigned)a.outer);
    switch (G) {
    case 1: attend_split_kernel<BITS, 1><<<grid, kAThreads, 0, st>>>(a); break;
    case 2: attend_split_kernel<BITS, 2><<<grid, kAThreads, 0, st>>>(a); break;
    case 4: attend_split_kernel<BITS, 4><<<grid, kAThreads, 0, st>>>(a); break;
    default: attend_split_kernel<BITS, 8><<<grid, kAThreads, 0, st>>>(a); break;
    }
    attend_merge_kernel<<<(unsigned)(a.outer * G), kAC, 0, st>>>(a.part, a.nsplit, out);
}

}  // namespace

int64_t attend_splits(int64_t T) { return (T + kAChunk - 1) / kAChunk; }

size_t attend_workspace(int64_t outer, int64_t T, int64_t group)
{
    return (size_t)outer * (size_t)group * (size_t)attend_splits(T) * (2 + kAC) * sizeof(float);
}

cudaError_t launch_attend(const AttendArgs& x, cudaStream_t st)
{
    const QSpec& k = x.k;
    const QSpec& v = x.v;
    AttnArgs a;
    a.q = x.q;
    a.kc = static_cast<const uint8_t*>(x.k_codes);
    a.ks = x.k_scale;
    a.kz = x.k_zero;
    a.kr = static_cast<const __nv_bfloat16*>(x.k_resid);
    a.vc = static_cast<const uint8_t*>(x.v_codes);
    a.vs = x.v_scale;
    a.vz = x.v_zero;
    a.vr = static_cast<const __nv_bfloat16*>(x.v_resid);
    a.ks_dt = k.scale_dt;
    a.kz_dt = k.mode == KVQ_ASYM ? k.zero_dt : KVQ_NONE;
    a.vs_dt = v.scale_dt;
    a.vz_dt = v.mode == KVQ_ASYM ? v.zero_dt : KVQ_NONE;
    a.k_signed = k.is_signed;
    a.v_signed = v.is_signed;
    a.k_off = k.is_signed ? 1 << (k.bits - 1) : 0;
    a.v_off = v.is_signed ? 1 << (v.bits - 1) : 0;
    a.outer = k.outer;
    a.T = k.T;
    a.Tq = k.Tq;
    a.R = k.R;
    a.gk = (int32_t)k.g;
    a.ngk = (int32_t)k.ngroups;
    a.gv = (int32_t)v.g;
    a.ngv = (int32_t)v.ngroups;
    a.nsplit = (int32_t)attend_splits(k.T);
    a.scale2 = (float)(1.4426950408889634 / 11.313708498984761);   // log2(e) / sqrt(128)
    a.part = static_cast<float*>(x.ws);
    if (a.outer == 0) return cudaSuccess;
    const int G = (int)x.group;
    switch (k.bits) {
    case 8: attend_typed<8>(a, G, x.out, st); break;
    case 4: attend_typed<4>(a, G, x.out, st); break;
    default: attend_typed<2>(a, G, x.out, st); break;
    }
    return cudaGetLastError();
}

}  // namespace kvq
