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

// ======================================================================
// Tensor-core path (2- and 4-bit codes): both contractions of a 16-token
// tile on mma.sync.m16n8k16 (bf16 operands, float32 accumulation).
//
//  * scores, D[16 x 8] = Q'[16 x 128] . K^T[128 x 8] per 8 tokens: the rows
//    of Q' are the 8 query heads' q * s (K scale of the channel folded in,
//    rounded to float32 as in the scalar path) split into bf16 hi (rows 0-7)
//    and lo = RN_bf16(x - hi) (rows 8-15), so hi + lo carries x to 2^-16
//    (bf16 significands have 8 bits);
//    the columns of K^T are code fields minus (off + zp), small integers that
//    bf16 holds exactly (checked per group: |off + zp| <= 112).  A channel
//    order chosen per 32-bit code word makes every B register one
//    mask-and-or of a code word: fields a and a + F/2 of a word (F fields per
//    word) land in the two halves as the bf16 values 128 + field, and one
//    bf16x2 subtraction of the pair (128 + off + zp) leaves field - off - zp.
//    Row g of the result is head g's hi part, row g + 8 its lo part: the
//    logit is their sum.
//  * The score fragment of a lane holds head g at tokens 2*tig, 2*tig + 1,
//    2*tig + 8, 2*tig + 9 -- exactly the A fragment of the value product,
//    so the probabilities never leave registers: Y[16 x 128] = P'[16 x 16] .
//    V[16 x 128] with P' = p * s_v(token, V group) split hi / lo the same
//    way and V the value fields minus (off + zp) per token.
//  * A tile whose tokens are all residual (or past T) takes the same two
//    products with the bf16 rows as operands; a tile straddling the
//    quantized / residual boundary, or a group whose zero points bf16 cannot
//    hold exactly, takes a float32 scalar path with the same register layout
//    (exact products, one FMA each).
// The online softmax, the merge of the warps of a CTA and the split
// partials are those of the scalar kernel above.
constexpr int kTcTile = 16;
constexpr int kTcTiles = kATokWarp / kTcTile;          // tiles per warp span

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// a - b on bf16 pairs (exact for the small integers used here)
__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// hi = RN_bf16(x), lo = RN_bf16(x - hi) for a pair (low element first)
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo)
{
    hi = pack_bf16x2(x0, x1);
    lo = pack_bf16x2(__fsub_rn(x0, lo_f(hi)), __fsub_rn(x1, hi_f(hi)));
}

// field of channel c in a code row held as 32-bit words
template <int BITS>
__device__ __forceinline__ uint32_t field_at(const uint32_t* row, int c)
{
    return (row[(c * BITS) >> 5] >> ((c * BITS) & 31)) & ((1u << BITS) - 1u);
}

template <int BITS, int G, int GV>
__global__ void __launch_bounds__(kAThreads, 3)
attend_tc_kernel(const AttnArgs a)
{
    constexpr int kRowB = kAC * BITS / 8;        // packed bytes per token row
    constexpr int kRowW = kRowB / 4;             // 32-bit words per row
    constexpr int kWpl = kRowW / 4;              // words of a row per lane of a quad
    constexpr int kF = 32 / BITS;                // fields per word
    constexpr int kKps = kF / 4;                 // k-steps per word (two pairs each)
    constexpr uint32_t kMask2 = BITS == 4 ? 0x000F000Fu : 0x00030003u;
    constexpr uint32_t kOne28 = 0x43004300u;     // bf16 128.0 in both halves
    constexpr int kVRowW = kRowW + 4;            // V rows padded: lanes of a quad read rows 2 apart without bank conflicts
    // dynamic shared memory (TcSmem<BITS> bytes), carved in this order:
    //   qs    [8][kAC] float                   queries, heads >= G zero
    //   kst   [kAWarps][kATokWarp][kRowW] u32  K code rows of each warp's span
    //   vst   [kAWarps][kATokWarp][kVRowW] u32 V code rows (padded)
    //   vm    [kAWarps][kATokWarp][kAMaxVG]    (scale, 128 + off + zp) per token and V group
    //   ksc, kcz [kAWarps][kAC] float          K group: scale, 128 + off + zp per channel
    //   pbuf  [kAWarps][8][kTcTile] float      probabilities of a scalar tile
    //   wm, wl [kAWarps][8] float
    // and wo [kAWarps][8][kAC] float (the warps' outputs) over kst / vst after the token loop
    extern __shared__ __align__(16) unsigned char tc_smem[];
    float (*qs)[kAC] = reinterpret_cast<float (*)[kAC]>(tc_smem);
    uint32_t (*kst)[kATokWarp][kRowW] = reinterpret_cast<uint32_t (*)[kATokWarp][kRowW]>(tc_smem + 8 * kAC * 4);
    uint32_t (*vst)[kATokWarp][kVRowW] = reinterpret_cast<uint32_t (*)[kATokWarp][kVRowW]>(kst + kAWarps);
    float2 (*vm)[kATokWarp][kAMaxVG] = reinterpret_cast<float2 (*)[kATokWarp][kAMaxVG]>(vst + kAWarps);
    float (*ksc)[kAC] = reinterpret_cast<float (*)[kAC]>(vm + kAWarps);
    float (*kcz)[kAC] = ksc + kAWarps;
    float (*pbuf)[8][kTcTile] = reinterpret_cast<float (*)[8][kTcTile]>(kcz + kAWarps);
    float (*wm)[8] = reinterpret_cast<float (*)[8]>(pbuf + kAWarps);
    float (*wl)[8] = wm + kAWarps;
    float (*wo)[8][kAC] = reinterpret_cast<float (*)[8][kAC]>(kst);   // reused after the token loop
    static_assert(kAWarps * kATokWarp * (kRowW + kVRowW) * 4 >= kAWarps * 8 * kAC * 4, "wo must fit over kst / vst");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, tig = lane & 3;     // mma fragment coordinates
    const int64_t o = blockIdx.y;
    const int split = blockIdx.x;
    const int64_t T = a.T, Tq = a.Tq;
    for (int i = tid; i < 8 * kAC; i += kAThreads) {
        const int j = i / kAC;
        qs[j][i % kAC] = j < G ? a.q[(o * G + j) * kAC + i % kAC] : 0.0f;
    }
    // ---- this warp's span: its quantized K / V code rows and V constants
    const int64_t s0 = (int64_t)split * kAChunk + warp * kATokWarp;
    const int64_t nq64 = Tq - s0;
    const int nq = nq64 <= 0 ? 0 : (nq64 >= kATokWarp ? kATokWarp : (int)nq64);   // quantized tokens of the span
    if (nq > 0) {
        const uint4* ksrc = reinterpret_cast<const uint4*>(a.kc + ((uint64_t)o * Tq + s0) * kRowB);
        const uint4* vsrc = reinterpret_cast<const uint4*>(a.vc + ((uint64_t)o * Tq + s0) * kRowB);
        uint4* kdst = reinterpret_cast<uint4*>(&kst[warp][0][0]);
        constexpr int kVec = kRowB / 16;         // 16-byte pieces per row
        for (int k = lane; k < nq * kVec; k += 32) {
            cp_async16(kdst + k, ksrc + k);
            cp_async16(reinterpret_cast<uint4*>(&vst[warp][k / kVec][0]) + (k % kVec), vsrc + k);
        }
        cp_async_commit();
        for (int t = lane; t < nq; t += 32)
            for (int vg = 0; vg < a.ngv; ++vg) {
                const int64_t mi = (o * Tq + s0 + t) * a.ngv + vg;
                const float sv = load_meta(a.vs, a.vs_dt, mi);
                const float zv = a.vz_dt == KVQ_NONE ? 0.0f : load_meta(a.vz, a.vz_dt, mi);
                vm[warp][t][vg] = make_float2(sv, __fadd_rn(128.0f, __fadd_rn((float)a.v_off, zv)));
            }
        cp_async_wait_all();
        if (a.k_signed || a.v_signed) {
            // two's complement fields -> offset binary (field + 2^(BITS-1)) in place
            __syncwarp();
            constexpr uint32_t kFlip = BITS == 4 ? 0x88888888u : 0xAAAAAAAAu;
            uint32_t* kw = &kst[warp][0][0];
            for (int k = lane; k < nq * kRowW; k += 32) {
                if (a.k_signed) kw[k] ^= kFlip;
                if (a.v_signed) vst[warp][k / kRowW][k % kRowW] ^= kFlip;
            }
        }
    }
    __syncthreads();
    // V exactness of the span's tokens, one bit per token (lane t: tokens t and t + 32)
    uint32_t vexact_lo, vexact_hi;
    {
        bool e0 = true, e1 = true;
        for (int vg = 0; vg < a.ngv; ++vg) {
            if (lane < nq) e0 = e0 && fabsf(vm[warp][lane][vg].y - 128.0f) <= 112.0f;
            if (lane + 32 < nq) e1 = e1 && fabsf(vm[warp][lane + 32][vg].y - 128.0f) <= 112.0f;
        }
        vexact_lo = __ballot_sync(0xFFFFFFFFu, e0);
        vexact_hi = __ballot_sync(0xFFFFFFFFu, e1);
    }

    float yacc[16][4];                           // n-tile nt: head g hi part (0, 1) and lo part (2, 3), channels 8nt + 2tig + {0, 1}
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) yacc[nt][0] = yacc[nt][1] = yacc[nt][2] = yacc[nt][3] = 0.0f;
    float m = -INFINITY, ell = 0.0f;             // head g; ell over this lane's tokens
    int cur_gk = -1;
    bool k_exact = false;
    uint32_t qa[8][4];                           // Q' fragments of the current K group
    uint32_t kzp[8][2];                          // (128 + off + zp) pairs of the b0 / b1 channels
    const int vshift = BITS == 4 ? 4 * g : 2 * g;  // bit of channel 8nt + g within its (byte-aligned) word slot

    for (int tile = 0; tile < kTcTiles; ++tile) {
        const int64_t t0 = s0 + tile * kTcTile;
        if (t0 >= T) break;                      // warp-uniform
        const int u0 = tile * kTcTile;           // first row of the tile within the span
        bool tc = false;
        if (t0 + kTcTile <= Tq) {
            const int gk = (int)(t0 / a.gk);
            if (gk != cur_gk) {
                // K group constants: this warp stages them, each lane derives its fragments
                cur_gk = gk;
                __syncwarp();
#pragma unroll
                for (int mm = 0; mm < kAC / 32; ++mm) {
                    const int c = lane + 32 * mm;
                    const int64_t mi = (o * a.ngk + gk) * kAC + c;
                    ksc[warp][c] = load_meta(a.ks, a.ks_dt, mi);
                    const float z = a.kz_dt == KVQ_NONE ? 0.0f : load_meta(a.kz, a.kz_dt, mi);
                    kcz[warp][c] = __fadd_rn(128.0f, __fadd_rn((float)a.k_off, z));
                }
                __syncwarp();
                bool ok = true;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int W = kWpl * tig + kk / kKps, j = kk % kKps;
                    const int c00 = W * kF + 2 * j, c01 = c00 + kF / 2, c10 = c00 + 1, c11 = c01 + 1;
                    uint32_t h0, l0, h1, l1;
                    split_bf16x2(__fmul_rn(qs[g][c00], ksc[warp][c00]), __fmul_rn(qs[g][c01], ksc[warp][c01]), h0, l0);
                    split_bf16x2(__fmul_rn(qs[g][c10], ksc[warp][c10]), __fmul_rn(qs[g][c11], ksc[warp][c11]), h1, l1);
                    qa[kk][0] = h0; qa[kk][1] = l0; qa[kk][2] = h1; qa[kk][3] = l1;
                    kzp[kk][0] = pack_bf16x2(kcz[warp][c00], kcz[warp][c01]);
                    kzp[kk][1] = pack_bf16x2(kcz[warp][c10], kcz[warp][c11]);
                    ok = ok && fabsf(kcz[warp][c00] - 128.0f) <= 112.0f && fabsf(kcz[warp][c01] - 128.0f) <= 112.0f &&
                         fabsf(kcz[warp][c10] - 128.0f) <= 112.0f && fabsf(kcz[warp][c11] - 128.0f) <= 112.0f;
                }
                k_exact = __all_sync(0xFFFFFFFFu, ok);
            }
            const uint32_t vmask = ((u0 < 32 ? vexact_lo : vexact_hi) >> (u0 & 31)) & 0xFFFFu;
            tc = k_exact && vmask == 0xFFFFu;
        }

        const bool rt = t0 >= Tq;                // every token residual (or past T): bf16 rows
        // ---- logits of head g at tokens u0 + {2tig, 2tig + 1, 8 + 2tig, 9 + 2tig}
        float lg[4];
        if (rt) {
            // rows t0 + g and t0 + 8 + g; channels in natural order: k-step kk
            // takes 16kk + 2tig, +1 (b0) and 16kk + 2tig + 8, +9 (b1)
            float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const int64_t ta = t0 + g, tb = t0 + 8 + g;
            const uint32_t* ka = reinterpret_cast<const uint32_t*>(a.kr + ((uint64_t)o * a.R + (ta - Tq)) * kAC);
            const uint32_t* kb = reinterpret_cast<const uint32_t*>(a.kr + ((uint64_t)o * a.R + (tb - Tq)) * kAC);
            uint32_t kra[16], krb[16];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                kra[2 * kk] = ta < T ? __ldcs(ka + 8 * kk + tig) : 0u;
                kra[2 * kk + 1] = ta < T ? __ldcs(ka + 8 * kk + 4 + tig) : 0u;
                krb[2 * kk] = tb < T ? __ldcs(kb + 8 * kk + tig) : 0u;
                krb[2 * kk + 1] = tb < T ? __ldcs(kb + 8 * kk + 4 + tig) : 0u;
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int c0 = 16 * kk + 2 * tig;
                uint32_t qf[4];
                split_bf16x2(qs[g][c0], qs[g][c0 + 1], qf[0], qf[1]);
                split_bf16x2(qs[g][c0 + 8], qs[g][c0 + 9], qf[2], qf[3]);
                mma_bf16_16816(d0, qf, kra[2 * kk], kra[2 * kk + 1]);
                mma_bf16_16816(d1, qf, krb[2 * kk], krb[2 * kk + 1]);
            }
            const int64_t tt[4] = {t0 + 2 * tig, t0 + 2 * tig + 1, t0 + 8 + 2 * tig, t0 + 9 + 2 * tig};
            lg[0] = tt[0] < T ? __fmul_rn(__fadd_rn(d0[0], d0[2]), a.scale2) : -INFINITY;
            lg[1] = tt[1] < T ? __fmul_rn(__fadd_rn(d0[1], d0[3]), a.scale2) : -INFINITY;
            lg[2] = tt[2] < T ? __fmul_rn(__fadd_rn(d1[0], d1[2]), a.scale2) : -INFINITY;
            lg[3] = tt[3] < T ? __fmul_rn(__fadd_rn(d1[1], d1[3]), a.scale2) : -INFINITY;
        } else if (tc) {
            float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const uint32_t* r0 = &kst[warp][u0 + g][kWpl * tig];
            const uint32_t* r1 = &kst[warp][u0 + 8 + g][kWpl * tig];
            uint32_t w0[kWpl], w1[kWpl];
#pragma unroll
            for (int i = 0; i < kWpl; ++i) { w0[i] = r0[i]; w1[i] = r1[i]; }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int i = kk / kKps, j = kk % kKps;
                const uint32_t b00 = bsub2(((w0[i] >> (2 * j * BITS)) & kMask2) | kOne28, kzp[kk][0]);
                const uint32_t b01 = bsub2(((w0[i] >> ((2 * j + 1) * BITS)) & kMask2) | kOne28, kzp[kk][1]);
                mma_bf16_16816(d0, qa[kk], b00, b01);
                const uint32_t b10 = bsub2(((w1[i] >> (2 * j * BITS)) & kMask2) | kOne28, kzp[kk][0]);
                const uint32_t b11 = bsub2(((w1[i] >> ((2 * j + 1) * BITS)) & kMask2) | kOne28, kzp[kk][1]);
                mma_bf16_16816(d1, qa[kk], b10, b11);
            }
            lg[0] = __fmul_rn(__fadd_rn(d0[0], d0[2]), a.scale2);
            lg[1] = __fmul_rn(__fadd_rn(d0[1], d0[3]), a.scale2);
            lg[2] = __fmul_rn(__fadd_rn(d1[0], d1[2]), a.scale2);
            lg[3] = __fmul_rn(__fadd_rn(d1[1], d1[3]), a.scale2);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int u = u0 + (e < 2 ? 2 * tig + e : 8 + 2 * tig + (e - 2));
                const int64_t t = s0 + u;
                float acc = 0.0f;
                if (t >= T) {
                    acc = -INFINITY;
                } else if (t >= Tq) {
                    const __nv_bfloat16* rr = a.kr + ((uint64_t)o * a.R + (t - Tq)) * kAC;
                    for (int c = 0; c < kAC; ++c) acc = __fmaf_rn(qs[g][c], __bfloat162float(rr[c]), acc);
                    acc = __fmul_rn(acc, a.scale2);
                } else {
                    const int gk = (int)(t / a.gk);
                    for (int c = 0; c < kAC; ++c) {
                        const int64_t mi = (o * a.ngk + gk) * kAC + c;
                        const float sk = load_meta(a.ks, a.ks_dt, mi);
                        const float zk = a.kz_dt == KVQ_NONE ? 0.0f : load_meta(a.kz, a.kz_dt, mi);
                        const float f = __fsub_rn((float)field_at<BITS>(&kst[warp][u][0], c),
                                                  __fadd_rn((float)a.k_off, zk));   // code - zp, exact
                        acc = __fmaf_rn(__fmul_rn(qs[g][c], sk), f, acc);
                    }
                    acc = __fmul_rn(acc, a.scale2);
                }
                lg[e] = acc;
            }
        }

        // ---- online softmax of head g (the four lanes of a quad share it)
        float mt = fmaxf(fmaxf(lg[0], lg[1]), fmaxf(lg[2], lg[3]));
        mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(0xFFFFFFFFu, mt, 2));
        const float mn = fmaxf(m, mt);
        float p[4], alpha = 1.0f;
        if (mn == -INFINITY) {
            p[0] = p[1] = p[2] = p[3] = 0.0f;
        } else {
            alpha = exp2f(m - mn);               // 0 while nothing was seen
#pragma unroll
            for (int e = 0; e < 4; ++e) p[e] = exp2f(lg[e] - mn);   // 0 for tokens past T
        }
        m = mn;
        ell = __fmaf_rn(ell, alpha, __fadd_rn(__fadd_rn(p[0], p[1]), __fadd_rn(p[2], p[3])));
        if (__any_sync(0xFFFFFFFFu, alpha != 1.0f)) {
            const u64 al2 = pk(alpha, alpha);
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const u64 x01 = mul2(pk(yacc[nt][0], yacc[nt][1]), al2);
                const u64 x23 = mul2(pk(yacc[nt][2], yacc[nt][3]), al2);
                yacc[nt][0] = lo_of(x01); yacc[nt][1] = hi_of(x01);
                yacc[nt][2] = lo_of(x23); yacc[nt][3] = hi_of(x23);
            }
        }

        // ---- values
        const int ua = u0 + 2 * tig, ub = ua + 1, uc = ua + 8, ud = ua + 9;   // this lane's tokens
        if (rt) {
            // P unscaled (hi / lo); B pairs tokens (2tig, 2tig + 1) and (2tig + 8, 2tig + 9) at channel 8nt + g
            uint32_t pf[4];
            split_bf16x2(p[0], p[1], pf[0], pf[1]);
            split_bf16x2(p[2], p[3], pf[2], pf[3]);
            const uint16_t* vr = reinterpret_cast<const uint16_t*>(a.vr);
            const int64_t tt[4] = {t0 + 2 * tig, t0 + 2 * tig + 1, t0 + 8 + 2 * tig, t0 + 9 + 2 * tig};
            const uint16_t* rows[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                rows[e] = tt[e] < T ? vr + ((uint64_t)o * a.R + (tt[e] - Tq)) * kAC + g : nullptr;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                uint32_t h[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) h[e] = rows[e] ? (uint32_t)__ldcs(rows[e] + 8 * nt) : 0u;
                mma_bf16_16816(yacc[nt], pf, h[0] | (h[1] << 16), h[2] | (h[3] << 16));
            }
        } else if (tc) {
            uint32_t pa[4], za = 0, zc = 0;      // P' fragment and (128 + off + zp) pairs of the current V group
            const uint4* ra = reinterpret_cast<const uint4*>(&vst[warp][ua][0]);
            const uint4* rb = reinterpret_cast<const uint4*>(&vst[warp][ub][0]);
            const uint4* rc = reinterpret_cast<const uint4*>(&vst[warp][uc][0]);
            const uint4* rd = reinterpret_cast<const uint4*>(&vst[warp][ud][0]);
            // channel 8nt + g sits in word nt (4-bit) or nt / 2 (2-bit) at bit vshift (+16 for odd nt, 2-bit)
            const uint32_t byte = (uint32_t)(vshift >> 3);
            const uint32_t sel = byte | (byte << 4) | ((4u + byte) << 8) | ((4u + byte) << 12);
            const uint32_t sel16 = sel + 0x2222u;            // the same two bytes 16 bits up (2-bit, odd nt)
            const int sh = vshift & 7;
#pragma unroll
            for (int q4 = 0; q4 < kRowW / 4; ++q4) {
                const uint4 wa = ra[q4], wb = rb[q4], wc = rc[q4], wd = rd[q4];
                const uint32_t wav[4] = {wa.x, wa.y, wa.z, wa.w}, wbv[4] = {wb.x, wb.y, wb.z, wb.w};
                const uint32_t wcv[4] = {wc.x, wc.y, wc.z, wc.w}, wdv[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
                for (int k4 = 0; k4 < 4 * (32 / (8 * BITS)); ++k4) {
                    const int nt = BITS == 4 ? 4 * q4 + k4 : 8 * q4 + k4;
                    const int wi = BITS == 4 ? k4 : k4 >> 1;         // word within the 16-byte piece
                    const uint32_t sl = (BITS == 2 && (k4 & 1)) ? sel16 : sel;
                    constexpr int kNtPerGroup = GV / 8;      // n-tiles of one V group (static after unrolling)
                    const int vg = nt / kNtPerGroup;
                    if (nt % kNtPerGroup == 0) {
                        split_bf16x2(__fmul_rn(p[0], vm[warp][ua][vg].x), __fmul_rn(p[1], vm[warp][ub][vg].x), pa[0], pa[1]);
                        split_bf16x2(__fmul_rn(p[2], vm[warp][uc][vg].x), __fmul_rn(p[3], vm[warp][ud][vg].x), pa[2], pa[3]);
                        za = pack_bf16x2(vm[warp][ua][vg].y, vm[warp][ub][vg].y);
                        zc = pack_bf16x2(vm[warp][uc][vg].y, vm[warp][ud][vg].y);
                    }
                    const uint32_t x0 = __byte_perm(wav[wi], wbv[wi], sl);
                    const uint32_t x1 = __byte_perm(wcv[wi], wdv[wi], sl);
                    const uint32_t b0 = bsub2(((x0 >> sh) & kMask2) | kOne28, za);
                    const uint32_t b1 = bsub2(((x1 >> sh) & kMask2) | kOne28, zc);
                    mma_bf16_16816(yacc[nt], pa, b0, b1);
                }
            }
        } else {
            // every probability of head g in the tile, then exact float32 products
            pbuf[warp][g][2 * tig] = p[0];
            pbuf[warp][g][2 * tig + 1] = p[1];
            pbuf[warp][g][8 + 2 * tig] = p[2];
            pbuf[warp][g][9 + 2 * tig] = p[3];
            __syncwarp();
            for (int uu = 0; uu < kTcTile; ++uu) {
                const int64_t t = t0 + uu;
                if (t >= T) break;
                const float pt = pbuf[warp][g][uu];
                const int u = u0 + uu;
#pragma unroll
                for (int nt = 0; nt < 16; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int c = 8 * nt + 2 * tig + e;
                        float v;
                        if (t >= Tq) {
                            v = __bfloat162float(a.vr[((uint64_t)o * a.R + (t - Tq)) * kAC + c]);
                        } else {
                            const float2 sm = vm[warp][u][c / GV];
                            v = __fmul_rn(__fsub_rn((float)field_at<BITS>(&vst[warp][u][0], c), __fsub_rn(sm.y, 128.0f)), sm.x);
                        }
                        yacc[nt][e] = __fmaf_rn(pt, v, yacc[nt][e]);
                    }
            }
            __syncwarp();
        }
    }

    // ---- merge the warps of the CTA, write this split's partial
    ell = __fadd_rn(ell, __shfl_xor_sync(0xFFFFFFFFu, ell, 1));
    ell = __fadd_rn(ell, __shfl_xor_sync(0xFFFFFFFFu, ell, 2));
    if (tig == 0) { wm[warp][g] = m; wl[warp][g] = ell; }
    __syncthreads();                             // wo overlays every warp's code rows
#pragma unroll
    for (int nt = 0; nt < 16; ++nt)
        *reinterpret_cast<float2*>(&wo[warp][g][8 * nt + 2 * tig]) =
            make_float2(__fadd_rn(yacc[nt][0], yacc[nt][2]), __fadd_rn(yacc[nt][1], yacc[nt][3]));
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

// out[o][j][c] = sum_s y_s[c] 2^(m_s - M) / sum_s l_s 2^(m_s - M).  Warp 0
// reads every split's (m_s, l_s) once and leaves M, the denominator and the
// weights 2^(m_s - M) of the first kMergeMaxSplits splits in shared memory
// (later splits' weights are recomputed where used); then each thread (one
// channel) sums the splits with independent loads.
constexpr int kMergeMaxSplits = 1024;

__global__ void __launch_bounds__(kAC)
attend_merge_kernel(const float* part, int nsplit, float* out)
{
    __shared__ float wt[kMergeMaxSplits];
    __shared__ float s_M, s_L;
    const int64_t oj = blockIdx.x;
    const int c = threadIdx.x;
    const float* p = part + oj * nsplit * (2 + kAC);
    if (c < 32) {
        float M = -INFINITY;
        for (int s = c; s < nsplit; s += 32) M = fmaxf(M, __ldcg(p + (int64_t)s * (2 + kAC)));
        M = warp_max(M);
        float L = 0.0f;
        for (int s = c; s < nsplit; s += 32) {
            const float e = M == -INFINITY ? 0.0f : exp2f(__ldcg(p + (int64_t)s * (2 + kAC)) - M);
            if (s < kMergeMaxSplits) wt[s] = e;
            L = __fmaf_rn(__ldcg(p + (int64_t)s * (2 + kAC) + 1), e, L);
        }
        L = warp_sum(L);
        if (c == 0) { s_M = M; s_L = L; }
    }
    __syncthreads();
    const float M = s_M, L = s_L;
    float y = 0.0f;
    for (int s = 0; s < nsplit; ++s) {
        const float* ps = p + (int64_t)s * (2 + kAC);
        const float e = s < kMergeMaxSplits ? wt[s] : (M == -INFINITY ? 0.0f : exp2f(__ldcg(ps) - M));
        y = __fmaf_rn(__ldcg(ps + 2 + c), e, y);
    }
    out[oj * kAC + c] = L > 0.0f ? __fdiv_rn(y, L) : 0.0f;
}

// dynamic shared memory of attend_tc_kernel<BITS, G>
template <int BITS>
constexpr int tc_smem_bytes()
{
    return 8 * kAC * 4 + kAWarps * kATokWarp * (2 * (kAC * BITS / 8) + 16) + kAWarps * kATokWarp * kAMaxVG * 8 +
           2 * kAWarps * kAC * 4 + kAWarps * 8 * kTcTile * 4 + 2 * kAWarps * 8 * 4;
}

template <int BITS, int G, int GV>
void tc_launch_gv(const AttnArgs& a, dim3 grid, cudaStream_t st)
{
    constexpr int smem = tc_smem_bytes<BITS>();
    // three CTAs per SM need the largest carve-out (3 x ~68 KB)
    if (ensure_kernel_attrs(reinterpret_cast<const void*>(attend_tc_kernel<BITS, G, GV>), smem, false, true) !=
        cudaSuccess)
        return;
    attend_tc_kernel<BITS, G, GV><<<grid, kAThreads, smem, st>>>(a);
}

template <int BITS, int G>
void tc_launch(const AttnArgs& a, dim3 grid, cudaStream_t st)
{
    switch (a.gv) {                              // V groups of 32, 64 or 128 channels (checked by the API)
    case 32: tc_launch_gv<BITS, G, 32>(a, grid, st); break;
    case 64: tc_launch_gv<BITS, G, 64>(a, grid, st); break;
    default: tc_launch_gv<BITS, G, 128>(a, grid, st); break;
    }
}

template <int BITS>
void attend_typed(const AttnArgs& a, int G, float* out, cudaStream_t st)
{
    const dim3 grid((unsigned)a.nsplit, (unsigned)a.outer);
    if ((BITS == 4 || BITS == 2) && G == 8) {
        // tensor cores (16-token tiles lie inside one K group: groups are a
        // multiple of 32 tokens, or one group over every quantized token).
        // Their cost hardly depends on the number of query heads; measured on
        // the KIVI workload they win at 8 heads (111 vs 150 us) and lose at
        // 1, 2 and 4 (96 / 99 / 103 vs 61 / 68 / 90 us), so fewer heads take
        // the CUDA-core kernel.
        tc_launch<BITS == 8 ? 4 : BITS, 8>(a, grid, st);
    } else {
        switch (G) {
        case 1: attend_split_kernel<BITS, 1><<<grid, kAThreads, 0, st>>>(a); break;
        case 2: attend_split_kernel<BITS, 2><<<grid, kAThreads, 0, st>>>(a); break;
        case 4: attend_split_kernel<BITS, 4><<<grid, kAThreads, 0, st>>>(a); break;
        default: attend_split_kernel<BITS, 8><<<grid, kAThreads, 0, st>>>(a); break;
        }
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
