// staged.cu -- quantize kernels fed by bulk asynchronous copies, and the
// coalesced streaming dequantize / statistics kernel (bf16 sources).
//
// Method: "KV Compression 公式到源码对照" §1.1-§1.3 and "KV cache 压缩：
// 把历史装得更小" (group-wise form, KIVI axes, residual window); same results
// as the other kernels, bit for bit.
//
// Quantize.  A persistent CTA walks 16 KB chunks of the source that are
// contiguous in memory: one group tile [g tokens x C channels] for groups
// along T (K), or 8192/C whole token rows for groups along C (V).  One thread
// issues cp.async.bulk into a 4-stage shared-memory ring, completion is
// signalled on an mbarrier per stage, so each SM keeps several chunks in
// flight without registers holding them.  Threads then read the chunk from
// shared memory, reduce each group, derive its constants once, and write
// codes and metadata with coalesced stores.
//
// Dequantize / statistics.  Lane = 8 channels of RPT consecutive tokens;
// lanes of a warp cover consecutive channel chunks, so every code load,
// source load and output store is coalesced; group constants are loaded once
// per lane item.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include <cudaTypedefs.h>

#include "kvq_bulk.cuh"
#include "kvq_elem.cuh"

namespace kvq {

namespace {

using namespace elem;

constexpr int kStages = 4;
constexpr int kStageBytes = 16384;
constexpr int kStagedSmem = kStages * kStageBytes + 64;   // ring + barriers

struct ChunkSrc { const void* ptr; uint32_t bytes; };

// metadata element of a compile-time dtype, widened to float
template <int DT>
__device__ __forceinline__ float ld_meta(const void* p, int64_t i) {
    if constexpr (DT == KVQ_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    else if constexpr (DT == KVQ_I8) return (float)static_cast<const int8_t*>(p)[i];
    else return static_cast<const float*>(p)[i];
}
// eight consecutive metadata elements (i a multiple of 8, buffer 16-byte aligned)
template <int DT>
__device__ __forceinline__ void ld_meta8(const void* p, int64_t i, float (&v)[8]) {
    if constexpr (DT == KVQ_BF16) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p) + i));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) { v[2 * k] = lo_f(ws[k]); v[2 * k + 1] = hi_f(ws[k]); }
    } else if constexpr (DT == KVQ_I8) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(static_cast<const int8_t*>(p) + i));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[k] = (float)(int8_t)(w.x >> (8 * k));
            v[k + 4] = (float)(int8_t)(w.y >> (8 * k));
        }
    } else if constexpr (DT == KVQ_F32) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p) + i));
        const float4 b = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p) + i + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = 0.0f;
    }
}

// the same from shared memory (plain loads)
template <int DT>
__device__ __forceinline__ void ld_meta8_smem(const unsigned char* p, int i, float (&v)[8]) {
    if constexpr (DT == KVQ_BF16) {
        const uint4 w = *reinterpret_cast<const uint4*>(p + 2 * i);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) { v[2 * k] = lo_f(ws[k]); v[2 * k + 1] = hi_f(ws[k]); }
    } else if constexpr (DT == KVQ_I8) {
        const uint2 w = *reinterpret_cast<const uint2*>(p + i);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[k] = (float)(int8_t)(w.x >> (8 * k));
            v[k + 4] = (float)(int8_t)(w.y >> (8 * k));
        }
    } else if constexpr (DT == KVQ_F32) {
        const float4 a = *reinterpret_cast<const float4*>(p + 4 * i);
        const float4 b = *reinterpret_cast<const float4*>(p + 4 * i + 16);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = 0.0f;
    }
}

template <int DT>
__device__ __forceinline__ void st_meta(void* p, int64_t i, float v) {
    if constexpr (DT == KVQ_BF16) static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    else if constexpr (DT == KVQ_I8) static_cast<int8_t*>(p)[i] = (int8_t)(int)v;
    else if constexpr (DT == KVQ_F32) static_cast<float*>(p)[i] = v;
}
template <int SDT, int ZDT>
__device__ __forceinline__ void write_meta_t(const QArgs& a, int64_t i, const GroupC& g) {
    st_meta<SDT>(a.scale, i, g.s);
    if constexpr (ZDT != KVQ_NONE) st_meta<ZDT>(a.zero, i, g.zp);
}

// The persistent chunk loop.  src(c) gives chunk c's source bytes, body(c,
// smem) consumes it; body is called by every thread of the CTA.
template <typename SrcFn, typename BodyFn>
__device__ __forceinline__ void staged_loop(uint64_t nchunks, SrcFn src, BodyFn body)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        mbar_init_fence();
    }
    __syncthreads();
    const uint64_t first = blockIdx.x, step = gridDim.x;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            const uint64_t c = first + (uint64_t)s * step;
            if (c < nchunks) {
                const ChunkSrc cs = src(c);
                mbar_expect_tx(&bars[s], cs.bytes);
                bulk_g2s(smem + s * kStageBytes, cs.ptr, cs.bytes, &bars[s]);
            }
        }
    }
    for (uint64_t k = 0;; ++k) {
        const uint64_t c = first + k * step;
        if (c >= nchunks) break;
        const int s = (int)(k % kStages);
        const uint32_t parity = (uint32_t)((k / kStages) & 1u);
        const bool ok = __syncthreads_and(mbar_wait(&bars[s], parity));
        if (!ok) {                                 // recorded in g_kvq_wait_timeouts
            // every copy issued must land before the CTA exits: thread 0 waits
            // (bounded) for this stage and each later one it has issued
            if (threadIdx.x == 0)
                for (uint64_t j = k; j < k + kStages && first + j * step < nchunks; ++j)
                    mbar_wait(&bars[j % kStages], (uint32_t)((j / kStages) & 1u));
            __syncthreads();
            return;
        }
        body(c, smem + s * kStageBytes);
        __syncthreads();                           // the stage is free again
        if (threadIdx.x == 0) {
            const uint64_t n = c + (uint64_t)kStages * step;
            if (n < nchunks) {
                const ChunkSrc cs = src(n);
                mbar_expect_tx(&bars[s], cs.bytes);
                bulk_g2s(smem + s * kStageBytes, cs.ptr, cs.bytes, &bars[s]);
            }
        }
    }
}

// ======================================================================
// groups along T: chunk = group tile [G tokens x C channels], C in {64,128,256}
// ======================================================================
template <int BITS, bool ASYM, int C, int SDT, int ZDT>
__global__ void __launch_bounds__(kThr)
sq_t_kernel(const QArgs a)
{
    constexpr int L8 = C / 8;                 // threads across a row (8 channels each)
    constexpr int NR = kThr / L8;             // row slices
    constexpr int MAXG = kStageBytes / (2 * C);
    constexpr int RPTH = (MAXG + NR - 1) / NR; // rows per thread at most
    constexpr int NW = kThr / 32;
    __shared__ uint32_t red_mn[NW][L8][4], red_mx[NW][L8][4];
    __shared__ __align__(16) float c_s[C], c_i[C];
    __shared__ __align__(16) int32_t c_z[C];

    const QSpec& q = a.q;
    const int t = threadIdx.x, c8 = t % L8, rs = t / L8, warp = t >> 5, lane = t & 31;
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const int lo_c = q.qmin + off, hi_c = q.qmax + off;
    const int G = (int)q.g;
    const uint32_t ng = (uint32_t)q.ngroups;
    const uint32_t nres = (uint32_t)((q.R + G - 1) / G);
    const uint32_t per_o = ng + nres;
    const uint64_t nchunks = (uint64_t)q.outer * per_o;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
    uint8_t* codes = static_cast<uint8_t*>(a.codes);
    const uint64_t code_row_B = (uint64_t)C * BITS / 8;

    const uint32_t Tq32 = (uint32_t)q.Tq, T32 = (uint32_t)q.T;
    // chunk -> (outer, group or residual slot k, first row, rows); 32-bit math
    auto geom = [&](uint64_t c, uint32_t& o, uint32_t& k, uint32_t& row0, int& nrows, bool& res) {
        const uint32_t c32 = (uint32_t)c;
        o = c32 / per_o;
        k = c32 - o * per_o;
        res = k >= ng;
        row0 = res ? Tq32 + (k - ng) * (uint32_t)G : k * (uint32_t)G;
        const uint32_t end = res ? T32 : Tq32;
        nrows = (int)min((uint32_t)G, end - row0);
    };
    auto src = [&](uint64_t c) {
        uint32_t o, k, row0; int nrows; bool res;
        geom(c, o, k, row0, nrows, res);
        return ChunkSrc{x + ((uint64_t)o * T32 + row0) * C, (uint32_t)(nrows * C * 2)};
    };
    auto body = [&](uint64_t c, const unsigned char* buf) {
        uint32_t o, k, row0; int nrows; bool res;
        geom(c, o, k, row0, nrows, res);
        uint4 w[RPTH];
#pragma unroll
        for (int j = 0; j < RPTH; ++j) {
            const int r = rs + NR * j;
            w[j] = r < nrows ? *reinterpret_cast<const uint4*>(buf + (size_t)r * C * 2 + c8 * 16) : make_uint4(0, 0, 0, 0);
        }
        if (res) {
            __nv_bfloat16* resid = static_cast<__nv_bfloat16*>(a.resid);
#pragma unroll
            for (int j = 0; j < RPTH; ++j) {
                const int r = rs + NR * j;
                if (r < nrows)
                    *reinterpret_cast<uint4*>(resid + (((uint64_t)o * q.R + (row0 - Tq32) + r) * C + c8 * 8)) = w[j];
            }
            return;
        }
        // per-thread statistics over its rows, then over the warp's row slices
        uint32_t mn[4], mx[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) { mn[p] = kBfPosInf2; mx[p] = ASYM ? kBfNegInf2 : 0u; }
#pragma unroll
        for (int j = 0; j < RPTH; ++j) {
            if (rs + NR * j < nrows) {
                const uint32_t ws[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    if (ASYM) { mn[p] = bmin2(mn[p], ws[p]); mx[p] = bmax2(mx[p], ws[p]); }
                    else mx[p] = bmax2(mx[p], babs2(ws[p]));
                }
            }
        }
#pragma unroll
        for (int sft = L8; sft < 32; sft <<= 1) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                if (ASYM) mn[p] = bmin2(mn[p], __shfl_xor_sync(0xFFFFFFFFu, mn[p], sft));
                mx[p] = bmax2(mx[p], __shfl_xor_sync(0xFFFFFFFFu, mx[p], sft));
            }
        }
        if (L8 >= 32 || lane < L8) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                red_mn[warp][c8][p] = mn[p];
                red_mx[warp][c8][p] = mx[p];
            }
        }
        __syncthreads();
        // one thread per channel: constants and metadata
        bool fast = true;
        if (t < C) {
            const int cc8 = t / 8, p = (t % 8) / 2, half = t & 1;
            constexpr int WARPS_WITH_DATA = L8 >= 32 ? NW : NW;   // every warp holds a partial
            uint32_t wm = red_mn[0][cc8][p], wx = red_mx[0][cc8][p];
#pragma unroll
            for (int wi = 1; wi < WARPS_WITH_DATA; ++wi) {
                if (ASYM) wm = bmin2(wm, red_mn[wi][cc8][p]);
                wx = bmax2(wx, red_mx[wi][cc8][p]);
            }
            const float fmn = half ? hi_f(wm) : lo_f(wm);
            const float fmx = half ? hi_f(wx) : lo_f(wx);
            const GroupC gc = make_group<ASYM>(fmn, fmx, q, off);
            write_meta_t<SDT, ZDT>(a, ((int64_t)o * ng + k) * C + t, gc);
            c_s[t] = gc.s;
            c_i[t] = gc.inv;
            c_z[t] = gc.zoff;
            fast = gc.fast;
        }
        const bool all_fast = __syncthreads_and(fast);
        float s8[8], i8[8], z8f[8];
        int32_t zo[8];
        {
            const float4* ps = reinterpret_cast<const float4*>(c_s + c8 * 8);
            const float4* pi = reinterpret_cast<const float4*>(c_i + c8 * 8);
            const int4* pz = reinterpret_cast<const int4*>(c_z + c8 * 8);
            const float4 s0 = ps[0], s1 = ps[1], i0 = pi[0], i1 = pi[1];
            const int4 z0 = pz[0], z1 = pz[1];
            s8[0] = s0.x; s8[1] = s0.y; s8[2] = s0.z; s8[3] = s0.w; s8[4] = s1.x; s8[5] = s1.y; s8[6] = s1.z; s8[7] = s1.w;
            i8[0] = i0.x; i8[1] = i0.y; i8[2] = i0.z; i8[3] = i0.w; i8[4] = i1.x; i8[5] = i1.y; i8[6] = i1.z; i8[7] = i1.w;
            zo[0] = z0.x; zo[1] = z0.y; zo[2] = z0.z; zo[3] = z0.w; zo[4] = z1.x; zo[5] = z1.y; zo[6] = z1.z; zo[7] = z1.w;
        }
        uint8_t* cbase = codes + ((uint64_t)o * q.Tq + row0) * code_row_B + (uint64_t)c8 * BITS;
        if (all_fast) {
            QuotK kq[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                kq[p].ns = pk(-s8[2 * p], -s8[2 * p + 1]);
                kq[p].inv = pk(i8[2 * p], i8[2 * p + 1]);
            }
#pragma unroll
            for (int j = 0; j < RPTH; ++j) {
                const int r = rs + NR * j;
                if (r < nrows) {
                    uint32_t cc[8];
                    codes8_fast<ASYM>(w[j], kq, zo, lo_c, hi_c, cc);
                    store_codes<BITS>(cbase + (uint64_t)r * code_row_B, finish_word<BITS>(cc, q.is_signed));
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) z8f[j] = (float)(zo[j] - off + (int32_t)kMagicBits);
#pragma unroll
            for (int j = 0; j < RPTH; ++j) {
                const int r = rs + NR * j;
                if (r < nrows) {
                    uint32_t cc[8];
                    codes8_slow<ASYM>(w[j], s8, z8f, q, off, cc);
                    store_codes<BITS>(cbase + (uint64_t)r * code_row_B, finish_word<BITS>(cc, q.is_signed));
                }
            }
        }
    };
    staged_loop(nchunks, src, body);
}

// ======================================================================
// groups along T, warp-specialised (C = 128, g in {16, 32, 64}).  A producer
// warp keeps a ring of kWStages stages full with bulk copies; each stage is
// one group tile [g tokens x 128 channels] and is consumed by one pair of
// warps, one per 64-channel half: lane = 8 channels x every fourth token of
// the tile, so a group's min / max is two shuffles away and no block-wide
// barrier is ever taken.  Stage s is handed back to the producer by one
// arrival of each warp of the pair on empty[s].  Stage s belongs to pair
// s % kWPairs (kWStages is a multiple of kWPairs): when a pair waits for the
// phase of chunk j on its stage it has itself consumed chunk j - kWStages
// there, so the phase parity it waits on cannot be confused with an older one.
// ======================================================================
constexpr int kWPairs = 6;
constexpr int kWStages = 12;
static_assert(kWStages % kWPairs == 0, "a stage must belong to one consumer pair");
constexpr int kWThreads = (2 * kWPairs + 1) * 32;
constexpr int kWSmem = kWStages * kStageBytes + 2 * kWStages * 8;

template <int BITS, bool ASYM, int G, int SDT, int ZDT>
__global__ void __launch_bounds__(kWThreads, 1)
wq_t_kernel(const QArgs a)
{
    constexpr int C = 128;
    constexpr int RPL = G / 4;                          // rows per lane in a full tile
    constexpr uint32_t kRowB = C * 2;                   // bytes of one bf16 row
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kWStages * kStageBytes);
    uint64_t* empty = full + kWStages;

    const QSpec& q = a.q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ng = (uint32_t)q.ngroups;
    const uint32_t nres = (uint32_t)((q.R + G - 1) / G);
    const uint32_t per_o = ng + nres;
    const uint32_t nchunks = (uint32_t)q.outer * per_o;   // < 2^31, checked by the dispatcher
    const uint32_t Tq32 = (uint32_t)q.Tq, T32 = (uint32_t)q.T;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);
        }
        mbar_init_fence();
    }
    __syncthreads();

    auto geom = [&](uint32_t c, uint32_t& o, uint32_t& k, uint32_t& row0, int& nrows, bool& res) {
        o = c / per_o;
        k = c - o * per_o;
        res = k >= ng;
        row0 = res ? Tq32 + (k - ng) * (uint32_t)G : k * (uint32_t)G;
        const uint32_t end = res ? T32 : Tq32;
        nrows = (int)min((uint32_t)G, end - row0);
    };
    const uint32_t first = blockIdx.x, step = gridDim.x;

    if (warp == 2 * kWPairs) {
        // ---- producer: one lane issues every copy of this CTA
        if (lane != 0) return;
        uint32_t n = 0;
        for (;; ++n) {
            const uint32_t c = first + n * step;
            if (c >= nchunks) break;
            const int s = (int)(n % kWStages);
            if (n >= (uint32_t)kWStages && !mbar_wait(&empty[s], ((n / kWStages) - 1) & 1u)) break;
            uint32_t o, k, row0; int nrows; bool res;
            geom(c, o, k, row0, nrows, res);
            const uint32_t bytes = (uint32_t)nrows * kRowB;
            mbar_expect_tx(&full[s], bytes);
            bulk_g2s(smem + s * kStageBytes, x + ((uint64_t)o * T32 + row0) * C, bytes, &full[s]);
        }
        // every copy issued must land before the CTA may exit
        for (uint32_t i = n > (uint32_t)kWStages ? n - kWStages : 0; i < n; ++i)
            mbar_wait(&full[i % kWStages], (i / kWStages) & 1u);
        return;
    }

    // ---- consumers: warp pair p, channel half e
    const int pair = warp >> 1, e = warp & 1;
    const int c8 = lane & 7, rq = lane >> 3;            // 8 channels x rows rq, rq+4, ...
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const int lo_c = q.qmin + off, hi_c = q.qmax + off;
    uint8_t* codes = static_cast<uint8_t*>(a.codes);
    constexpr uint32_t kCodeRowB = C * BITS / 8;
    const int chan0 = e * 64 + c8 * 8;                   // first of this lane's 8 channels
    for (uint32_t j = pair;; j += kWPairs) {
        const uint32_t c = first + j * step;
        if (c >= nchunks) break;
        const int s = (int)(j % kWStages);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (j / kWStages) & 1u))) return;   // recorded in g_kvq_wait_timeouts
        const unsigned char* tile = smem + s * kStageBytes + chan0 * 2 + rq * kRowB;
        uint32_t o, k, row0; int nrows; bool res;
        geom(c, o, k, row0, nrows, res);
        const bool whole = nrows == G;
        if (res) {
            __nv_bfloat16* rp = static_cast<__nv_bfloat16*>(a.resid) +
                                (((uint64_t)o * q.R + (row0 - Tq32) + rq) * C + chan0);
#pragma unroll 4
            for (int i = 0; i < RPL; ++i)
                if (4 * i + rq < nrows)
                    *reinterpret_cast<uint4*>(rp + (uint64_t)i * 4 * C) = *reinterpret_cast<const uint4*>(tile + i * 4 * kRowB);
        } else {
            // group min / max (abs-max when symmetric) over the lane's rows, then over the 4 row slices
            uint32_t mn[4], mx[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) { mn[p] = kBfPosInf2; mx[p] = ASYM ? kBfNegInf2 : 0u; }
            auto fold = [&](const uint4& w) {     // per channel pair
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    if (ASYM) { mn[p] = bmin2(mn[p], ws[p]); mx[p] = bmax2(mx[p], ws[p]); }
                    else mx[p] = bmax2(mx[p], babs2(ws[p]));
                }
            };
            if (whole) {
#pragma unroll 8
                for (int i = 0; i < RPL; ++i) fold(*reinterpret_cast<const uint4*>(tile + i * 4 * kRowB));
            } else {
#pragma unroll 4
                for (int i = 0; i < RPL; ++i)
                    if (4 * i + rq < nrows) fold(*reinterpret_cast<const uint4*>(tile + i * 4 * kRowB));
            }
#pragma unroll
            for (int sft = 8; sft < 32; sft <<= 1) {
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    if (ASYM) mn[p] = bmin2(mn[p], __shfl_xor_sync(0xFFFFFFFFu, mn[p], sft));
                    mx[p] = bmax2(mx[p], __shfl_xor_sync(0xFFFFFFFFu, mx[p], sft));
                }
            }
            // row slice rq derives the constants of channel pair rq (channels 2rq, 2rq+1)
            const uint32_t wmn = rq == 0 ? mn[0] : rq == 1 ? mn[1] : rq == 2 ? mn[2] : mn[3];
            const uint32_t wmx = rq == 0 ? mx[0] : rq == 1 ? mx[1] : rq == 2 ? mx[2] : mx[3];
            const int64_t mi = ((int64_t)o * ng + k) * C + chan0 + 2 * rq;
            const GroupC g0 = make_group<ASYM>(lo_f(wmn), lo_f(wmx), q, off);
            const GroupC g1 = make_group<ASYM>(hi_f(wmn), hi_f(wmx), q, off);
            write_meta_t<SDT, ZDT>(a, mi, g0);
            write_meta_t<SDT, ZDT>(a, mi + 1, g1);
            const bool all_fast = __all_sync(0xFFFFFFFFu, g0.fast && g1.fast);
            const bool no_lo_clip = __all_sync(0xFFFFFFFFu, g0.lo_ok && g1.lo_ok);
            // every lane gathers the constants of its four channel pairs from row slices 0..3
            float s8[8], i8[8];
            int32_t zo[8];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const int src = c8 + 8 * p;
                s8[2 * p] = __shfl_sync(0xFFFFFFFFu, g0.s, src);
                s8[2 * p + 1] = __shfl_sync(0xFFFFFFFFu, g1.s, src);
                i8[2 * p] = __shfl_sync(0xFFFFFFFFu, g0.inv, src);
                i8[2 * p + 1] = __shfl_sync(0xFFFFFFFFu, g1.inv, src);
                zo[2 * p] = __shfl_sync(0xFFFFFFFFu, g0.zoff, src);
                zo[2 * p + 1] = __shfl_sync(0xFFFFFFFFu, g1.zoff, src);
            }
            uint8_t* cp = codes + ((uint64_t)o * Tq32 + row0 + rq) * kCodeRowB + (uint32_t)(chan0 / 8) * BITS;
            if (all_fast) {
                QuotK kq[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    kq[p].ns = pk(-s8[2 * p], -s8[2 * p + 1]);
                    kq[p].inv = pk(i8[2 * p], i8[2 * p + 1]);
                }
                auto emit = [&](int i, auto lo_clip) {
                    uint32_t cc[8];
                    codes8_fast<ASYM, decltype(lo_clip)::value>(*reinterpret_cast<const uint4*>(tile + i * 4 * kRowB),
                                                                kq, zo, lo_c, hi_c, cc);
                    store_codes<BITS>(cp + (uint64_t)i * 4 * kCodeRowB, finish_word<BITS>(cc, q.is_signed));
                };
                if (whole && (!ASYM || no_lo_clip)) {
#pragma unroll 4
                    for (int i = 0; i < RPL; ++i) emit(i, std::false_type{});
                } else {
                    for (int i = 0; i < RPL; ++i)
                        if (4 * i + rq < nrows) emit(i, std::true_type{});
                }
            } else {
                float z8[8];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const int src = c8 + 8 * p;
                    z8[2 * p] = __shfl_sync(0xFFFFFFFFu, g0.zp, src);
                    z8[2 * p + 1] = __shfl_sync(0xFFFFFFFFu, g1.zp, src);
                }
                for (int i = 0; i < RPL; ++i)
                    if (4 * i + rq < nrows) {
                        uint32_t cc[8];
                        codes8_slow<ASYM>(*reinterpret_cast<const uint4*>(tile + i * 4 * kRowB), s8, z8, q, off, cc);
                        store_codes<BITS>(cp + (uint64_t)i * 4 * kCodeRowB, finish_word<BITS>(cc, q.is_signed));
                    }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// ======================================================================
// groups along C, warp-specialised (C = 128, g in {32, 64, 128}).  A chunk is
// 32 consecutive token rows, brought in by two 2-D TMA loads (channels 0-63
// and 64-127, 4 KB each) with the 128-byte swizzle: within each 1 KB block the
// 16-byte column u of row r lands at slot u ^ (r & 7), so lane l reading
// column u of row l hits a different bank group than lanes l+1 .. l+7.  Each
// of the kCConsumers consumer warps owns whole chunks: lane = one token row,
// so a group's reduction and constants stay in one thread.
// ======================================================================
constexpr int kCConsumers = 12;
constexpr int kCRows = 32;
constexpr int kCHalfB = kCRows * 128;                      // one 64-channel box
constexpr int kCStageB = 2 * kCHalfB;                      // 8192
constexpr int kCStages = 24;
static_assert(kCStages % kCConsumers == 0, "a stage must belong to one consumer warp");
constexpr int kCThreads = (kCConsumers + 1) * 32;
constexpr int kCSmem = 1024 + kCStages * kCStageB + 2 * kCStages * 8;   // + alignment slack

template <int BITS, bool ASYM, int G, int SDT, int ZDT>
__global__ void __launch_bounds__(kCThreads, 1)
wq_c_kernel(const QArgs a, const __grid_constant__ CUtensorMap tmap)
{
    constexpr int C = 128;
    constexpr int GPR = C / G;                 // groups per row
    constexpr int WPG = G / 8;                 // 16-byte words per group
    using W = typename CodeWord<BITS>::T;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // the swizzled boxes need 1 KB alignment
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kCStages * kCStageB);
    uint64_t* empty = full + kCStages;

    const QSpec& q = a.q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t T32 = (uint32_t)q.T, Tq32 = (uint32_t)q.Tq;
    const uint32_t nrows_total = (uint32_t)(q.outer * q.T);       // < 2^31, checked by the dispatcher
    const uint32_t nchunks = (nrows_total + kCRows - 1) / kCRows;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kCStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init_fence();
    }
    __syncthreads();
    const uint32_t first = blockIdx.x, step = gridDim.x;

    if (warp == kCConsumers) {
        // ---- producer: one lane issues both boxes of every chunk of this CTA
        if (lane != 0) return;
        uint32_t n = 0;
        for (;; ++n) {
            const uint32_t c = first + n * step;
            if (c >= nchunks) break;
            const int s = (int)(n % kCStages);
            if (n >= (uint32_t)kCStages && !mbar_wait(&empty[s], ((n / kCStages) - 1) & 1u)) break;
            // rows past the end are zero-filled and still counted in the box bytes
            mbar_expect_tx(&full[s], (uint32_t)kCStageB);
            tma_load_2d(smem + s * kCStageB, &tmap, 0, (int)(c * kCRows), &full[s]);
            tma_load_2d(smem + s * kCStageB + kCHalfB, &tmap, 64, (int)(c * kCRows), &full[s]);
        }
        for (uint32_t i = n > (uint32_t)kCStages ? n - kCStages : 0; i < n; ++i)
            mbar_wait(&full[i % kCStages], (i / kCStages) & 1u);
        return;
    }

    // ---- consumers
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const int lo_c = q.qmin + off, hi_c = q.qmax + off;
    uint8_t* codes = static_cast<uint8_t*>(a.codes);
    constexpr uint32_t kCodeRowB = C * BITS / 8;
    for (uint32_t j = warp;; j += kCConsumers) {
        const uint32_t c = first + j * step;
        if (c >= nchunks) break;
        const int s = (int)(j % kCStages);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (j / kCStages) & 1u))) return;   // recorded in g_kvq_wait_timeouts
        const uint32_t row = c * kCRows + lane;
        const unsigned char* rp = smem + s * kCStageB + lane * 128;
        const int sw = lane & 7;
        // 16-byte column k (0..15) of this lane's row
        auto word = [&](int k) -> uint4 {
            return *reinterpret_cast<const uint4*>(rp + (k >> 3) * kCHalfB + (((k & 7) ^ sw) << 4));
        };
        if (row < nrows_total) {
            const uint32_t o = row / T32, t = row - o * T32;
            if (t >= Tq32) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.resid) +
                                                      ((uint64_t)o * q.R + (t - Tq32)) * C);
#pragma unroll
                for (int k = 0; k < C / 8; ++k) dst[k] = word(k);
            } else {
                const uint64_t qrow = (uint64_t)o * Tq32 + t;
                W cw[C / 8];
#pragma unroll
                for (int gi = 0; gi < GPR; ++gi) {
                    uint32_t mn = kBfPosInf2, mx = ASYM ? kBfNegInf2 : 0u;
#pragma unroll
                    for (int k = 0; k < WPG; ++k) {
                        const uint4 w = word(gi * WPG + k);
                        if (ASYM) fold_minmax(w, mn, mx);
                        else fold_absmax(w, mx);
                    }
                    const GroupC gc = make_group<ASYM>(fminf(lo_f(mn), hi_f(mn)), fmaxf(lo_f(mx), hi_f(mx)), q, off);
                    write_meta_t<SDT, ZDT>(a, (int64_t)qrow * GPR + gi, gc);
                    if (gc.fast) {
                        QuotK kq[4];
                        kq[0].ns = pk(-gc.s, -gc.s);
                        kq[0].inv = pk(gc.inv, gc.inv);
                        kq[1] = kq[2] = kq[3] = kq[0];
                        int32_t zo[8];
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) zo[jj] = gc.zoff;
                        if (!ASYM || gc.lo_ok) {
#pragma unroll
                            for (int k = 0; k < WPG; ++k) {
                                uint32_t cc[8];
                                codes8_fast<ASYM, false>(word(gi * WPG + k), kq, zo,
                                                         lo_c, hi_c, cc);
                                cw[gi * WPG + k] = finish_word<BITS>(cc, q.is_signed);
                            }
                        } else {
#pragma unroll
                            for (int k = 0; k < WPG; ++k) {
                                uint32_t cc[8];
                                codes8_fast<ASYM>(word(gi * WPG + k), kq, zo,
                                                  lo_c, hi_c, cc);
                                cw[gi * WPG + k] = finish_word<BITS>(cc, q.is_signed);
                            }
                        }
                    } else {
                        float s8[8], z8[8];
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) { s8[jj] = gc.s; z8[jj] = gc.zp; }
#pragma unroll
                        for (int k = 0; k < WPG; ++k) {
                            uint32_t cc[8];
                            codes8_slow<ASYM>(word(gi * WPG + k), s8, z8, q, off, cc);
                            cw[gi * WPG + k] = finish_word<BITS>(cc, q.is_signed);
                        }
                    }
                }
                // the row's codes: kCodeRowB bytes, 16-byte stores
                uint4* cdst = reinterpret_cast<uint4*>(codes + qrow * kCodeRowB);
                constexpr int WPS = 16 / sizeof(W);          // code words per 16-byte store
#pragma unroll
                for (int k = 0; k < (C / 8) / WPS; ++k) {
                    uint4 v;
                    if constexpr (BITS == 8) {
                        v = make_uint4(cw[2 * k].x, cw[2 * k].y, cw[2 * k + 1].x, cw[2 * k + 1].y);
                    } else if constexpr (BITS == 4) {
                        v = make_uint4(cw[4 * k], cw[4 * k + 1], cw[4 * k + 2], cw[4 * k + 3]);
                    } else {
                        v = make_uint4((uint32_t)cw[8 * k] | ((uint32_t)cw[8 * k + 1] << 16),
                                       (uint32_t)cw[8 * k + 2] | ((uint32_t)cw[8 * k + 3] << 16),
                                       (uint32_t)cw[8 * k + 4] | ((uint32_t)cw[8 * k + 5] << 16),
                                       (uint32_t)cw[8 * k + 6] | ((uint32_t)cw[8 * k + 7] << 16));
                    }
                    cdst[k] = v;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

// ======================================================================
// groups along C: chunk = 8192/C whole token rows; thread = 32 channels
// ======================================================================
template <int BITS, bool ASYM, int G, int SDT, int ZDT>
__global__ void __launch_bounds__(kThr)
sq_c_kernel(const QArgs a)
{
    constexpr int GPT = G >= 32 ? 1 : 32 / G;    // groups per thread
    constexpr int TPG = G >= 32 ? G / 32 : 1;    // threads per group
    constexpr int WPG = G >= 32 ? 4 : G / 8;     // 8-element words per group in a thread
    const QSpec& q = a.q;
    const int t = threadIdx.x;
    const int C = (int)q.C;
    const int TPR = C / 32;                      // threads per row
    const int RC = kStageBytes / (2 * C);        // rows per chunk
    const int r = t / TPR, part = t - r * TPR;
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const int lo_c = q.qmin + off, hi_c = q.qmax + off;
    const uint32_t T = (uint32_t)q.T, Tq = (uint32_t)q.Tq;
    const uint64_t nrows_total = (uint64_t)q.outer * q.T;
    const uint64_t nchunks = (nrows_total + RC - 1) / RC;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
    uint8_t* codes = static_cast<uint8_t*>(a.codes);
    const int gpr = C / G;

    auto src = [&](uint64_t c) {
        const uint64_t row0 = c * RC;
        const uint64_t n = min((uint64_t)RC, nrows_total - row0);
        return ChunkSrc{x + row0 * C, (uint32_t)(n * C * 2)};
    };
    auto body = [&](uint64_t c, const unsigned char* buf) {
        const uint64_t grow = c * RC + r;
        const bool valid = r < RC && grow < nrows_total;
        uint4 w[4];
        const unsigned char* p = buf + (size_t)r * C * 2 + part * 64;
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = valid ? *reinterpret_cast<const uint4*>(p + k * 16) : make_uint4(0, 0, 0, 0);
        const uint32_t g32 = (uint32_t)grow;
        const uint32_t o = valid ? g32 / T : 0u;
        const uint32_t tt = valid ? g32 - o * T : 0u;
        // group statistics
        float gmn[GPT], gmx[GPT];
#pragma unroll
        for (int gg = 0; gg < GPT; ++gg) {
            uint32_t mn = kBfPosInf2, mx = ASYM ? kBfNegInf2 : 0u;
#pragma unroll
            for (int k = 0; k < WPG; ++k) {
                if (ASYM) fold_minmax(w[gg * WPG + k], mn, mx);
                else fold_absmax(w[gg * WPG + k], mx);
            }
            gmn[gg] = fminf(lo_f(mn), hi_f(mn));
            gmx[gg] = fmaxf(lo_f(mx), hi_f(mx));
#pragma unroll
            for (int sft = 1; sft < TPG; sft <<= 1) {
                gmn[gg] = fminf(gmn[gg], __shfl_xor_sync(0xFFFFFFFFu, gmn[gg], sft));
                gmx[gg] = fmaxf(gmx[gg], __shfl_xor_sync(0xFFFFFFFFu, gmx[gg], sft));
            }
        }
        if (!valid) return;
        if (tt >= Tq) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.resid) +
                                                 (((uint64_t)o * q.R + (tt - Tq)) * C + (uint64_t)part * 32));
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[k] = w[k];
            return;
        }
        const uint64_t qrow = (uint64_t)o * Tq + tt;
        typename CodeWord<BITS>::T cw[4];
#pragma unroll
        for (int gg = 0; gg < GPT; ++gg) {
            const GroupC gc = make_group<ASYM>(gmn[gg], gmx[gg], q, off);
            const int64_t gidx = G >= 32 ? (int64_t)part / TPG : (int64_t)part * GPT + gg;
            if (TPG == 1 || (part % TPG) == 0) write_meta_t<SDT, ZDT>(a, (int64_t)qrow * gpr + gidx, gc);
            if (gc.fast) {
                QuotK kq[4];
                kq[0].ns = pk(-gc.s, -gc.s);
                kq[0].inv = pk(gc.inv, gc.inv);
                kq[1] = kq[2] = kq[3] = kq[0];
                int32_t zo[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) zo[j] = gc.zoff;
                if (gc.lo_ok) {
#pragma unroll
                    for (int k = 0; k < WPG; ++k) {
                        uint32_t cc[8];
                        codes8_fast<ASYM, false>(w[gg * WPG + k], kq, zo, lo_c, hi_c, cc);
                        cw[gg * WPG + k] = finish_word<BITS>(cc, q.is_signed);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < WPG; ++k) {
                        uint32_t cc[8];
                        codes8_fast<ASYM>(w[gg * WPG + k], kq, zo, lo_c, hi_c, cc);
                        cw[gg * WPG + k] = finish_word<BITS>(cc, q.is_signed);
                    }
                }
            } else {
                float s8[8], z8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) { s8[j] = gc.s; z8[j] = gc.zp; }
#pragma unroll
                for (int k = 0; k < WPG; ++k) {
                    uint32_t cc[8];
                    codes8_slow<ASYM>(w[gg * WPG + k], s8, z8, q, off, cc);
                    cw[gg * WPG + k] = finish_word<BITS>(cc, q.is_signed);
                }
            }
        }
        uint8_t* cdst = codes + qrow * (uint64_t)(C * BITS / 8) + (uint64_t)part * 4 * BITS;
#pragma unroll
        for (int k = 0; k < 4; ++k) store_codes<BITS>(cdst + k * BITS, cw[k]);
    };
    staged_loop(nchunks, src, body);
}

// ======================================================================
// dequantize / statistics: lane = 8 channels x RPT tokens
// ======================================================================
// Constants of one group for all four pairs of a lane's eight channels.
__device__ __forceinline__ void dq_pair_consts(float s, float z, int off, u64& cp, u64& sp) {
    const float c = __fadd_rn(8388608.0f + (float)off, z);
    cp = pk(c, c);
    sp = pk(s, s);
}

// The final fixed-order reduction of the block partials by one block (the
// last to finish): thread t sums partials t, t + kThr, ... in order, then a
// fixed tree; the result does not depend on which block ran last.
__device__ __forceinline__ void finalize_in_block(const Partial* partials, int64_t n, double N, kvq_err* out)
{
    __shared__ double f1[kThr], f2[kThr], fm[kThr];
    double s1 = 0.0, s2 = 0.0, mx = 0.0;
    for (int64_t i = threadIdx.x; i < n; i += kThr) {
        s1 += __ldcg(&partials[i].s1);
        s2 += __ldcg(&partials[i].s2);
        mx = fmax(mx, __ldcg(&partials[i].mx));
    }
    f1[threadIdx.x] = s1; f2[threadIdx.x] = s2; fm[threadIdx.x] = mx;
    __syncthreads();
    for (int o = kThr / 2; o > 0; o >>= 1) {
        if (threadIdx.x < o) {
            f1[threadIdx.x] += f1[threadIdx.x + o];
            f2[threadIdx.x] += f2[threadIdx.x + o];
            fm[threadIdx.x] = fmax(fm[threadIdx.x], fm[threadIdx.x + o]);
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        out->rmse = sqrt(f2[0] / N);
        out->max_abs = fm[0];
        out->mean_abs = f1[0] / N;
    }
}

template <int BITS, bool ASYM, bool ALONG_T, int RPT, bool STATS, int SDT, int ZDT>
__global__ void __launch_bounds__(kThr)
ds_kernel(const QArgs a, int lcpr, int lg, Partial* partials, unsigned int* done, kvq_err* out_dev)
{
    const QSpec& q = a.q;
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const int64_t C = q.C;
    const uint32_t cpr = 1u << lcpr;                         // 8-channel chunks per row
    const int64_t Tq = q.Tq;
    const uint32_t nrb_q = (uint32_t)(Tq / RPT);              // full row blocks of quantized tokens
    const uint32_t nrb = (uint32_t)((q.T + RPT - 1) / RPT);  // all row blocks
    const uint64_t items_per_o = (uint64_t)nrb << lcpr;
    const uint8_t* codes = static_cast<const uint8_t*>(a.codes);
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    const __nv_bfloat16* resid = static_cast<const __nv_bfloat16*>(a.resid);
    const uint64_t code_row_B = (uint64_t)C * BITS / 8;
    const uint32_t gpr = ALONG_T ? 0u : (uint32_t)q.ngroups;  // groups per row (along C)
    using W = typename CodeWord<BITS>::T;
    Acc2 A;
    for (uint64_t o = blockIdx.y; o < (uint64_t)q.outer; o += gridDim.y) {
        for (uint64_t it = (uint64_t)blockIdx.x * kThr + threadIdx.x; it < items_per_o;
             it += (uint64_t)gridDim.x * kThr) {
            const uint32_t c8 = (uint32_t)(it & (cpr - 1));
            const uint32_t rb = (uint32_t)(it >> lcpr);
            const int64_t t0 = (int64_t)rb * RPT;
            const uint64_t cofs = (uint64_t)c8 * 8;
            if (rb < nrb_q) {
                // RPT quantized rows
                const W* cptr = reinterpret_cast<const W*>(codes + ((uint64_t)o * Tq + t0) * code_row_B) + c8;
                const size_t cstride = code_row_B / sizeof(W);
                const uint4* xptr = reinterpret_cast<const uint4*>(x + ((o * (uint64_t)q.T + t0) * C + cofs));
                uint4* optr = reinterpret_cast<uint4*>(out + ((o * (uint64_t)q.T + t0) * C + cofs));
                const size_t vstride = (size_t)C / 8;
                W cw[RPT];
                uint4 xw[RPT];
#pragma unroll
                for (int j = 0; j < RPT; ++j) {
                    cw[j] = __ldcs(cptr + j * cstride);
                    if (STATS) xw[j] = __ldcs(xptr + j * vstride);
                }
                u64 cp[4], sp[4];
                bool fast_t = true;
                if (ALONG_T) {
                    // eight per-channel groups shared by the RPT rows: two 16-byte loads at most
                    const int64_t mi = ((int64_t)o * q.ngroups + (t0 >> lg)) * C + (int64_t)cofs;
                    float sf[8], zf[8];
                    ld_meta8<SDT>(a.scale, mi, sf);
                    if (ASYM) ld_meta8<ZDT>(a.zero, mi, zf);
                    const float base = 8388608.0f + (float)off;
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const float z0 = ASYM ? zf[2 * p] : 0.0f, z1 = ASYM ? zf[2 * p + 1] : 0.0f;
                        cp[p] = add2(pk(z0, z1), pk(base, base));
                        sp[p] = pk(sf[2 * p], sf[2 * p + 1]);
                        if (ASYM) fast_t = fast_t && fmaxf(fabsf(z0), fabsf(z1)) < 0x1p21f;
                    }
                }
                // groups along C: every row's scale and zero point, all loads issued together
                float ssr[RPT], zsr[RPT];
                if (!ALONG_T) {
#pragma unroll
                    for (int j = 0; j < RPT; ++j) {
                        const int64_t mi = ((int64_t)o * Tq + t0 + j) * gpr + (int64_t)(cofs >> lg);
                        ssr[j] = ld_meta<SDT>(a.scale, mi);
                        zsr[j] = ASYM ? ld_meta<ZDT>(a.zero, mi) : 0.0f;
                    }
                }
                TileAcc ta;
#pragma unroll
                for (int j = 0; j < RPT; ++j) {
                    float zs = 0.0f, ss = 1.0f;
                    if (!ALONG_T) {
                        ss = ssr[j];
                        zs = zsr[j];
                        u64 c1, s1;
                        dq_pair_consts(ss, zs, off, c1, s1);
                        cp[0] = cp[1] = cp[2] = cp[3] = c1;
                        sp[0] = sp[1] = sp[2] = sp[3] = s1;
                    }
                    uint32_t u[8];
                    unpack_biased8<BITS>(q.is_signed ? flip_signs<BITS>(cw[j]) : cw[j], u);
                    const bool fast = ALONG_T ? fast_t : (!ASYM || fabsf(zs) < 0x1p21f);
                    uint4 ow;
                    if (fast) {
                        ow = dq8<STATS>(u, cp, sp, xw[j], ta, A.mxb);
                    } else {
                        // exact reference order for groups with a very large zero point
                        float sf[8], zf[8];
                        const int64_t mi = ALONG_T ? ((int64_t)o * q.ngroups + (t0 >> lg)) * C + (int64_t)cofs
                                                   : ((int64_t)o * Tq + t0 + j) * gpr + (int64_t)(cofs >> lg);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            sf[k] = ld_meta<SDT>(a.scale, ALONG_T ? mi + k : mi);
                            zf[k] = ASYM ? ld_meta<ZDT>(a.zero, ALONG_T ? mi + k : mi) : 0.0f;
                        }
                        ow = dq8_slow<STATS>(u, off, zf, sf, xw[j], ta, A.mxb);
                    }
                    if (!STATS) optr[j * vstride] = ow;
                }
                if (STATS) A.fold(ta);
            } else {
                // tail: the last partial row block and the residual window
                for (int j = 0; j < RPT; ++j) {
                    const int64_t tr = t0 + j;
                    if (tr >= q.T) break;
                    const uint64_t xo = (o * (uint64_t)q.T + tr) * C + cofs;
                    if (tr >= Tq) {
                        if (!STATS)
                            *reinterpret_cast<uint4*>(out + xo) =
                                __ldcs(reinterpret_cast<const uint4*>(resid + ((o * (uint64_t)q.R + (tr - Tq)) * C + cofs)));
                        continue;
                    }
                    const W w = __ldcs(reinterpret_cast<const W*>(codes + ((uint64_t)o * Tq + tr) * code_row_B + (uint64_t)c8 * BITS));
                    const uint4 xv = STATS ? __ldcs(reinterpret_cast<const uint4*>(x + xo)) : make_uint4(0, 0, 0, 0);
                    float sf[8], zf[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int64_t mi = ALONG_T ? ((int64_t)o * q.ngroups + (tr >> lg)) * C + (int64_t)cofs + k
                                                   : ((int64_t)o * Tq + tr) * gpr + (int64_t)(cofs >> lg);
                        sf[k] = ld_meta<SDT>(a.scale, mi);
                        zf[k] = ASYM ? ld_meta<ZDT>(a.zero, mi) : 0.0f;
                    }
                    uint32_t u[8];
                    unpack_biased8<BITS>(q.is_signed ? flip_signs<BITS>(w) : w, u);
                    TileAcc ta;
                    const uint4 ow = dq8_slow<STATS>(u, off, zf, sf, xv, ta, A.mxb);
                    if (STATS) A.fold(ta);
                    else *reinterpret_cast<uint4*>(out + xo) = ow;
                }
            }
        }
    }
    if (STATS) {
        block_reduce_partial(A, partials);
        if (done) {
            // the last block to finish reduces every partial in a fixed order
            __shared__ bool s_last;
            __threadfence();
            __syncthreads();
            const unsigned int nb = gridDim.x * gridDim.y;
            if (threadIdx.x == 0) s_last = atomicAdd(done, 1u) == nb - 1;
            __syncthreads();
            if (s_last) {
                __threadfence();
                finalize_in_block(partials, nb, (double)q.outer * (double)q.T * (double)q.C, out_dev);
            }
        }
    }
}

// ======================================================================
// dequantize / statistics along T, warp-specialised (bf16, C = 128, g in
// {16, 32, 64}).  A chunk is one quantized group tile of an outer slice: the
// producer warp bulk-copies its codes [g rows x 16*BITS B], the 128 scales
// and zero points and, for the statistics, the source tile [g x 128] bf16
// into one ring stage.  Stage s belongs to warp pair s % P (two stages per
// pair); the two warps of a pair take one 64-channel half each: lane = 8
// channels x every fourth row, with the group constants of its channels read
// from the stage once per tile.  Dequantize writes x_hat rows straight from
// registers (16 B per lane, 128 B per 8 lanes) and copies the residual rows;
// statistics accumulate as in ds_kernel, and the last CTA reduces the block
// partials in a fixed order.
// ======================================================================
template <int BITS, int G, bool STATS, int SDT, int ZDT>
struct DtShape {
    static constexpr int CR = G;                                     // rows per chunk: one group tile
    static constexpr uint32_t kXB = STATS ? (uint32_t)G * 256u : 0u;  // the source tile (statistics)
    static constexpr int WT = STATS ? 4 : 2;                          // consumer warps sharing one stage
    static constexpr uint32_t kCodeRowB = 16u * BITS;
    static constexpr uint32_t kCodesB = (uint32_t)CR * kCodeRowB;
    static constexpr uint32_t kSB = 128u * (SDT == KVQ_F32 ? 4u : 2u);
    static constexpr uint32_t kZB = ZDT == KVQ_NONE ? 0u : 128u * (ZDT == KVQ_I8 ? 1u : ZDT == KVQ_F32 ? 4u : 2u);
    static constexpr uint32_t offCodes = kXB, offS = kXB + kCodesB, offZ = offS + kSB;
    static constexpr uint32_t kStage = (offZ + kZB + 127u) / 128u * 128u;
    static constexpr int kConsumers = 16;                            // consumer warps (+ 1 producer)
    static constexpr int kTeams = kConsumers / WT;                   // a team of WT warps owns two stages
    static constexpr int kStages = 2 * kTeams;
    static constexpr int kThreads = (kConsumers + 1) * 32;
    static constexpr int kSmem = kStages * (int)kStage + 2 * kStages * 8;
    static_assert(kSmem <= 227 * 1024, "ring does not fit in shared memory");
};

template <int BITS, bool ASYM, int G, bool STATS, int SDT, int ZDT>
__global__ void __launch_bounds__(DtShape<BITS, G, STATS, SDT, ZDT>::kThreads, 1)
wds_t_kernel(const QArgs a, Partial* partials, unsigned int* done, kvq_err* out_dev)
{
    using L = DtShape<BITS, G, STATS, SDT, ZDT>;
    using W = typename CodeWord<BITS>::T;
    constexpr int C = 128;
    constexpr int P = L::kTeams, S = L::kStages, WT = L::WT, NCW = L::kConsumers;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * L::kStage);
    uint64_t* empty = full + S;

    constexpr int CR = L::CR, CPG = G / CR;                // rows per chunk, chunks per group
    const QSpec& q = a.q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ng = (uint32_t)q.ngroups;
    const uint32_t nchunks = (uint32_t)q.outer * ng * CPG; // < 2^31, checked by the dispatcher
    const uint32_t Tq32 = (uint32_t)q.Tq, T32 = (uint32_t)q.T;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], WT);
        }
        mbar_init_fence();
    }
    __syncthreads();
    const uint32_t first = blockIdx.x, step = gridDim.x;
    // chunk c -> (outer o, group k, first row, rows); the tail chunks of a
    // short last group may hold no rows (only the group constants are copied)
    auto geom = [&](uint32_t c, uint32_t& o, uint32_t& grp, uint32_t& row0, uint32_t& nrows) {
        grp = c / CPG;
        o = grp / ng;
        const uint32_t k = grp - o * ng;
        row0 = k * (uint32_t)G + (c - grp * CPG) * (uint32_t)CR;
        nrows = row0 < Tq32 ? min((uint32_t)CR, Tq32 - row0) : 0u;
    };

    if (warp == NCW) {
        // ---- producer
        if (lane != 0) return;
        const unsigned char* codes = static_cast<const unsigned char*>(a.codes);
        uint32_t n = 0;
        for (;; ++n) {
            const uint32_t c = first + n * step;
            if (c >= nchunks) break;
            const int s = (int)(n % S);
            if (n >= (uint32_t)S && !mbar_wait(&empty[s], ((n / S) - 1) & 1u)) break;
            uint32_t o, grp, row0, nrows;
            geom(c, o, grp, row0, nrows);
            unsigned char* st = smem + s * L::kStage;
            mbar_expect_tx(&full[s], nrows * (L::kXB ? 256u : 0u) + nrows * L::kCodeRowB + L::kSB + L::kZB);
            if (STATS && nrows)
                bulk_g2s(st, static_cast<const __nv_bfloat16*>(a.x) + ((uint64_t)o * T32 + row0) * C, nrows * 256u, &full[s]);
            if (nrows)
                bulk_g2s(st + L::offCodes, codes + ((uint64_t)o * Tq32 + row0) * L::kCodeRowB, nrows * L::kCodeRowB, &full[s]);
            bulk_g2s(st + L::offS, static_cast<const unsigned char*>(a.scale) + (uint64_t)grp * L::kSB, L::kSB, &full[s]);
            if (L::kZB)
                bulk_g2s(st + L::offZ, static_cast<const unsigned char*>(a.zero) + (uint64_t)grp * L::kZB, L::kZB, &full[s]);
            if (!STATS) {
                // dequantize: the codes one ring-length ahead into L2 (measured
                // faster; the statistics' larger tiles measured slower with it)
                const uint32_t cq = c + (uint32_t)S * step;
                if (cq < nchunks && cq > c) {
                    uint32_t po, pgrp, prow0, pn;
                    geom(cq, po, pgrp, prow0, pn);
                    if (pn) bulk_prefetch_l2(codes + ((uint64_t)po * Tq32 + prow0) * L::kCodeRowB, pn * L::kCodeRowB);
                }
            }
        }
        for (uint32_t i = n > (uint32_t)S ? n - S : 0; i < n; ++i) mbar_wait(&full[i % S], (i / S) & 1u);
        return;
    }

    // ---- consumers: team p of WT warps; warp wt of the team, lane = 8 channels
    // (c8) x rows r0 + 2*WT*i with r0 = 2*wt + (lane >> 4)
    const int pair = warp / WT, wt = warp - pair * WT;
    const int c8 = lane & 15, rq = 2 * wt + (lane >> 4);
    constexpr int RSTEP = 2 * WT;
    const int chan0 = c8 * 8;
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    Acc2 A;
    for (uint32_t j = pair;; j += P) {
        const uint32_t c = first + j * step;
        if (c >= nchunks) break;
        const int s = (int)(j % S);
        // on a timeout (recorded in g_kvq_wait_timeouts) leave the loop but still reach the barriers below
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (j / S) & 1u))) break;
        const unsigned char* st = smem + s * L::kStage;
        uint32_t o, grp, row0, nr;
        geom(c, o, grp, row0, nr);
        const int nrows = (int)nr;
        // the group constants of this lane's eight channels
        float sf[8], zf[8];
        ld_meta8_smem<SDT>(st + L::offS, chan0, sf);
        if (ASYM) ld_meta8_smem<ZDT>(st + L::offZ, chan0, zf);
        u64 cp[4], sp[4];
        bool fast = true;
        const float base = 8388608.0f + (float)off;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float z0 = ASYM ? zf[2 * p] : 0.0f, z1 = ASYM ? zf[2 * p + 1] : 0.0f;
            cp[p] = add2(pk(z0, z1), pk(base, base));
            sp[p] = pk(sf[2 * p], sf[2 * p + 1]);
            if (ASYM) fast = fast && fmaxf(fabsf(z0), fabsf(z1)) < 0x1p21f;
        }
        const unsigned char* cbase = st + L::offCodes + (uint32_t)(chan0 / 8) * BITS;
        const unsigned char* xbase = st + chan0 * 2;
        __nv_bfloat16* obase = out + ((uint64_t)o * T32 + row0) * C + chan0;
        TileAcc ta;
        auto row_from = [&](int r, W cw, const uint4& xw) {
            uint32_t u[8];
            unpack_biased8<BITS>(q.is_signed ? flip_signs<BITS>(cw) : cw, u);
            uint4 ow;
            if (fast) ow = dq8<STATS>(u, cp, sp, xw, ta, A.mxb);
            else ow = dq8_slow<STATS>(u, off, zf, sf, xw, ta, A.mxb);
            if (!STATS) *reinterpret_cast<uint4*>(obase + (uint64_t)r * C) = ow;
        };
        auto row = [&](int r) {
            const W cw = *reinterpret_cast<const W*>(cbase + (uint32_t)r * L::kCodeRowB);
            const uint4 xw = STATS ? *reinterpret_cast<const uint4*>(xbase + (uint32_t)r * 256u) : make_uint4(0, 0, 0, 0);
            row_from(r, cw, xw);
        };
        if (nrows == CR && STATS) {
            // a whole tile: every shared-memory load of the lane's rows first
            constexpr int NR = CR / RSTEP;
            W cws[NR];
            uint4 xws[NR];
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                cws[i] = *reinterpret_cast<const W*>(cbase + (uint32_t)(rq + RSTEP * i) * L::kCodeRowB);
                xws[i] = *reinterpret_cast<const uint4*>(xbase + (uint32_t)(rq + RSTEP * i) * 256u);
            }
#pragma unroll
            for (int i = 0; i < NR; ++i) row_from(rq + RSTEP * i, cws[i], xws[i]);
        } else if (nrows == CR) {
#pragma unroll 4
            for (int i = 0; i < CR / RSTEP; ++i) row(rq + RSTEP * i);
        } else {
            for (int i = 0; i < CR / RSTEP; ++i)
                if (rq + RSTEP * i < nrows) row(rq + RSTEP * i);
        }
        if (STATS) A.fold(ta);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    constexpr int kCons = NCW * 32;                        // consumer threads
    if (!STATS) {
        // residual rows: resid [outer][R][C] -> out rows Tq .. T-1, 16 bytes per item
        const uint64_t nres = (uint64_t)q.outer * (uint64_t)q.R * (C / 8);
        const uint4* rs = static_cast<const uint4*>(a.resid);
        for (uint64_t i = (uint64_t)blockIdx.x * kCons + threadIdx.x; i < nres; i += (uint64_t)gridDim.x * kCons) {
            const uint64_t rr = i / (C / 8), piece = i % (C / 8);
            const uint64_t o = rr / (uint64_t)q.R, t = rr % (uint64_t)q.R;
            *reinterpret_cast<uint4*>(out + ((o * T32 + Tq32 + t) * C + piece * 8)) = rs[i];
        }
        return;
    }

    // ---- block partial over the consumer warps, then the fused final reduction
    __shared__ double w1[NCW], w2[NCW], wm[NCW];
    __shared__ bool s_last;
    double d1, d2, dm;
    warp_partial(A, d1, d2, dm);
    if (lane == 0) { w1[warp] = d1; w2[warp] = d2; wm[warp] = dm; }
    asm volatile("bar.sync 1, %0;" ::"r"(kCons) : "memory");
    if (threadIdx.x == 0) {
        Partial pp = {0.0, 0.0, 0.0};
        for (int i = 0; i < NCW; ++i) { pp.s1 += w1[i]; pp.s2 += w2[i]; pp.mx = fmax(pp.mx, wm[i]); }
        partials[blockIdx.x] = pp;
        __threadfence();
        s_last = atomicAdd(done, 1u) == gridDim.x - 1;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCons) : "memory");
    if (!s_last || warp != 0) return;
    __threadfence();
    // warp 0 of the last CTA: partials in a fixed order (lane l takes l, l+32, ...), then a fixed tree
    double f1 = 0.0, f2 = 0.0, fm = 0.0;
    for (uint32_t i = lane; i < gridDim.x; i += 32) {
        f1 += __ldcg(&partials[i].s1);
        f2 += __ldcg(&partials[i].s2);
        fm = fmax(fm, __ldcg(&partials[i].mx));
    }
    for (int o2 = 16; o2 > 0; o2 >>= 1) {
        f1 += __shfl_xor_sync(0xFFFFFFFFu, f1, o2);
        f2 += __shfl_xor_sync(0xFFFFFFFFu, f2, o2);
        fm = fmax(fm, __shfl_xor_sync(0xFFFFFFFFu, fm, o2));
    }
    if (lane == 0) {
        const double N = (double)q.outer * (double)q.T * (double)q.C;
        out_dev->rmse = sqrt(f2 / N);
        out_dev->max_abs = fm;
        out_dev->mean_abs = f1 / N;
    }
}

// ======================================================================
// dequantize along C, warp-specialised (bf16, C = 128, groups of 32, 64 or
// 128 channels per token).  A chunk is kDcRows consecutive quantized token
// rows of one slice: the producer warp bulk-copies their codes into a ring
// stage (and the codes one ring-length ahead into L2); the group constants
// belong to each token, so every lane loads the scale and zero point of its
// rows' group straight from global memory before it waits on the tile, all
// loads in flight together.  Teams, stages, lane mapping and the residual
// copy are those of wds_t_kernel.  (The statistics along C stay on ds_kernel:
// this form of them measured slower.)
// ======================================================================
constexpr int kDcRows = 64;

template <int BITS>
struct DcShape {
    static constexpr int CR = kDcRows;
    static constexpr int WT = 2;                                      // consumer warps sharing one stage
    static constexpr uint32_t kCodeRowB = 16u * BITS;
    static constexpr uint32_t kStage = ((uint32_t)CR * kCodeRowB + 127u) / 128u * 128u;
    static constexpr int kConsumers = 16;
    static constexpr int kTeams = kConsumers / WT;
    static constexpr int kStages = 2 * kTeams;
    static constexpr int kThreads = (kConsumers + 1) * 32;
    static constexpr int kSmem = kStages * (int)kStage + 2 * kStages * 8;
    static_assert(kSmem <= 227 * 1024, "ring does not fit in shared memory");
};

template <int BITS, bool ASYM, int G, int SDT, int ZDT>
__global__ void __launch_bounds__(DcShape<BITS>::kThreads, 1)
wds_c_kernel(const QArgs a)
{
    using L = DcShape<BITS>;
    using W = typename CodeWord<BITS>::T;
    constexpr int C = 128, NG = C / G, CR = L::CR;
    constexpr int P = L::kTeams, S = L::kStages, WT = L::WT, NCW = L::kConsumers;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * L::kStage);
    uint64_t* empty = full + S;

    const QSpec& q = a.q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t Tq32 = (uint32_t)q.Tq, T32 = (uint32_t)q.T;
    const uint32_t per_o = (Tq32 + CR - 1) / CR;
    const uint32_t nchunks = (uint32_t)q.outer * per_o;      // < 2^31, checked by the dispatcher

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], WT);
        }
        mbar_init_fence();
    }
    __syncthreads();
    const uint32_t first = blockIdx.x, step = gridDim.x;
    auto geom = [&](uint32_t c, uint32_t& o, uint32_t& row0, uint32_t& nrows) {
        o = c / per_o;
        row0 = (c - o * per_o) * (uint32_t)CR;
        nrows = min((uint32_t)CR, Tq32 - row0);
    };

    if (warp == NCW) {
        // ---- producer
        if (lane != 0) return;
        const unsigned char* codes = static_cast<const unsigned char*>(a.codes);
        uint32_t n = 0;
        for (;; ++n) {
            const uint32_t c = first + n * step;
            if (c >= nchunks) break;
            const int s = (int)(n % S);
            if (n >= (uint32_t)S && !mbar_wait(&empty[s], ((n / S) - 1) & 1u)) break;
            uint32_t o, row0, nrows;
            geom(c, o, row0, nrows);
            mbar_expect_tx(&full[s], nrows * L::kCodeRowB);
            bulk_g2s(smem + s * L::kStage, codes + ((uint64_t)o * Tq32 + row0) * L::kCodeRowB, nrows * L::kCodeRowB,
                     &full[s]);
            const uint32_t cq = c + (uint32_t)S * step;        // the codes one ring-length ahead into L2
            if (cq < nchunks && cq > c) {
                uint32_t po, prow0, pn;
                geom(cq, po, prow0, pn);
                bulk_prefetch_l2(codes + ((uint64_t)po * Tq32 + prow0) * L::kCodeRowB, pn * L::kCodeRowB);
            }
        }
        for (uint32_t i = n > (uint32_t)S ? n - S : 0; i < n; ++i) mbar_wait(&full[i % S], (i / S) & 1u);
        return;
    }

    // ---- consumers: team p of WT warps; warp wt of the team, lane = 8 channels
    // (c8) x rows r0 + 2*WT*i with r0 = 2*wt + (lane >> 4)
    const int pair = warp / WT, wt = warp - pair * WT;
    const int c8 = lane & 15, rq = 2 * wt + (lane >> 4);
    constexpr int RSTEP = 2 * WT, NR = CR / RSTEP;
    const int chan0 = c8 * 8, grp = chan0 / G;
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    TileAcc ta;                                             // unused: dequantize only
    uint32_t mxb = 0;
    for (uint32_t j = pair;; j += P) {
        const uint32_t c = first + j * step;
        if (c >= nchunks) break;
        uint32_t o, row0, nr;
        geom(c, o, row0, nr);
        const int nrows = (int)nr;
        // this lane's rows' group constants, all loads issued before the wait
        float sr[NR], zr[NR];
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const int r = rq + RSTEP * i;
            const int64_t mi = ((int64_t)o * q.Tq + row0 + (r < nrows ? r : 0)) * NG + grp;
            sr[i] = ld_meta<SDT>(a.scale, mi);
            zr[i] = ASYM ? ld_meta<ZDT>(a.zero, mi) : 0.0f;
        }
        const int s = (int)(j % S);
        // on a timeout (recorded in g_kvq_wait_timeouts) leave the loop
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (j / S) & 1u))) break;
        const unsigned char* cbase = smem + s * L::kStage + (uint32_t)c8 * BITS;
        __nv_bfloat16* obase = out + ((uint64_t)o * T32 + row0) * C + chan0;
#pragma unroll
        for (int i = 0; i < NR; ++i) {                     // fully unrolled: sr / zr stay in registers
            const int r = rq + RSTEP * i;
            if (r < nrows) {
                const W cw = *reinterpret_cast<const W*>(cbase + (uint32_t)r * L::kCodeRowB);
                uint32_t u[8];
                unpack_biased8<BITS>(q.is_signed ? flip_signs<BITS>(cw) : cw, u);
                uint4 ow;
                if (!ASYM || fabsf(zr[i]) < 0x1p21f) {
                    u64 c1, s1;
                    dq_pair_consts(sr[i], zr[i], off, c1, s1);
                    const u64 cp[4] = {c1, c1, c1, c1}, sp[4] = {s1, s1, s1, s1};
                    ow = dq8<false>(u, cp, sp, make_uint4(0, 0, 0, 0), ta, mxb);
                } else {
                    // exact reference order for groups with a very large zero point
                    float sf[8], zf[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) { sf[k] = sr[i]; zf[k] = zr[i]; }
                    ow = dq8_slow<false>(u, off, zf, sf, make_uint4(0, 0, 0, 0), ta, mxb);
                }
                *reinterpret_cast<uint4*>(obase + (uint64_t)r * C) = ow;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }

    // residual rows: resid [outer][R][C] -> out rows Tq .. T-1, 16 bytes per item
    constexpr int kCons = NCW * 32;                        // consumer threads
    const uint64_t nres = (uint64_t)q.outer * (uint64_t)q.R * (C / 8);
    const uint4* rs = static_cast<const uint4*>(a.resid);
    for (uint64_t i = (uint64_t)blockIdx.x * kCons + threadIdx.x; i < nres; i += (uint64_t)gridDim.x * kCons) {
        const uint64_t rr = i / (C / 8), piece = i % (C / 8);
        const uint64_t o = rr / (uint64_t)q.R, t = rr % (uint64_t)q.R;
        *reinterpret_cast<uint4*>(out + ((o * T32 + Tq32 + t) * C + piece * 8)) = rs[i];
    }
}

int log2_exact(int64_t v) {
    int l = 0;
    while ((int64_t(1) << l) < v) ++l;
    return (int64_t(1) << l) == v ? l : -1;
}

// Metadata layouts with dedicated kernels: 0 = bf16 scale + bf16 zero,
// 1 = f32 scale + int8 zero (asymmetric); 2 = bf16 scale, 3 = f32 scale
// (symmetric).  -1: handled by the other paths.
int meta_kind(const QSpec& q) {
    if (q.mode == KVQ_ASYM) {
        if (q.scale_dt == KVQ_BF16 && q.zero_dt == KVQ_BF16) return 0;
        if (q.scale_dt == KVQ_F32 && q.zero_dt == KVQ_I8) return 1;
        return -1;
    }
    return q.scale_dt == KVQ_BF16 ? 2 : 3;
}

template <typename K>
bool ensure_smem(K kernel, int bytes = kStagedSmem) {
    return ensure_kernel_attrs(reinterpret_cast<const void*>(kernel), bytes) == cudaSuccess;
}

unsigned staged_grid(int sms, uint64_t nchunks) {
    // three CTAs of 64 KB ring per SM
    return (unsigned)std::max<uint64_t>(1, std::min<uint64_t>(nchunks, (uint64_t)sms * 3));
}

bool staged_t_ok(const QSpec& q) {
    return q.x_dt == KVQ_BF16 && q.aligned && q.C == 128 && q.g * q.C * 2 <= kStageBytes && q.Tq > 0 &&
           meta_kind(q) >= 0 && q.outer * (q.ngroups + (q.R + q.g - 1) / q.g) < (int64_t(1) << 31);
}
bool staged_c_ok(const QSpec& q) {
    if (q.x_dt != KVQ_BF16 || !q.aligned || q.C % 32 != 0 || q.C > kStageBytes / 2) return false;
    if ((kStageBytes / 2) % q.C != 0 || meta_kind(q) < 0) return false;      // whole rows per chunk
    if (q.outer * q.T >= (int64_t(1) << 31)) return false;
    const int64_t g = q.g;
    return q.C % g == 0 && (g == 32 || g == 64 || g == 128);
}

template <int BITS, bool ASYM, int G, int SDT, int ZDT>
void wq_t_launch(const QArgs& a, uint64_t nchunks, cudaStream_t st) {
    const unsigned grid = (unsigned)std::max<uint64_t>(1, std::min<uint64_t>(nchunks, (uint64_t)sm_count()));
    if (!ensure_smem(wq_t_kernel<BITS, ASYM, G, SDT, ZDT>, kWSmem)) return;    // the error stays the last error
    wq_t_kernel<BITS, ASYM, G, SDT, ZDT><<<grid, kWThreads, kWSmem, st>>>(a);
}

template <int BITS, bool ASYM, int SDT, int ZDT>
void sq_t_launch(const QArgs& a, cudaStream_t st) {
    const QSpec& q = a.q;
    const uint64_t nchunks = (uint64_t)q.outer * (q.ngroups + (q.R + q.g - 1) / q.g);
    switch (q.g) {
    case 16: wq_t_launch<BITS, ASYM, 16, SDT, ZDT>(a, nchunks, st); return;
    case 32: wq_t_launch<BITS, ASYM, 32, SDT, ZDT>(a, nchunks, st); return;
    case 64: wq_t_launch<BITS, ASYM, 64, SDT, ZDT>(a, nchunks, st); return;
    default: break;
    }
    const unsigned grid = staged_grid(sm_count(), nchunks);
    if (!ensure_smem(sq_t_kernel<BITS, ASYM, 128, SDT, ZDT>)) return;
    sq_t_kernel<BITS, ASYM, 128, SDT, ZDT><<<grid, kThr, kStagedSmem, st>>>(a);
}

// The driver's tensor-map encoder, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &r) != cudaSuccess ||
            r != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// [rows, 128] bf16 rows of x as boxes of 64 channels x kCRows rows, 128-byte swizzle.
bool encode_rows_map(const QSpec& q, const void* x, CUtensorMap* map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)q.C, (cuuint64_t)(q.outer * q.T)};
    const cuuint64_t strides[1] = {(cuuint64_t)q.C * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kCRows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BITS, bool ASYM, int G, int SDT, int ZDT>
bool wq_c_launch(const QArgs& a, cudaStream_t st) {
    const QSpec& q = a.q;
    CUtensorMap map;
    if (!encode_rows_map(q, a.x, &map)) return false;
    const uint64_t nchunks = ((uint64_t)q.outer * q.T + kCRows - 1) / kCRows;
    const unsigned grid = (unsigned)std::max<uint64_t>(1, std::min<uint64_t>(nchunks, (uint64_t)sm_count()));
    if (!ensure_smem(wq_c_kernel<BITS, ASYM, G, SDT, ZDT>, kCSmem)) return true;    // the error stays the last error
    wq_c_kernel<BITS, ASYM, G, SDT, ZDT><<<grid, kCThreads, kCSmem, st>>>(a, map);
    return true;
}

template <int BITS, bool ASYM, int SDT, int ZDT>
void sq_c_launch(const QArgs& a, cudaStream_t st) {
    const QSpec& q = a.q;
    if (q.C == 128) {
        bool done = false;
        switch (q.g) {
        case 32: done = wq_c_launch<BITS, ASYM, 32, SDT, ZDT>(a, st); break;
        case 64: done = wq_c_launch<BITS, ASYM, 64, SDT, ZDT>(a, st); break;
        case 128: done = wq_c_launch<BITS, ASYM, 128, SDT, ZDT>(a, st); break;
        default: break;
        }
        if (done) return;
    }
    const uint64_t rc = kStageBytes / (2 * q.C);
    const uint64_t nchunks = ((uint64_t)q.outer * q.T + rc - 1) / rc;
    const unsigned grid = staged_grid(sm_count(), nchunks);
    switch (q.g) {
    case 32: if (ensure_smem(sq_c_kernel<BITS, ASYM, 32, SDT, ZDT>)) sq_c_kernel<BITS, ASYM, 32, SDT, ZDT><<<grid, kThr, kStagedSmem, st>>>(a); break;
    case 64: if (ensure_smem(sq_c_kernel<BITS, ASYM, 64, SDT, ZDT>)) sq_c_kernel<BITS, ASYM, 64, SDT, ZDT><<<grid, kThr, kStagedSmem, st>>>(a); break;
    default: if (ensure_smem(sq_c_kernel<BITS, ASYM, 128, SDT, ZDT>)) sq_c_kernel<BITS, ASYM, 128, SDT, ZDT><<<grid, kThr, kStagedSmem, st>>>(a); break;
    }
}

// (bits, meta kind) -> a launcher templated on the mode and metadata dtypes
template <template <int, bool, int, int> class L>
void by_meta(const QArgs& a, cudaStream_t st) {
    const int mk = meta_kind(a.q);
    switch (a.q.bits) {
    case 8:
        if (mk == 0) L<8, true, KVQ_BF16, KVQ_BF16>::run(a, st);
        else if (mk == 1) L<8, true, KVQ_F32, KVQ_I8>::run(a, st);
        else if (mk == 2) L<8, false, KVQ_BF16, KVQ_NONE>::run(a, st);
        else L<8, false, KVQ_F32, KVQ_NONE>::run(a, st);
        break;
    case 4:
        if (mk == 0) L<4, true, KVQ_BF16, KVQ_BF16>::run(a, st);
        else if (mk == 1) L<4, true, KVQ_F32, KVQ_I8>::run(a, st);
        else if (mk == 2) L<4, false, KVQ_BF16, KVQ_NONE>::run(a, st);
        else L<4, false, KVQ_F32, KVQ_NONE>::run(a, st);
        break;
    default:
        if (mk == 0) L<2, true, KVQ_BF16, KVQ_BF16>::run(a, st);
        else if (mk == 1) L<2, true, KVQ_F32, KVQ_I8>::run(a, st);
        else if (mk == 2) L<2, false, KVQ_BF16, KVQ_NONE>::run(a, st);
        else L<2, false, KVQ_F32, KVQ_NONE>::run(a, st);
        break;
    }
}

template <int B, bool A, int S, int Z> struct SqT { static void run(const QArgs& a, cudaStream_t st) { sq_t_launch<B, A, S, Z>(a, st); } };
template <int B, bool A, int S, int Z> struct SqC { static void run(const QArgs& a, cudaStream_t st) { sq_c_launch<B, A, S, Z>(a, st); } };

// ---- dequantize / statistics geometry
// rows per lane item: 8 for dequantize along T (group constants shared by
// more rows), else 4 (fewer registers, more resident warps)
int ds_rpt(const QSpec& q, bool stats) { return (!stats && q.axis == KVQ_GROUP_ALONG_T && q.g % 8 == 0) ? 8 : 4; }

bool ds_ok(const QSpec& q) {
    if (q.x_dt != KVQ_BF16 || !q.aligned || q.C % 8 != 0 || log2_exact(q.C / 8) < 0 || meta_kind(q) < 0) return false;
    if (log2_exact(q.g) < 0) return false;
    if (q.axis == KVQ_GROUP_ALONG_T) return q.g % 4 == 0;
    return q.g % 8 == 0 && q.C % q.g == 0;
}

// blocks_per_sm resident blocks on each of sms SMs, at most one item per thread
dim3 ds_grid(const QSpec& q, int sms, bool stats, int blocks_per_sm = 8) {
    const int lcpr = log2_exact(q.C / 8);
    const int rpt = ds_rpt(q, stats);
    const uint64_t items = (uint64_t)((q.T + rpt - 1) / rpt) << lcpr;
    const unsigned gy = (unsigned)std::max<int64_t>(1, std::min<int64_t>(q.outer, 65535));
    const uint64_t want_total = (uint64_t)sms * (uint64_t)std::max(blocks_per_sm, 1);
    const uint64_t gx = std::max<uint64_t>(1, std::min<uint64_t>((items + kThr - 1) / kThr, want_total / gy));
    return dim3((unsigned)gx, gy);
}

// resident blocks per SM of a kernel at kThr threads, queried once per kernel
// (a small table keyed by the kernel's address)
template <typename K>
int resident_blocks(K kernel) {
    constexpr int kSlots = 256;
    static const void* keys[kSlots];
    static int vals[kSlots];
    static std::mutex mu;
    const void* key = reinterpret_cast<const void*>(kernel);
    std::lock_guard<std::mutex> lock(mu);
    int i = 0;
    for (; i < kSlots && keys[i]; ++i)
        if (keys[i] == key) return vals[i];
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThr, 0) != cudaSuccess || b < 1) b = 1;
    if (i < kSlots) { keys[i] = key; vals[i] = b; }
    return b;
}

// Launch context of the statistics pass: block partials, and (when the
// final reduction is fused) the completion counter and the result.
struct DsStats { Partial* partials; unsigned int* done; kvq_err* out; };

template <bool STATS>
struct DsL {
    template <int B, bool A, int S, int Z> struct L {
        template <typename K>
        static void go(K kernel, const QArgs& a, const DsStats& ctx, cudaStream_t st) {
            const QSpec& q = a.q;
            const dim3 grid = ds_grid(q, sm_count(), STATS, resident_blocks(kernel));
            kernel<<<grid, kThr, 0, st>>>(a, log2_exact(q.C / 8), log2_exact(q.g), ctx.partials, ctx.done, ctx.out);
        }
        static void run(const QArgs& a, const DsStats& ctx, cudaStream_t st) {
            const QSpec& q = a.q;
            if (q.axis == KVQ_GROUP_ALONG_T) {
                if (ds_rpt(q, STATS) == 8) go(ds_kernel<B, A, true, 8, STATS, S, Z>, a, ctx, st);
                else go(ds_kernel<B, A, true, 4, STATS, S, Z>, a, ctx, st);
            } else {
                go(ds_kernel<B, A, false, 4, STATS, S, Z>, a, ctx, st);
            }
        }
    };
};

// (bits, meta kind) dispatch for launchers that take the statistics context
template <template <int, bool, int, int> class L>
void by_meta_ctx(const QArgs& a, const DsStats& ctx, cudaStream_t st) {
    const int mk = meta_kind(a.q);
    switch (a.q.bits) {
    case 8:
        if (mk == 0) L<8, true, KVQ_BF16, KVQ_BF16>::run(a, ctx, st);
        else if (mk == 1) L<8, true, KVQ_F32, KVQ_I8>::run(a, ctx, st);
        else if (mk == 2) L<8, false, KVQ_BF16, KVQ_NONE>::run(a, ctx, st);
        else L<8, false, KVQ_F32, KVQ_NONE>::run(a, ctx, st);
        break;
    case 4:
        if (mk == 0) L<4, true, KVQ_BF16, KVQ_BF16>::run(a, ctx, st);
        else if (mk == 1) L<4, true, KVQ_F32, KVQ_I8>::run(a, ctx, st);
        else if (mk == 2) L<4, false, KVQ_BF16, KVQ_NONE>::run(a, ctx, st);
        else L<4, false, KVQ_F32, KVQ_NONE>::run(a, ctx, st);
        break;
    default:
        if (mk == 0) L<2, true, KVQ_BF16, KVQ_BF16>::run(a, ctx, st);
        else if (mk == 1) L<2, true, KVQ_F32, KVQ_I8>::run(a, ctx, st);
        else if (mk == 2) L<2, false, KVQ_BF16, KVQ_NONE>::run(a, ctx, st);
        else L<2, false, KVQ_F32, KVQ_NONE>::run(a, ctx, st);
        break;
    }
}

}  // namespace

// ---- warp-specialised dequantize / statistics along T
bool wds_t_ok(const QSpec& q) {
    return q.axis == KVQ_GROUP_ALONG_T && q.x_dt == KVQ_BF16 && q.aligned && q.C == 128 &&
           (q.g == 16 || q.g == 32 || q.g == 64) && meta_kind(q) >= 0 && q.Tq > 0 &&
           q.outer * q.ngroups * 2 < (int64_t(1) << 31) && q.outer * q.T < (int64_t(1) << 31);
}

template <bool STATS>
struct WdsL {
    template <int B, bool A, int S, int Z> struct L {
        template <int G>
        static void go(const QArgs& a, const DsStats& ctx, cudaStream_t st) {
            using Sh = DtShape<B, G, STATS, S, Z>;
            auto kernel = wds_t_kernel<B, A, G, STATS, S, Z>;
            if (!ensure_smem(kernel, Sh::kSmem)) return;        // the error stays the last error
            const uint64_t nchunks = (uint64_t)a.q.outer * a.q.ngroups * (G / Sh::CR);
            const unsigned grid = (unsigned)std::max<uint64_t>(1, std::min<uint64_t>(nchunks, (uint64_t)sm_count()));
            kernel<<<grid, Sh::kThreads, Sh::kSmem, st>>>(a, ctx.partials, ctx.done, ctx.out);
        }
        static void run(const QArgs& a, const DsStats& ctx, cudaStream_t st) {
            switch (a.q.g) {
            case 16: go<16>(a, ctx, st); break;
            case 32: go<32>(a, ctx, st); break;
            default: go<64>(a, ctx, st); break;
            }
        }
    };
};

// ---- warp-specialised dequantize along C
bool wds_c_ok(const QSpec& q) {
    return q.axis == KVQ_GROUP_ALONG_C && q.x_dt == KVQ_BF16 && q.aligned && q.C == 128 &&
           (q.g == 32 || q.g == 64 || q.g == 128) && meta_kind(q) >= 0 && q.Tq > 0 &&
           q.outer * ((q.Tq + kDcRows - 1) / kDcRows) < (int64_t(1) << 31) && q.outer * q.T < (int64_t(1) << 31);
}

struct WdcL {
    template <int B, bool A, int S, int Z> struct L {
        template <int G>
        static void go(const QArgs& a, cudaStream_t st) {
            using Sh = DcShape<B>;
            auto kernel = wds_c_kernel<B, A, G, S, Z>;
            if (!ensure_smem(kernel, Sh::kSmem)) return;        // the error stays the last error
            const uint64_t nchunks = (uint64_t)a.q.outer * ((a.q.Tq + kDcRows - 1) / kDcRows);
            const unsigned grid = (unsigned)std::max<uint64_t>(1, std::min<uint64_t>(nchunks, (uint64_t)sm_count()));
            kernel<<<grid, Sh::kThreads, Sh::kSmem, st>>>(a);
        }
        static void run(const QArgs& a, const DsStats&, cudaStream_t st) {
            switch (a.q.g) {
            case 32: go<32>(a, st); break;
            case 64: go<64>(a, st); break;
            default: go<128>(a, st); break;
            }
        }
    };
};

// ---- entry points (see kvq_internal.h)

void* tensor_map_encode_fn() { return reinterpret_cast<void*>(tensor_map_encoder()); }

bool staged_quantize_supported(const QSpec& q)
{
    return q.axis == KVQ_GROUP_ALONG_T ? staged_t_ok(q) : staged_c_ok(q);
}

bool staged_quantize(const QArgs& a, cudaStream_t st)
{
    const QSpec& q = a.q;
    if (q.axis == KVQ_GROUP_ALONG_T && staged_t_ok(q)) { by_meta<SqT>(a, st); return true; }
    if (q.axis == KVQ_GROUP_ALONG_C && staged_c_ok(q)) { by_meta<SqC>(a, st); return true; }
    return false;
}

bool stream_dequant_supported(const QSpec& q, int out_dt) { return out_dt == KVQ_BF16 && ds_ok(q) && q.Tq > 0; }

cudaError_t stream_dequantize(const QArgs& a, cudaStream_t st)
{
    if (wds_t_ok(a.q)) by_meta_ctx<WdsL<false>::L>(a, DsStats{nullptr, nullptr, nullptr}, st);
    else if (wds_c_ok(a.q)) by_meta_ctx<WdcL::L>(a, DsStats{nullptr, nullptr, nullptr}, st);
    else by_meta_ctx<DsL<false>::L>(a, DsStats{nullptr, nullptr, nullptr}, st);
    return cudaGetLastError();
}

int64_t stream_stats_blocks(const QSpec& q, int sms)
{
    if (!ds_ok(q)) return -1;
    const dim3 g = ds_grid(q, sms, true);      // an upper bound: at most 8 blocks per SM
    return (int64_t)g.x * g.y;
}

cudaError_t stream_error_stats(const QArgs& a, void* partials, unsigned int* done, kvq_err* out_dev, cudaStream_t st)
{
    // the warp-specialised kernel always fuses the final reduction (needs done)
    if (done && wds_t_ok(a.q)) by_meta_ctx<WdsL<true>::L>(a, DsStats{static_cast<Partial*>(partials), done, out_dev}, st);
    else by_meta_ctx<DsL<true>::L>(a, DsStats{static_cast<Partial*>(partials), done, out_dev}, st);
    return cudaGetLastError();
}

}  // namespace kvq
