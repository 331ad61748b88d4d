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
//
// Kernels.  A CTA takes a chunk of one slice (at most 32 chunks per slice) and
// finds its first record offset by summing the record sizes of the tags before
// it (a few KB of L2 reads), so no pass over the whole slice precedes it.  It
// then walks sub-rounds of 16384/C tokens, whose records fit a 32 KB
// shared-memory stage: a block scan of the record sizes gives the offsets, the
// tokens are bucketed by tag so that a warp mostly runs one format, each token
// is handled by C/32 lanes of 32 channels (group constants once per 32
// channels), the records are built in the stage, and the stage goes to memory
// with 16-byte stores (records start at even offsets only).  Dequantization
// mirrors it: 16-byte loads of the sub-round's record bytes into the stage,
// bucketing, decode, 16-byte stores of the rows.
#include <algorithm>

#include "kvq_bulk.cuh"
#include "kvq_elem.cuh"

namespace kvq {

namespace {

using namespace elem;

// record bytes of a token with tag g (0..3 -> 2/4/8/16 bits) and C channels
__host__ __device__ __forceinline__ int64_t record_bytes(int g, int64_t C) {
    return g == 0 ? C / 4 + 2 : g == 1 ? C / 2 + 2 : g == 2 ? C + 4 : 2 * C;
}

struct MixedFormats { QSpec f2, f4, f8; };                         // per-token formats of tags 0, 1, 2

constexpr int kXThreads = 256;
constexpr int kXWarps = kXThreads / 32;
constexpr int kMaxChunks = 32;                                     // CTAs per slice at most

// Tokens per sub-round: quantize stages up to kQStage bytes of records per
// sub-round (16-bit records included), dequantize 32 KB.
constexpr int kQStage = 32768;
template <int C> constexpr int qsub_tokens() { return kQStage / (2 * C) < kXThreads ? kQStage / (2 * C) : kXThreads; }
template <int C> constexpr int dsub_tokens() { return 16384 / C; }

// Order this thread's earlier generic accesses of shared memory before later
// bulk copies into it.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Exclusive prefix of v over the block's threads (all threads call); *total
// receives the sum.  Uses ws[kXWarps].
__device__ __forceinline__ int block_excl_scan(int v, int* ws, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += u;
    }
    if (lane == 31) ws[warp] = incl;
    __syncthreads();
    int before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kXWarps; ++w) {
        const int x = ws[w];
        before += w < warp ? x : 0;
        all += x;
    }
    *total = all;
    return before + incl - v;
}

// Bytes [0, total) of the stage (from byte s0, s0 = the global start's
// address mod 16) to global memory at g (even address): whole 16-byte blocks
// with 16-byte stores, the partial first and last blocks in 2-byte pieces.
__device__ __forceinline__ void stage_to_global(const unsigned char* stage, uint32_t s0, uint32_t total, uint8_t* g) {
    unsigned char* a0 = g - s0;                                    // 16-byte aligned
    const uint32_t end = s0 + total, nblk = (end + 15) / 16;
    for (uint32_t b = threadIdx.x; b < nblk; b += kXThreads) {
        const uint32_t lo = b * 16, hi = lo + 16;
        if (lo >= s0 && hi <= end) {
            *reinterpret_cast<uint4*>(a0 + lo) = *reinterpret_cast<const uint4*>(stage + lo);
        } else {
            for (uint32_t k = max(lo, s0); k < min(hi, end); k += 2)
                *reinterpret_cast<uint16_t*>(a0 + k) = *reinterpret_cast<const uint16_t*>(stage + k);
        }
    }
}
// nw 32-bit words to a 2-byte aligned shared-memory address.
__device__ __forceinline__ void put_words(unsigned char* p, const uint32_t* w, int nw) {
    if (((uintptr_t)p & 3u) == 0) {
        for (int i = 0; i < nw; ++i) reinterpret_cast<uint32_t*>(p)[i] = w[i];
    } else {
        for (int i = 0; i < nw; ++i) {
            reinterpret_cast<uint16_t*>(p)[2 * i] = (uint16_t)w[i];
            reinterpret_cast<uint16_t*>(p)[2 * i + 1] = (uint16_t)(w[i] >> 16);
        }
    }
}
__device__ __forceinline__ void get_words(const unsigned char* p, uint32_t* w, int nw) {
    if (((uintptr_t)p & 3u) == 0) {
        for (int i = 0; i < nw; ++i) w[i] = reinterpret_cast<const uint32_t*>(p)[i];
    } else {
        for (int i = 0; i < nw; ++i)
            w[i] = (uint32_t)reinterpret_cast<const uint16_t*>(p)[2 * i] |
                   ((uint32_t)reinterpret_cast<const uint16_t*>(p)[2 * i + 1] << 16);
    }
}

// Codes of 32 channels (four 16-byte words of bf16) in one record format,
// by the exact fast quotient when the group allows it (the same constants and
// steps as the uniform per-token kernels), else by the IEEE division; the
// BITS*4 bytes as 32-bit words.
template <int BITS, bool ASYM>
__device__ __forceinline__ void codes32(const uint4 (&v)[4], const GroupC& gc, const QSpec& q, uint32_t* out) {
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    typename CodeWord<BITS>::T cw[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint32_t cc[8];
        if (gc.fast) {
            QuotK kq[4];
            kq[0].ns = pk(-gc.s, -gc.s);
            kq[0].inv = pk(gc.inv, gc.inv);
            kq[1] = kq[2] = kq[3] = kq[0];
            int32_t zo[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) zo[j] = gc.zoff;
            if (!ASYM || gc.lo_ok) codes8_fast<ASYM, false>(v[k], kq, zo, q.qmin + off, q.qmax + off, cc);
            else codes8_fast<ASYM, true>(v[k], kq, zo, q.qmin + off, q.qmax + off, cc);
        } else {
            float s8[8], z8[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) { s8[j] = gc.s; z8[j] = gc.zp; }
            codes8_slow<ASYM>(v[k], s8, z8, q, off, cc);
        }
        cw[k] = finish_word<BITS>(cc, q.is_signed);
    }
    if constexpr (BITS == 8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) { out[2 * k] = cw[k].x; out[2 * k + 1] = cw[k].y; }
    } else if constexpr (BITS == 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) out[k] = cw[k];
    } else {
        out[0] = (uint32_t)cw[0] | ((uint32_t)cw[1] << 16);
        out[1] = (uint32_t)cw[2] | ((uint32_t)cw[3] << 16);
    }
}

// The chunk's first record offset: bytes of the slice's records before token t0.
__device__ __forceinline__ int64_t bytes_before(const uint8_t* tg, int64_t t0, int64_t C, int64_t* red) {
    int64_t acc = 0;
    for (int64_t i = threadIdx.x; i < t0; i += kXThreads) acc += record_bytes(tg[i] & 3, C);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, d);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    int64_t all = 0;
#pragma unroll
    for (int w = 0; w < kXWarps; ++w) all += red[w];
    return all;
}

// Tokens of the sub-round grouped by tag: order[] lists them tag 0 first.
// g < 0 for threads without a token.  cnt[4] must be zero on entry.
__device__ __forceinline__ void bucket_by_tag(int g, int* cnt, uint8_t* order) {
    int pos = 0;
    if (g >= 0) pos = atomicAdd(&cnt[g], 1);
    __syncthreads();
    if (g >= 0) {
        int start = 0;
        for (int k = 0; k < g; ++k) start += cnt[k];
        order[start + pos] = (uint8_t)threadIdx.x;
    }
    __syncthreads();
}

// CTA (chunk of `chunk` tokens, slice o).  The chunk's first record offset
// comes from its tags before it; then per sub-round of qsub_tokens<C>()
// tokens (records of up to kQStage bytes): a block scan gives the records'
// offsets (written to off[], with the packed tags), the tokens are bucketed by
// tag, warps build the records (lane = 32 channels read straight from global
// memory, C/32 lanes per token, so a warp mostly runs one format) into a
// shared-memory stage, and the stage goes out with 16-byte stores.
template <int C>
__global__ void __launch_bounds__(kXThreads)
mixed_quant_kernel(const __nv_bfloat16* x, const uint8_t* tags, int64_t T, int64_t chunk, int64_t* off,
                   uint8_t* tags2, uint8_t* stream, const MixedFormats F)
{
    constexpr int LPT = C / 32, TPW = 32 / LPT, SUB = qsub_tokens<C>();
    static_assert(SUB <= kXThreads && SUB % 4 == 0, "one token per thread, whole tag bytes");
    extern __shared__ __align__(128) unsigned char smem_raw[];    // the record stage, kQStage + 16 bytes
    unsigned char* stage = smem_raw + ((16u - (smem_u32(smem_raw) & 15u)) & 15u);
    __shared__ int32_t roff[SUB];
    __shared__ uint8_t tg_s[SUB], order[SUB];
    __shared__ int ws[kXWarps], cnt[4];
    __shared__ int64_t red[kXWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t o = blockIdx.y;
    const int64_t t_lo = (int64_t)blockIdx.x * chunk, t_hi = min(T, t_lo + chunk);
    const uint8_t* tg = tags + o * T;
    uint8_t* sl = stream + o * T * 2 * C;
    // the source rows of a sub-round are contiguous: the first one into L2 now,
    // each following one a sub-round ahead, so the bucketed loads hit L2
    auto prefetch_rows = [&](int64_t r0) {
        if (tid == 0 && r0 < t_hi)
            bulk_prefetch_l2(x + ((uint64_t)o * T + r0) * C, (uint32_t)min((int64_t)SUB, t_hi - r0) * (uint32_t)(2 * C));
    };
    prefetch_rows(t_lo);
    int64_t base = bytes_before(tg, t_lo, C, red);
    for (int64_t sr = t_lo; sr < t_hi; sr += SUB) {
        prefetch_rows(sr + SUB);
        const int n = (int)min((int64_t)SUB, t_hi - sr);
        const int g = tid < n ? (tg[sr + tid] & 3) : -1;
        if (tid < 4) cnt[tid] = 0;
        int total;
        const int ex = block_excl_scan(g >= 0 ? (int)record_bytes(g, C) : 0, ws, &total);
        if (g >= 0) {
            roff[tid] = ex;
            tg_s[tid] = (uint8_t)g;
            off[o * (T + 1) + sr + tid] = base + ex;
        }
        if (tid == 0 && sr + n == T) off[o * (T + 1) + T] = base + total;
        bucket_by_tag(g, cnt, order);
        if (tid < (n + 3) / 4) {                                   // sr is a multiple of 4
            uint32_t bt = 0;
            for (int j = 0; j < 4 && 4 * tid + j < n; ++j) bt |= (uint32_t)tg_s[4 * tid + j] << (2 * j);
            tags2[o * ((T + 3) / 4) + sr / 4 + tid] = (uint8_t)bt;
        }
        const uint32_t s0 = (uint32_t)((uintptr_t)(sl + base) & 15u);
        for (int e0 = warp * TPW; e0 < n; e0 += kXWarps * TPW) {
            const int e = e0 + lane / LPT, q = lane % LPT;
            const bool live = e < n;
            const int tk = live ? order[e] : 0;
            uint4 v[4];
            const uint4* src = reinterpret_cast<const uint4*>(x + ((uint64_t)o * T + sr + tk) * C + q * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = live ? __ldcs(src + j) : make_uint4(0u, 0u, 0u, 0u);
            uint32_t mn = kBfPosInf2, mx = kBfNegInf2, am = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) { fold_minmax(v[j], mn, mx); fold_absmax(v[j], am); }
#pragma unroll
            for (int d = 1; d < LPT; d <<= 1) {
                mn = bmin2(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, d));
                mx = bmax2(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, d));
                am = bmax2(am, __shfl_xor_sync(0xFFFFFFFFu, am, d));
            }
            if (!live) continue;
            const int gt = tg_s[tk];
            unsigned char* rec = stage + s0 + roff[tk];
            if (gt == 3) {                                         // 16 bits: the values as stored
                const uint32_t w[16] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w,
                                        v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
                put_words(rec + q * 64, w, 16);
                continue;
            }
            const float fmn = fminf(lo_f(mn), hi_f(mn)), fmx = fmaxf(lo_f(mx), hi_f(mx));
            const float fam = fmaxf(lo_f(am), hi_f(am));
            uint32_t cw[8];
            GroupC gc;
            int bits;
            if (gt == 2) {
                gc = make_group<true>(fmn, fmx, F.f8, 0);
                codes32<8, true>(v, gc, F.f8, cw);
                put_words(rec + q * 32, cw, 8);
                bits = 8;
            } else if (gt == 1) {
                gc = make_group<false>(0.0f, fam, F.f4, 8);
                codes32<4, false>(v, gc, F.f4, cw);
                put_words(rec + q * 16, cw, 4);
                bits = 4;
            } else {
                gc = make_group<false>(0.0f, fam, F.f2, 2);
                codes32<2, false>(v, gc, F.f2, cw);
                put_words(rec + q * 8, cw, 2);
                bits = 2;
            }
            if (q == 0) {
                const int pb = C * bits / 8;
                *reinterpret_cast<__nv_bfloat16*>(rec + pb) = __float2bfloat16_rn(gc.s);
                if (gt == 2) *reinterpret_cast<__nv_bfloat16*>(rec + pb + 2) = __float2bfloat16_rn(gc.zp);
            }
        }
        __syncthreads();
        stage_to_global(stage, s0, (uint32_t)total, sl + base);
        __syncthreads();
        base += total;
    }
}

// CTA (chunk, slice o), per sub-round of dsub_tokens<C>() tokens: the
// records' bytes (the 16-byte aligned span around them) arrive by a bulk copy
// into one of two 32 KB shared-memory stages, the next sub-round's in flight
// while the current one is decoded; the tokens are bucketed by tag, and each
// token's C/32 lanes decode 32 channels each from the stage and write them with
// 16-byte stores.
template <int C>
__global__ void __launch_bounds__(kXThreads)
mixed_dequant_kernel(const uint8_t* stream, const uint8_t* tags2, int64_t T, int64_t chunk, const int64_t* off,
                     __nv_bfloat16* out)
{
    constexpr int LPT = C / 32, TPW = 32 / LPT, SUB = dsub_tokens<C>();
    constexpr uint32_t kStage = SUB * 2 * C + 32;
    extern __shared__ __align__(128) unsigned char smem_raw[];    // two record stages
    unsigned char* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    __shared__ __align__(8) uint64_t full[2];
    __shared__ int64_t first_s[2];
    __shared__ int32_t roff[SUB];
    __shared__ uint8_t tg_s[SUB], order[SUB];
    __shared__ int cnt[4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t o = blockIdx.y;
    const int64_t t_lo = (int64_t)blockIdx.x * chunk, t_hi = min(T, t_lo + chunk);
    const int64_t nsub = (t_hi - t_lo + SUB - 1) / SUB;
    const uint8_t* sl = stream + o * T * 2 * C;                    // 16-byte aligned: T * 2C is a multiple of 16
    const int64_t* of = off + o * (T + 1);
    const int64_t tb = (T + 3) / 4;
    auto issue = [&](int64_t k) {                                  // one thread
        const int64_t sr = t_lo + k * SUB;
        const int64_t first = of[sr], last = of[min(t_hi, sr + SUB)];
        first_s[k & 1] = first;
        const uintptr_t a = (uintptr_t)(sl + first) & ~(uintptr_t)15;
        const uintptr_t b = ((uintptr_t)(sl + last) + 15) & ~(uintptr_t)15;   // within the slice's region
        mbar_expect_tx(&full[k & 1], (uint32_t)(b - a));
        bulk_g2s(smem + (k & 1) * kStage, reinterpret_cast<const void*>(a), (uint32_t)(b - a), &full[k & 1]);
    };
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init_fence();
        for (int64_t k = 0; k < 2 && k < nsub; ++k) issue(k);
    }
    __syncthreads();
    int64_t k = 0;
    bool ok = true;
    for (; k < nsub; ++k) {
        const int64_t sr = t_lo + k * SUB;
        const int n = (int)min((int64_t)SUB, t_hi - sr);
        if (tid < 4) cnt[tid] = 0;
        const int64_t first = first_s[k & 1];
        int g = -1;
        if (tid < n) {
            const int64_t t = sr + tid;
            g = (tags2[o * tb + t / 4] >> (2 * (t % 4))) & 3;
            tg_s[tid] = (uint8_t)g;
            roff[tid] = (int32_t)(of[t] - first);
        }
        __syncthreads();                                           // cnt zero before the bucketing
        bucket_by_tag(g, cnt, order);
        ok = __syncthreads_and(mbar_wait(&full[k & 1], (uint32_t)(k >> 1) & 1u));   // a timeout is recorded
        if (!ok) break;
        const unsigned char* rs = smem + (k & 1) * kStage + ((uintptr_t)(sl + first) & 15u);
        for (int e0 = warp * TPW; e0 < n; e0 += kXWarps * TPW) {
            const int e = e0 + lane / LPT, q = lane % LPT;
            if (e >= n) continue;
            const int tk = order[e], gt = tg_s[tk];
            const unsigned char* rec = rs + roff[tk];
            uint4 r[4];
            if (gt == 3) {
                uint32_t w[16];
                get_words(rec + q * 64, w, 16);
#pragma unroll
                for (int j = 0; j < 4; ++j) r[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
            } else {
                const int bits = gt == 0 ? 2 : (gt == 1 ? 4 : 8);
                const int pb = C * bits / 8;
                Meta m;
                m.s = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(rec + pb));
                m.z = gt == 2 ? __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(rec + pb + 2)) : 0.0f;
                const int offb = gt == 2 ? 0 : (1 << (bits - 1));  // offset binary of the symmetric codes
                uint32_t w[8];
                get_words(rec + q * (bits * 4), w, bits);          // bits * 4 bytes = bits words of 4 bytes
                u64 cph, sph;
                bool fast;
                dq_consts(m.s, m.z, offb, cph, sph, fast);
                u64 cp[4] = {cph, cph, cph, cph}, sp[4] = {sph, sph, sph, sph};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t u[8];
                    if (gt == 2) unpack_biased8<8>(make_uint2(w[2 * j], w[2 * j + 1]), u);
                    else if (gt == 1) unpack_biased8<4>(flip_signs<4>(w[j]), u);
                    else unpack_biased8<2>(flip_signs<2>((uint16_t)(w[j / 2] >> (16 * (j & 1)))), u);
                    TileAcc ta;
                    uint32_t mxb = 0;
                    if (fast) {
                        r[j] = dq8<false>(u, cp, sp, make_uint4(0, 0, 0, 0), ta, mxb);
                    } else {
                        float zs[8], ss[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) { zs[i] = m.z; ss[i] = m.s; }
                        r[j] = dq8_slow<false>(u, offb, zs, ss, make_uint4(0, 0, 0, 0), ta, mxb);
                    }
                }
            }
            uint4* dst = reinterpret_cast<uint4*>(out + ((uint64_t)o * T + sr + tk) * C + q * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j] = r[j];
        }
        __syncthreads();                                           // record stage read
        if (tid == 0 && k + 2 < nsub) {
            fence_proxy_async();
            issue(k + 2);
        }
    }
    // after a timed-out wait: wait (bounded) for the copies still in flight
    if (!ok && tid == 0)
        for (int64_t j = k; j < nsub && j < k + 2; ++j) mbar_wait(&full[j & 1], (uint32_t)(j >> 1) & 1u);
}

// Tokens per CTA: whole sub-rounds of `sub` tokens, at most kMaxChunks CTAs per slice.
int64_t mixed_chunk(int64_t T, int64_t sub)
{
    const int64_t subs = (T + sub - 1) / sub;
    return sub * ((subs + kMaxChunks - 1) / kMaxChunks);
}

template <int C>
cudaError_t mixed_quant_launch(const __nv_bfloat16* x, const uint8_t* tags, int64_t outer, int64_t T, int64_t* off,
                               uint8_t* tags2, uint8_t* sb, const MixedFormats& F, cudaStream_t st)
{
    const int smem = kQStage + 16 + 16;                           // + alignment slack
    cudaError_t e = ensure_kernel_attrs(reinterpret_cast<const void*>(mixed_quant_kernel<C>), smem);
    if (e != cudaSuccess) return e;
    const int64_t chunk = mixed_chunk(T, qsub_tokens<C>());
    const dim3 grid((unsigned)((T + chunk - 1) / chunk), (unsigned)outer);
    mixed_quant_kernel<C><<<grid, kXThreads, smem, st>>>(x, tags, T, chunk, off, tags2, sb, F);
    return cudaGetLastError();
}

template <int C>
cudaError_t mixed_dequant_launch(const uint8_t* sb, const uint8_t* tags2, int64_t outer, int64_t T, const int64_t* off,
                                 __nv_bfloat16* ob, cudaStream_t st)
{
    const int smem = 2 * (dsub_tokens<C>() * 2 * C + 32) + 128;     // + alignment slack
    cudaError_t e = ensure_kernel_attrs(reinterpret_cast<const void*>(mixed_dequant_kernel<C>), smem);
    if (e != cudaSuccess) return e;
    const int64_t chunk = mixed_chunk(T, dsub_tokens<C>());
    const dim3 grid((unsigned)((T + chunk - 1) / chunk), (unsigned)outer);
    mixed_dequant_kernel<C><<<grid, kXThreads, smem, st>>>(sb, tags2, T, chunk, off, ob);
    return cudaGetLastError();
}

}  // namespace

int64_t mixed_record_bytes(int tag, int64_t C) { return record_bytes(tag & 3, C); }

cudaError_t launch_mixed_quantize(const void* x, const uint8_t* tags, int64_t outer, int64_t T, int64_t C,
                                  void* stream_buf, int64_t* off, uint8_t* tags2, const QSpec& f2, const QSpec& f4,
                                  const QSpec& f8, cudaStream_t st)
{
    if (outer == 0 || T == 0) return cudaSuccess;
    const MixedFormats F = {f2, f4, f8};
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    uint8_t* sb = static_cast<uint8_t*>(stream_buf);
    switch (C) {
    case 64: return mixed_quant_launch<64>(xb, tags, outer, T, off, tags2, sb, F, st);
    case 128: return mixed_quant_launch<128>(xb, tags, outer, T, off, tags2, sb, F, st);
    default: return mixed_quant_launch<256>(xb, tags, outer, T, off, tags2, sb, F, st);
    }
}

cudaError_t launch_mixed_dequantize(const void* stream_buf, const int64_t* off, const uint8_t* tags2, int64_t outer,
                                    int64_t T, int64_t C, void* out, cudaStream_t st)
{
    if (outer == 0 || T == 0) return cudaSuccess;
    const uint8_t* sb = static_cast<const uint8_t*>(stream_buf);
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out);
    switch (C) {
    case 64: return mixed_dequant_launch<64>(sb, tags2, outer, T, off, ob, st);
    case 128: return mixed_dequant_launch<128>(sb, tags2, outer, T, off, ob, st);
    default: return mixed_dequant_launch<256>(sb, tags2, outer, T, off, ob, st);
    }
}

}  // namespace kvq
