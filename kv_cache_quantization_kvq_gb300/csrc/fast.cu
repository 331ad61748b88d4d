// fast.cu -- bf16 fast paths of quantize, dequantize and error statistics.
//
// Same method and results as quant.cu / dequant.cu ("KV Compression
// 公式到源码对照" §1.1-§1.3; "KV cache 压缩：把历史装得更小" group-wise form,
// KIVI axes and residual window), restructured so that each element costs a
// few issue slots (see kvq_fast.cuh):
//
//  groups along C ("per token", V):  a lane owns 64 consecutive channels of
//      one token (128 B of bf16, eight 16-B loads); a group is 64/G of those
//      (G < 64) or G/64 adjacent lanes (G > 64, one shuffle level).  Group
//      constants are computed once per lane and group.
//  groups along T ("per channel", K), g <= 128:  a warp owns a tile of
//      g tokens x (8*LC) channels; lane (lr, lc) holds RPT = g/LR rows of 8
//      channels in registers, the group min/max is reduced over lr with
//      shuffles, and each lane derives the constants of 8/LR channels and
//      shares them with shuffles.
//  groups along T longer than 128 tokens:  a stats pass folds per-tile
//      min/max into the workspace with integer atomics, then an apply pass
//      re-reads the tile (from L2 when the chunk fits) to write codes.
//  dequantize / error statistics along T use the same tiles (a group is
//      split into slices of LR*RPT tokens); along C the same lane items.
#include <algorithm>

#include "kvq_elem.cuh"

namespace kvq {

namespace {

using namespace elem;

// ======================================================================
// quantize, groups along C: lane item = 64 channels of one token
// ======================================================================
template <int BITS, bool ASYM, int G>
__global__ void __launch_bounds__(kThr)
qc_kernel(const QArgs a, int lcpr)
{
    constexpr int GPL = G >= 64 ? 1 : 64 / G;    // groups per lane
    constexpr int LPG = G >= 64 ? G / 64 : 1;    // lanes per group
    constexpr int WPG = G >= 64 ? 8 : G / 8;     // 8-element words per group in a lane
    const QSpec& q = a.q;
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const int lo_c = q.qmin + off, hi_c = q.qmax + off;
    const uint32_t T = (uint32_t)q.T, Tq = (uint32_t)q.Tq;
    const uint64_t nitems = ((uint64_t)q.outer * q.T) << lcpr;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
    __nv_bfloat16* resid = static_cast<__nv_bfloat16*>(a.resid);
    uint8_t* codes = static_cast<uint8_t*>(a.codes);
    const int gpr = (int)(q.C / G);

    for (uint64_t base = (uint64_t)blockIdx.x * kThr; base < nitems; base += (uint64_t)gridDim.x * kThr) {
        const uint64_t i = base + threadIdx.x;
        const bool valid = i < nitems;
        const uint32_t row = (uint32_t)(i >> lcpr);
        const uint32_t ch = (uint32_t)(i & ((1u << lcpr) - 1u));
        const uint32_t o = valid ? row / T : 0u;
        const uint32_t t = valid ? row - o * T : 0u;
        uint4 w[8];
        const uint4* src = reinterpret_cast<const uint4*>(x + ((uint64_t)row * q.C + (uint64_t)ch * 64));
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = valid ? __ldcs(src + k) : make_uint4(0, 0, 0, 0);
        const bool is_res = valid && t >= Tq;
        // group statistics (every lane of the warp takes part in the shuffles)
        float gmn[GPL], gmx[GPL];
#pragma unroll
        for (int gg = 0; gg < GPL; ++gg) {
            uint32_t mn = kBfPosInf2, mx = ASYM ? kBfNegInf2 : 0u;
#pragma unroll
            for (int k = 0; k < WPG; ++k) {
                if (ASYM) fold_minmax(w[gg * WPG + k], mn, mx);
                else fold_absmax(w[gg * WPG + k], mx);
            }
            gmn[gg] = fminf(lo_f(mn), hi_f(mn));
            gmx[gg] = fmaxf(lo_f(mx), hi_f(mx));
            if (LPG > 1) {
#pragma unroll
                for (int s = 1; s < LPG; s <<= 1) {
                    gmn[gg] = fminf(gmn[gg], __shfl_xor_sync(0xFFFFFFFFu, gmn[gg], s));
                    gmx[gg] = fmaxf(gmx[gg], __shfl_xor_sync(0xFFFFFFFFu, gmx[gg], s));
                }
            }
        }
        if (!valid) continue;
        if (is_res) {
            uint4* dst = reinterpret_cast<uint4*>(resid + (((uint64_t)o * q.R + (t - Tq)) * q.C + (uint64_t)ch * 64));
#pragma unroll
            for (int k = 0; k < 8; ++k) dst[k] = w[k];
            continue;
        }
        const uint64_t qrow = (uint64_t)o * Tq + t;
        uint8_t* cdst = codes + qrow * (uint64_t)(q.C * BITS / 8) + (uint64_t)ch * 8 * BITS;
        typename CodeWord<BITS>::T cw[8];
#pragma unroll
        for (int gg = 0; gg < GPL; ++gg) {
            const GroupC gc = make_group<ASYM>(gmn[gg], gmx[gg], q, off);
            const int64_t mi = (int64_t)qrow * gpr + (G >= 64 ? (int64_t)ch / LPG : (int64_t)ch * GPL + gg);
            if (LPG == 1 || (ch % LPG) == 0) {
                Meta m;
                m.s = gc.s;
                m.z = gc.zp;
                write_meta(a, mi, m);
            }
            if (gc.fast) {
                QuotK kq[4];
                kq[0].ns = pk(-gc.s, -gc.s);
                kq[0].inv = pk(gc.inv, gc.inv);
                kq[1] = kq[2] = kq[3] = kq[0];
                int32_t zo[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) zo[j] = gc.zoff;
#pragma unroll
                for (int k = 0; k < WPG; ++k) {
                    uint32_t c[8];
                    codes8_fast<ASYM>(w[gg * WPG + k], kq, zo, lo_c, hi_c, c);
                    cw[gg * WPG + k] = finish_word<BITS>(c, q.is_signed);
                }
            } else {
                float s8[8], z8[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) { s8[j] = gc.s; z8[j] = gc.zp; }
#pragma unroll
                for (int k = 0; k < WPG; ++k) {
                    uint32_t c[8];
                    codes8_slow<ASYM>(w[gg * WPG + k], s8, z8, q, off, c);
                    cw[gg * WPG + k] = finish_word<BITS>(c, q.is_signed);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) store_codes<BITS>(cdst + k * BITS, cw[k]);
    }
}

// ======================================================================
// quantize, groups along T with g = LR*RPT <= 128: warp tile
// ======================================================================
template <int BITS, bool ASYM, int LR, int RPT>
__global__ void __launch_bounds__(kThr)
qt_kernel(const QArgs a, uint32_t ncb)
{
    constexpr int LC = 32 / LR;           // lane columns, 8 channels each
    constexpr int CPL = 8 / LR;           // channels whose constants a lane derives
    const QSpec& q = a.q;
    const int lane = threadIdx.x & 31;
    const int lr = lane / LC, lc = lane % LC;
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const int lo_c = q.qmin + off, hi_c = q.qmax + off;
    const uint32_t ng = (uint32_t)q.ngroups;
    const uint32_t nres = (uint32_t)((q.R + LR * RPT - 1) / (LR * RPT));
    const uint32_t tiles_per_o = (ng + nres) * ncb;
    const uint64_t ntiles = (uint64_t)q.outer * tiles_per_o;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
    uint8_t* codes = static_cast<uint8_t*>(a.codes);
    const uint64_t code_row_B = (uint64_t)q.C * BITS / 8;
    const uint64_t wstride = (uint64_t)gridDim.x * (kThr / 32);

    for (uint64_t tile = (uint64_t)blockIdx.x * (kThr / 32) + (threadIdx.x >> 5); tile < ntiles; tile += wstride) {
        const uint32_t o = (uint32_t)(tile / tiles_per_o);
        const uint32_t rem = (uint32_t)(tile - (uint64_t)o * tiles_per_o);
        const uint32_t gi = rem / ncb, cb = rem - gi * ncb;
        const uint64_t c0 = (uint64_t)cb * (8 * LC) + (uint64_t)lc * 8;
        if (gi >= ng) {
            // residual window rows
            __nv_bfloat16* resid = static_cast<__nv_bfloat16*>(a.resid);
            const int64_t r0 = (int64_t)(gi - ng) * (LR * RPT) + lr * RPT;
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                const int64_t r = r0 + j;
                if (r < q.R) {
                    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(x + (((uint64_t)o * q.T + q.Tq + r) * q.C + c0)));
                    *reinterpret_cast<uint4*>(resid + (((uint64_t)o * q.R + r) * q.C + c0)) = v;
                }
            }
            continue;
        }
        const int64_t t0 = (int64_t)gi * q.g;
        const int64_t glen = min(q.g, q.Tq - t0);
        uint4 w[RPT];
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int64_t r = lr * RPT + j;
            w[j] = r < glen ? __ldcs(reinterpret_cast<const uint4*>(x + (((uint64_t)o * q.T + t0 + r) * q.C + c0)))
                            : make_uint4(0, 0, 0, 0);
        }
        // per-channel statistics of the lane's rows, then across lane rows
        uint32_t mn[4], mx[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) { mn[p] = kBfPosInf2; mx[p] = ASYM ? kBfNegInf2 : 0u; }
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            if (lr * RPT + j < glen) {
                const uint32_t ws[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    if (ASYM) { mn[p] = bmin2(mn[p], ws[p]); mx[p] = bmax2(mx[p], ws[p]); }
                    else mx[p] = bmax2(mx[p], babs2(ws[p]));
                }
            }
        }
#pragma unroll
        for (int s = LC; s < 32; s <<= 1) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                if (ASYM) mn[p] = bmin2(mn[p], __shfl_xor_sync(0xFFFFFFFFu, mn[p], s));
                mx[p] = bmax2(mx[p], __shfl_xor_sync(0xFFFFFFFFu, mx[p], s));
            }
        }
        // this lane derives the constants of channels [lr*CPL, lr*CPL + CPL)
        float cs[CPL], ci[CPL];
        int32_t cz[CPL];
        bool cfast = true;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            const int ch = lr * CPL + k;            // 0..7
            const uint32_t wm = mn[ch >> 1], wx = mx[ch >> 1];
            const float fmn = (ch & 1) ? hi_f(wm) : lo_f(wm);
            const float fmx = (ch & 1) ? hi_f(wx) : lo_f(wx);
            const GroupC gc = make_group<ASYM>(fmn, fmx, q, off);
            Meta m;
            m.s = gc.s;
            m.z = gc.zp;
            write_meta(a, ((int64_t)o * ng + gi) * q.C + (int64_t)(c0 + ch), m);
            cs[k] = gc.s;
            ci[k] = gc.inv;
            cz[k] = gc.zoff;
            cfast = cfast && gc.fast;
        }
        const bool all_fast = __all_sync(0xFFFFFFFFu, cfast);
        // gather the eight channels' constants
        float s8[8], i8[8], z8f[8];
        int32_t zo[8];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            const int src = (ch / CPL) * LC + lc;
            s8[ch] = __shfl_sync(0xFFFFFFFFu, cs[ch % CPL], src);
            i8[ch] = __shfl_sync(0xFFFFFFFFu, ci[ch % CPL], src);
            zo[ch] = __shfl_sync(0xFFFFFFFFu, cz[ch % CPL], src);
            z8f[ch] = (float)(zo[ch] - off + (int32_t)kMagicBits);
        }
        uint8_t* cdst = codes + ((uint64_t)o * q.Tq + t0 + lr * RPT) * code_row_B + (c0 / 8) * BITS;
        if (all_fast) {
            QuotK kq[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                kq[p].ns = pk(-s8[2 * p], -s8[2 * p + 1]);
                kq[p].inv = pk(i8[2 * p], i8[2 * p + 1]);
            }
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                if (lr * RPT + j < glen) {
                    uint32_t c[8];
                    codes8_fast<ASYM>(w[j], kq, zo, lo_c, hi_c, c);
                    store_codes<BITS>(cdst + j * code_row_B, finish_word<BITS>(c, q.is_signed));
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                if (lr * RPT + j < glen) {
                    uint32_t c[8];
                    codes8_slow<ASYM>(w[j], s8, z8f, q, off, c);
                    store_codes<BITS>(cdst + j * code_row_B, finish_word<BITS>(c, q.is_signed));
                }
            }
        }
    }
}

// ======================================================================
// quantize, groups along T longer than 128 tokens: stats pass, apply pass
// ======================================================================
// tile = (outer, group, 64-channel block, slice of kLongRows tokens);
// lane (lr, lc), lr in 0..3, lc in 0..7: rows lr, lr+4, ... of the slice.
constexpr int kLongRows = 256;

template <bool ASYM>
__global__ void __launch_bounds__(kThr)
ql_stats_kernel(const QArgs a, uint32_t ncb, uint32_t nsl, uint32_t o_base, uint32_t o_count)
{
    const QSpec& q = a.q;
    const int lane = threadIdx.x & 31, lr = lane >> 3, lc = lane & 7;
    const uint32_t tiles_per_o = (uint32_t)q.ngroups * nsl * ncb;
    const uint64_t ntiles = (uint64_t)o_count * tiles_per_o;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
    uint32_t* kmax = static_cast<uint32_t*>(a.ws);
    const int64_t nkeys = q.outer * q.ngroups * q.C;
    for (uint64_t tile = (uint64_t)blockIdx.x * (kThr / 32) + (threadIdx.x >> 5); tile < ntiles;
         tile += (uint64_t)gridDim.x * (kThr / 32)) {
        const uint32_t o = o_base + (uint32_t)(tile / tiles_per_o);
        uint32_t rem = (uint32_t)(tile % tiles_per_o);
        const uint32_t cb = rem % ncb;
        rem /= ncb;
        const uint32_t sl = rem % nsl, gi = rem / nsl;
        const uint64_t c0 = (uint64_t)cb * 64 + (uint64_t)lc * 8;
        const int64_t gend = min((int64_t)(gi + 1) * q.g, q.Tq);
        const int64_t tb = (int64_t)gi * q.g + (int64_t)sl * kLongRows;
        const int64_t te = min(tb + kLongRows, gend);
        uint32_t mn[4], mx[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) { mn[p] = kBfPosInf2; mx[p] = ASYM ? kBfNegInf2 : 0u; }
        const __nv_bfloat16* base = x + ((uint64_t)o * q.T) * q.C + c0;
        for (int64_t t = tb + lr; t < te; t += 4 * 8) {
            uint4 w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t tt = t + 4 * u;
                w[u] = tt < te ? *reinterpret_cast<const uint4*>(base + (uint64_t)tt * q.C) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (t + 4 * u < te) {
                    const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        if (ASYM) { mn[p] = bmin2(mn[p], ws[p]); mx[p] = bmax2(mx[p], ws[p]); }
                        else mx[p] = bmax2(mx[p], babs2(ws[p]));
                    }
                }
            }
        }
#pragma unroll
        for (int s = 8; s < 32; s <<= 1) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                if (ASYM) mn[p] = bmin2(mn[p], __shfl_xor_sync(0xFFFFFFFFu, mn[p], s));
                mx[p] = bmax2(mx[p], __shfl_xor_sync(0xFFFFFFFFu, mx[p], s));
            }
        }
        if (te <= tb) continue;
        // lane row lr folds channels 2*lr and 2*lr+1 into the workspace
        const int p = lr;
        const int64_t k0 = ((int64_t)o * q.ngroups + gi) * q.C + (int64_t)(c0 + 2 * p);
        if (ASYM) {
            atomicMax(kmax + k0, float_key(lo_f(mx[p])));
            atomicMax(kmax + k0 + 1, float_key(hi_f(mx[p])));
            atomicMin(kmax + nkeys + k0, float_key(lo_f(mn[p])));
            atomicMin(kmax + nkeys + k0 + 1, float_key(hi_f(mn[p])));
        } else {
            atomicMax(kmax + k0, __float_as_uint(lo_f(mx[p])));
            atomicMax(kmax + k0 + 1, __float_as_uint(hi_f(mx[p])));
        }
    }
}

template <int BITS, bool ASYM>
__global__ void __launch_bounds__(kThr)
ql_apply_kernel(const QArgs a, uint32_t ncb, uint32_t nsl, uint32_t o_base, uint32_t o_count)
{
    const QSpec& q = a.q;
    const int lane = threadIdx.x & 31, lr = lane >> 3, lc = lane & 7;
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const int lo_c = q.qmin + off, hi_c = q.qmax + off;
    const uint32_t tiles_per_o = (uint32_t)q.ngroups * nsl * ncb;
    const uint64_t ntiles = (uint64_t)o_count * tiles_per_o;
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
    const uint32_t* kmax = static_cast<const uint32_t*>(a.ws);
    const int64_t nkeys = q.outer * q.ngroups * q.C;
    uint8_t* codes = static_cast<uint8_t*>(a.codes);
    const uint64_t code_row_B = (uint64_t)q.C * BITS / 8;
    for (uint64_t tile = (uint64_t)blockIdx.x * (kThr / 32) + (threadIdx.x >> 5); tile < ntiles;
         tile += (uint64_t)gridDim.x * (kThr / 32)) {
        const uint32_t o = o_base + (uint32_t)(tile / tiles_per_o);
        uint32_t rem = (uint32_t)(tile % tiles_per_o);
        const uint32_t cb = rem % ncb;
        rem /= ncb;
        const uint32_t sl = rem % nsl, gi = rem / nsl;
        const uint64_t c0 = (uint64_t)cb * 64 + (uint64_t)lc * 8;
        const int64_t gend = min((int64_t)(gi + 1) * q.g, q.Tq);
        const int64_t tb = (int64_t)gi * q.g + (int64_t)sl * kLongRows;
        const int64_t te = min(tb + kLongRows, gend);
        // constants of channels 2*lr, 2*lr+1, shared across lane rows
        const int64_t k0 = ((int64_t)o * q.ngroups + gi) * q.C + (int64_t)(c0 + 2 * lr);
        float cs[2], ci[2];
        int32_t cz[2];
        bool cfast = true;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float fmx = ASYM ? key_float(kmax[k0 + k]) : __uint_as_float(kmax[k0 + k]);
            const float fmn = ASYM ? key_float(kmax[nkeys + k0 + k]) : 0.0f;
            const GroupC gc = make_group<ASYM>(fmn, fmx, q, off);
            if (sl == 0) {
                Meta m;
                m.s = gc.s;
                m.z = gc.zp;
                write_meta(a, k0 + k, m);
            }
            cs[k] = gc.s;
            ci[k] = gc.inv;
            cz[k] = gc.zoff;
            cfast = cfast && gc.fast;
        }
        const bool all_fast = __all_sync(0xFFFFFFFFu, cfast);
        float s8[8], i8[8], z8f[8];
        int32_t zo[8];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
            const int src = (ch >> 1) * 8 + lc;
            s8[ch] = __shfl_sync(0xFFFFFFFFu, cs[ch & 1], src);
            i8[ch] = __shfl_sync(0xFFFFFFFFu, ci[ch & 1], src);
            zo[ch] = __shfl_sync(0xFFFFFFFFu, cz[ch & 1], src);
            z8f[ch] = (float)(zo[ch] - off + (int32_t)kMagicBits);
        }
        QuotK kq[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            kq[p].ns = pk(-s8[2 * p], -s8[2 * p + 1]);
            kq[p].inv = pk(i8[2 * p], i8[2 * p + 1]);
        }
        const __nv_bfloat16* base = x + ((uint64_t)o * q.T) * q.C + c0;
        uint8_t* cbase = codes + ((uint64_t)o * q.Tq) * code_row_B + (c0 / 8) * BITS;
        for (int64_t t = tb + lr; t < te; t += 4 * 8) {
            uint4 w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t tt = t + 4 * u;
                w[u] = tt < te ? __ldcs(reinterpret_cast<const uint4*>(base + (uint64_t)tt * q.C)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t tt = t + 4 * u;
                if (tt < te) {
                    uint32_t c[8];
                    if (all_fast) codes8_fast<ASYM>(w[u], kq, zo, lo_c, hi_c, c);
                    else codes8_slow<ASYM>(w[u], s8, z8f, q, off, c);
                    store_codes<BITS>(cbase + (uint64_t)tt * code_row_B, finish_word<BITS>(c, q.is_signed));
                }
            }
        }
    }
}

// ======================================================================
// dequantize / error statistics
// ======================================================================

// ---------------- groups along C
template <int BITS, bool ASYM, int G, bool STATS>
__global__ void __launch_bounds__(kThr)
dc_kernel(const QArgs a, int lcpr, Partial* partials)
{
    constexpr int GPL = G >= 64 ? 1 : 64 / G;
    constexpr int LPG = G >= 64 ? G / 64 : 1;
    constexpr int WPG = G >= 64 ? 8 : G / 8;
    constexpr int CW = 8 * BITS / 16;           // uint4 words of codes per lane item
    const QSpec& q = a.q;
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const uint32_t T = (uint32_t)q.T, Tq = (uint32_t)q.Tq;
    const uint64_t nitems = ((uint64_t)q.outer * q.T) << lcpr;
    const uint8_t* codes = static_cast<const uint8_t*>(a.codes);
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    const __nv_bfloat16* resid = static_cast<const __nv_bfloat16*>(a.resid);
    const int gpr = (int)(q.C / G);
    Acc2 A;
    for (uint64_t i = (uint64_t)blockIdx.x * kThr + threadIdx.x; i < nitems; i += (uint64_t)gridDim.x * kThr) {
        const uint32_t row = (uint32_t)(i >> lcpr);
        const uint32_t ch = (uint32_t)(i & ((1u << lcpr) - 1u));
        const uint32_t o = row / T, t = row - o * T;
        if (t >= Tq) {
            if (!STATS) {
                const uint4* src = reinterpret_cast<const uint4*>(resid + (((uint64_t)o * q.R + (t - Tq)) * q.C + (uint64_t)ch * 64));
                uint4* dst = reinterpret_cast<uint4*>(out + ((uint64_t)row * q.C + (uint64_t)ch * 64));
#pragma unroll
                for (int k = 0; k < 8; ++k) dst[k] = __ldcs(src + k);
            }
            continue;
        }
        const uint64_t qrow = (uint64_t)o * Tq + t;
        // codes of 64 channels: BITS*8 bytes
        typename CodeWord<BITS>::T cw[8];
        {
            const uint4* cs = reinterpret_cast<const uint4*>(codes + qrow * (uint64_t)(q.C * BITS / 8) + (uint64_t)ch * 8 * BITS);
            uint4 raw[CW];
#pragma unroll
            for (int k = 0; k < CW; ++k) raw[k] = __ldcs(cs + k);
            const typename CodeWord<BITS>::T* pw = reinterpret_cast<const typename CodeWord<BITS>::T*>(raw);
#pragma unroll
            for (int k = 0; k < 8; ++k) cw[k] = pw[k];
        }
        uint4 xw[8];
        if (STATS) {
            const uint4* xs = reinterpret_cast<const uint4*>(x + ((uint64_t)row * q.C + (uint64_t)ch * 64));
#pragma unroll
            for (int k = 0; k < 8; ++k) xw[k] = __ldcs(xs + k);
        }
        uint4 ow[8];
        TileAcc ta;
#pragma unroll
        for (int gg = 0; gg < GPL; ++gg) {
            const int64_t mi = (int64_t)qrow * gpr + (G >= 64 ? (int64_t)ch / LPG : (int64_t)ch * GPL + gg);
            const float s = load_meta(a.scale, q.scale_dt, mi);
            const float zp = ASYM ? load_meta(a.zero, q.zero_dt, mi) : 0.0f;
            u64 cph, sph;
            bool fast;
            dq_consts(s, zp, off, cph, sph, fast);
            const u64 cp[4] = {cph, cph, cph, cph}, sp[4] = {sph, sph, sph, sph};
#pragma unroll
            for (int k = 0; k < WPG; ++k) {
                const int wi = gg * WPG + k;
                uint32_t u[8];
                unpack_biased8<BITS>(q.is_signed ? flip_signs<BITS>(cw[wi]) : cw[wi], u);
                if (fast) {
                    ow[wi] = dq8<STATS>(u, cp, sp, xw[wi], ta, A.mxb);
                } else {
                    float zs[8], ss[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) { zs[j] = zp; ss[j] = s; }
                    ow[wi] = dq8_slow<STATS>(u, off, zs, ss, xw[wi], ta, A.mxb);
                }
            }
        }
        if (STATS) {
            A.fold(ta);
        } else {
            uint4* dst = reinterpret_cast<uint4*>(out + ((uint64_t)row * q.C + (uint64_t)ch * 64));
#pragma unroll
            for (int k = 0; k < 8; ++k) dst[k] = ow[k];
        }
    }
    if (STATS) block_reduce_partial(A, partials);
}

// ---------------- groups along T: tile = (outer, group, slice of LR*RPT tokens, 8*LC channels)
template <int BITS, bool ASYM, int LR, int RPT, bool STATS>
__global__ void __launch_bounds__(kThr)
dt_kernel(const QArgs a, uint32_t ncb, uint32_t nsl, Partial* partials)
{
    constexpr int LC = 32 / LR;
    constexpr int TR = LR * RPT;
    const QSpec& q = a.q;
    const int lane = threadIdx.x & 31;
    const int lr = lane / LC, lc = lane % LC;
    const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
    const uint32_t ng = (uint32_t)q.ngroups;
    const uint32_t nres = STATS ? 0u : (uint32_t)((q.R + TR - 1) / TR);
    const uint32_t tiles_per_o = (ng * nsl + nres) * ncb;
    const uint64_t ntiles = (uint64_t)q.outer * tiles_per_o;
    const uint8_t* codes = static_cast<const uint8_t*>(a.codes);
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    const __nv_bfloat16* resid = static_cast<const __nv_bfloat16*>(a.resid);
    const uint64_t code_row_B = (uint64_t)q.C * BITS / 8;
    using W = typename CodeWord<BITS>::T;
    Acc2 A;
    for (uint64_t tile = (uint64_t)blockIdx.x * (kThr / 32) + (threadIdx.x >> 5); tile < ntiles;
         tile += (uint64_t)gridDim.x * (kThr / 32)) {
        const uint32_t o = (uint32_t)(tile / tiles_per_o);
        const uint32_t rem = (uint32_t)(tile - (uint64_t)o * tiles_per_o);
        const uint32_t gs = rem / ncb, cb = rem - gs * ncb;
        const uint64_t c0 = (uint64_t)cb * (8 * LC) + (uint64_t)lc * 8;
        if (gs >= ng * nsl) {
            const int64_t r0 = (int64_t)(gs - ng * nsl) * TR + lr * RPT;
#pragma unroll
            for (int j = 0; j < RPT; ++j) {
                const int64_t r = r0 + j;
                if (r < q.R)
                    *reinterpret_cast<uint4*>(out + (((uint64_t)o * q.T + q.Tq + r) * q.C + c0)) =
                        __ldcs(reinterpret_cast<const uint4*>(resid + (((uint64_t)o * q.R + r) * q.C + c0)));
            }
            continue;
        }
        const uint32_t gi = gs / nsl, sl = gs - gi * nsl;
        const int64_t gend = min((int64_t)(gi + 1) * q.g, q.Tq);
        const int64_t tb = (int64_t)gi * q.g + (int64_t)sl * TR + lr * RPT;
        // constants of the lane's 8 channels
        const int64_t mi = ((int64_t)o * ng + gi) * q.C + (int64_t)c0;
        u64 cp[4], sp[4];
        float sf[8], zsf[8];
        bool fast = true;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const float s0 = load_meta(a.scale, q.scale_dt, mi + 2 * p), s1 = load_meta(a.scale, q.scale_dt, mi + 2 * p + 1);
            const float z0 = ASYM ? load_meta(a.zero, q.zero_dt, mi + 2 * p) : 0.0f;
            const float z1 = ASYM ? load_meta(a.zero, q.zero_dt, mi + 2 * p + 1) : 0.0f;
            fast = fast && fabsf(z0) < 0x1p21f && fabsf(z1) < 0x1p21f;
            cp[p] = pk(__fadd_rn(8388608.0f + (float)off, z0), __fadd_rn(8388608.0f + (float)off, z1));
            sp[p] = pk(s0, s1);
            sf[2 * p] = s0;
            sf[2 * p + 1] = s1;
            zsf[2 * p] = z0;
            zsf[2 * p + 1] = z1;
        }
        W cw[RPT];
        uint4 xw[RPT];
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int64_t t = tb + j;
            if (t < gend) {
                cw[j] = __ldcs(reinterpret_cast<const W*>(codes + ((uint64_t)o * q.Tq + t) * code_row_B + (c0 / 8) * BITS));
                if (STATS) xw[j] = __ldcs(reinterpret_cast<const uint4*>(x + (((uint64_t)o * q.T + t) * q.C + c0)));
            }
        }
        TileAcc ta;
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            const int64_t t = tb + j;
            if (t >= gend) continue;
            uint32_t u[8];
            unpack_biased8<BITS>(q.is_signed ? flip_signs<BITS>(cw[j]) : cw[j], u);
            const uint4 ow = fast ? dq8<STATS>(u, cp, sp, xw[j], ta, A.mxb)
                                  : dq8_slow<STATS>(u, off, zsf, sf, xw[j], ta, A.mxb);
            if (!STATS) *reinterpret_cast<uint4*>(out + (((uint64_t)o * q.T + t) * q.C + c0)) = ow;
        }
        if (STATS) A.fold(ta);
    }
    if (STATS) block_reduce_partial(A, partials);
}

// ======================================================================
// dispatch
// ======================================================================

int log2_exact(int64_t v) {
    int l = 0;
    while ((int64_t(1) << l) < v) ++l;
    return (int64_t(1) << l) == v ? l : -1;
}

bool c_ok(const QSpec& q) {
    if (q.x_dt != KVQ_BF16 || !q.aligned || q.C % 64 != 0 || log2_exact(q.C / 64) < 0) return false;
    if (q.outer * q.T >= (int64_t(1) << 31)) return false;
    const int64_t g = q.g;
    return q.C % g == 0 && (g == 8 || g == 16 || g == 32 || g == 64 || g == 128 || g == 256);
}

bool t_ok(const QSpec& q) {
    return q.x_dt == KVQ_BF16 && q.aligned && q.C % 64 == 0;
}

// tile shape for groups along T: g <= 128 quantized in one tile
bool t_tile_g(int64_t g) { return g == 8 || g == 16 || g == 32 || g == 64 || g == 128; }

unsigned grid_cap(int sms, int64_t work_units, int per_block) {
    const int64_t want = (work_units + per_block - 1) / per_block;
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * 8));
}

template <int BITS, bool ASYM>
bool quantize_typed(const QArgs& a, cudaStream_t st)
{
    const QSpec& q = a.q;
    const int sms = sm_count();
    if (q.axis == KVQ_GROUP_ALONG_C) {
        if (!c_ok(q)) return false;
        const int lcpr = log2_exact(q.C / 64);
        const unsigned grid = grid_cap(sms, (q.outer * q.T) << lcpr, kThr);
        switch (q.g) {
        case 8: qc_kernel<BITS, ASYM, 8><<<grid, kThr, 0, st>>>(a, lcpr); break;
        case 16: qc_kernel<BITS, ASYM, 16><<<grid, kThr, 0, st>>>(a, lcpr); break;
        case 32: qc_kernel<BITS, ASYM, 32><<<grid, kThr, 0, st>>>(a, lcpr); break;
        case 64: qc_kernel<BITS, ASYM, 64><<<grid, kThr, 0, st>>>(a, lcpr); break;
        case 128: qc_kernel<BITS, ASYM, 128><<<grid, kThr, 0, st>>>(a, lcpr); break;
        default: qc_kernel<BITS, ASYM, 256><<<grid, kThr, 0, st>>>(a, lcpr); break;
        }
        return true;
    }
    if (!t_ok(q)) return false;
    if (t_tile_g(q.g) || q.Tq <= 0) {
        if (!t_tile_g(q.g)) return false;
        const uint32_t ncb = (uint32_t)(q.C / (q.g == 128 ? 32 : 64));
        const int64_t TR = q.g;
        const int64_t nres = (q.R + TR - 1) / TR;
        const int64_t ntiles = q.outer * (q.ngroups + nres) * ncb;
        const unsigned grid = grid_cap(sms, ntiles, kThr / 32);
        switch (q.g) {
        case 8: qt_kernel<BITS, ASYM, 4, 2><<<grid, kThr, 0, st>>>(a, ncb); break;
        case 16: qt_kernel<BITS, ASYM, 4, 4><<<grid, kThr, 0, st>>>(a, ncb); break;
        case 32: qt_kernel<BITS, ASYM, 4, 8><<<grid, kThr, 0, st>>>(a, ncb); break;
        case 64: qt_kernel<BITS, ASYM, 4, 16><<<grid, kThr, 0, st>>>(a, ncb); break;
        default: qt_kernel<BITS, ASYM, 8, 16><<<grid, kThr, 0, st>>>(a, ncb); break;
        }
        return true;
    }
    return false;   // long groups: see quantize_long
}

}  // namespace

// ---- entry points used by quant.cu / dequant.cu

bool fast_quantize_supported(const QSpec& q)
{
    if (q.x_dt != KVQ_BF16 || !q.aligned) return false;
    if (q.axis == KVQ_GROUP_ALONG_C) return c_ok(q);
    return t_ok(q);
}

bool fast_quantize_copies_residual(const QSpec& q)
{
    return q.axis == KVQ_GROUP_ALONG_C || t_tile_g(q.g) || staged_quantize_supported(q);
}

size_t fast_quantize_workspace(const QSpec& q)
{
    if (q.axis == KVQ_GROUP_ALONG_T && t_ok(q) && !t_tile_g(q.g) && q.Tq > 0)
        return (size_t)(q.outer * q.ngroups * q.C) * 4 * (q.mode == KVQ_ASYM ? 2 : 1);
    return 0;
}

cudaError_t fast_quantize(const QArgs& a, cudaStream_t st)
{
    const QSpec& q = a.q;
    if (staged_quantize(a, st)) return cudaGetLastError();
    const bool asym = q.mode == KVQ_ASYM;
    if (q.axis == KVQ_GROUP_ALONG_C || t_tile_g(q.g)) {
        bool ok;
        switch (q.bits) {
        case 8: ok = asym ? quantize_typed<8, true>(a, st) : quantize_typed<8, false>(a, st); break;
        case 4: ok = asym ? quantize_typed<4, true>(a, st) : quantize_typed<4, false>(a, st); break;
        default: ok = asym ? quantize_typed<2, true>(a, st) : quantize_typed<2, false>(a, st); break;
        }
        return ok ? cudaGetLastError() : cudaErrorInvalidValue;
    }
    // long groups along T: one cluster per group and channel block, else a
    // stats pass and an apply pass through the workspace
    if (cluster_quantize(a, st)) return cudaGetLastError();
    const uint32_t ncb = (uint32_t)(q.C / 64);
    const uint32_t nsl = (uint32_t)((q.g + kLongRows - 1) / kLongRows);
    const size_t n_keys = (size_t)(q.outer * q.ngroups * q.C);
    cudaError_t e = cudaMemsetAsync(a.ws, 0, n_keys * 4, st);
    if (e == cudaSuccess && asym) e = cudaMemsetAsync(static_cast<uint32_t*>(a.ws) + n_keys, 0xFF, n_keys * 4, st);
    if (e != cudaSuccess) return e;
    int dev = 0, l2 = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    const int64_t per_o = q.T * q.C * 2;
    const int64_t chunk = std::max<int64_t>(1, (int64_t)l2 / 2 / std::max<int64_t>(per_o, 1));
    const int sms = sm_count();
    for (int64_t ob = 0; ob < q.outer; ob += chunk) {
        const uint32_t n = (uint32_t)std::min(chunk, q.outer - ob);
        const int64_t ntiles = (int64_t)n * q.ngroups * nsl * ncb;
        const unsigned grid = grid_cap(sms, ntiles, kThr / 32);
        if (asym) ql_stats_kernel<true><<<grid, kThr, 0, st>>>(a, ncb, nsl, (uint32_t)ob, n);
        else ql_stats_kernel<false><<<grid, kThr, 0, st>>>(a, ncb, nsl, (uint32_t)ob, n);
        switch (q.bits) {
        case 8: asym ? ql_apply_kernel<8, true><<<grid, kThr, 0, st>>>(a, ncb, nsl, (uint32_t)ob, n)
                     : ql_apply_kernel<8, false><<<grid, kThr, 0, st>>>(a, ncb, nsl, (uint32_t)ob, n); break;
        case 4: asym ? ql_apply_kernel<4, true><<<grid, kThr, 0, st>>>(a, ncb, nsl, (uint32_t)ob, n)
                     : ql_apply_kernel<4, false><<<grid, kThr, 0, st>>>(a, ncb, nsl, (uint32_t)ob, n); break;
        default: asym ? ql_apply_kernel<2, true><<<grid, kThr, 0, st>>>(a, ncb, nsl, (uint32_t)ob, n)
                      : ql_apply_kernel<2, false><<<grid, kThr, 0, st>>>(a, ncb, nsl, (uint32_t)ob, n); break;
        }
    }
    return cudaGetLastError();
}

// ---- dequantize / statistics

namespace {

struct DGeo { int kind; unsigned grid; int lcpr; uint32_t ncb, nsl; int lr_rpt; };

DGeo dgeo(const QSpec& q, int sms)
{
    DGeo G = {-1, 1, 0, 0, 0, 0};
    if (q.axis == KVQ_GROUP_ALONG_C) {
        if (!c_ok(q)) return G;
        G.kind = 0;
        G.lcpr = log2_exact(q.C / 64);
        G.grid = grid_cap(sms, (q.outer * q.T) << G.lcpr, kThr);
        return G;
    }
    if (!t_ok(q)) return G;
    G.kind = 1;
    const int64_t TR = 64;                  // LR=4 x RPT=16 tokens per tile
    G.ncb = (uint32_t)(q.C / 64);
    G.nsl = (uint32_t)((q.g + TR - 1) / TR);
    const int64_t nres = (q.R + TR - 1) / TR;
    G.grid = grid_cap(sms, q.outer * (q.ngroups * G.nsl + nres) * G.ncb, kThr / 32);
    return G;
}

template <int BITS, bool ASYM, bool STATS>
void dq_typed(const QArgs& a, const DGeo& G, Partial* partials, cudaStream_t st)
{
    const QSpec& q = a.q;
    if (G.kind == 0) {
        switch (q.g) {
        case 8: dc_kernel<BITS, ASYM, 8, STATS><<<G.grid, kThr, 0, st>>>(a, G.lcpr, partials); break;
        case 16: dc_kernel<BITS, ASYM, 16, STATS><<<G.grid, kThr, 0, st>>>(a, G.lcpr, partials); break;
        case 32: dc_kernel<BITS, ASYM, 32, STATS><<<G.grid, kThr, 0, st>>>(a, G.lcpr, partials); break;
        case 64: dc_kernel<BITS, ASYM, 64, STATS><<<G.grid, kThr, 0, st>>>(a, G.lcpr, partials); break;
        case 128: dc_kernel<BITS, ASYM, 128, STATS><<<G.grid, kThr, 0, st>>>(a, G.lcpr, partials); break;
        default: dc_kernel<BITS, ASYM, 256, STATS><<<G.grid, kThr, 0, st>>>(a, G.lcpr, partials); break;
        }
    } else {
        dt_kernel<BITS, ASYM, 4, 16, STATS><<<G.grid, kThr, 0, st>>>(a, G.ncb, G.nsl, partials);
    }
}

template <bool STATS>
void dq_dispatch(const QArgs& a, const DGeo& G, Partial* partials, cudaStream_t st)
{
    const bool asym = a.q.mode == KVQ_ASYM;
    switch (a.q.bits) {
    case 8: asym ? dq_typed<8, true, STATS>(a, G, partials, st) : dq_typed<8, false, STATS>(a, G, partials, st); break;
    case 4: asym ? dq_typed<4, true, STATS>(a, G, partials, st) : dq_typed<4, false, STATS>(a, G, partials, st); break;
    default: asym ? dq_typed<2, true, STATS>(a, G, partials, st) : dq_typed<2, false, STATS>(a, G, partials, st); break;
    }
}

}  // namespace

bool fast_dequant_supported(const QSpec& q, int out_dt)
{
    return stream_dequant_supported(q, out_dt) || (out_dt == KVQ_BF16 && dgeo(q, 1).kind >= 0);
}

cudaError_t fast_dequantize(const QArgs& a, cudaStream_t st)
{
    if (stream_dequant_supported(a.q, KVQ_BF16)) return stream_dequantize(a, st);
    const DGeo G = dgeo(a.q, sm_count());
    dq_dispatch<false>(a, G, nullptr, st);
    return cudaGetLastError();
}

// block count of the statistics launch (bounds the workspace)
int64_t fast_stats_blocks(const QSpec& q, int sms)
{
    const int64_t sb = stream_stats_blocks(q, sms);
    if (sb > 0) return sb;
    const DGeo G = dgeo(q, sms);
    return G.kind >= 0 ? (int64_t)G.grid : -1;
}

cudaError_t fast_error_stats(const QArgs& a, void* partials, cudaStream_t st)
{
    if (stream_stats_blocks(a.q, 1) > 0) return stream_error_stats(a, partials, nullptr, nullptr, st);
    const DGeo G = dgeo(a.q, sm_count());
    dq_dispatch<true>(a, G, static_cast<Partial*>(partials), st);
    return cudaGetLastError();
}

}  // namespace kvq
