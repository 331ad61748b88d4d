// quant.cu -- quantize kernels.
//
// Method ("KV Compression 公式到源码对照" §1.1 and §1.2; "KV cache 压缩：
// 把历史装得更小" §"量化：位置都留着，每个数更短" for the group-wise form and
// the KIVI axes, §"带残差区的压缩预算，逐项加起来" for the residual window):
//   per group: amax = max|x| (or min, max), floored at 1e-8;
//   s = amax/qmax (or (max-min)/(qmax-qmin)), rounded to its storage dtype;
//   zp = rint(qmin - min/s), stored; q = clip(rint(x/s) [+ zp], lo, hi);
//   codes packed along C; the last min(R, T) tokens copied to the residual.
//
// Kernel families (all HBM-bound; no tensor cores -- nothing here is a
// contraction):
//   quant_c_kernel      groups of g channels of one token (V / "per token"):
//                       each lane owns 8 consecutive channels (one 16-byte
//                       load), a group is g/8 adjacent lanes reduced with
//                       warp shuffles, codes leave as one 2/4/8-byte store.
//   quant_t_tile_kernel groups of g <= 128 tokens of one channel (K / "per
//                       channel"): a CTA owns a [g x 128-channel] tile held
//                       in registers, reduces over tokens through shared
//                       memory and writes the packed tile.
//   quant_t_stats/apply groups longer than 128 tokens: a stats pass folds
//                       per-slice abs-max (or min/max) into the workspace with
//                       order-preserving integer atomics, then an apply pass
//                       re-reads the slice (from L2 where the chunk fits) and
//                       writes codes and metadata.
//   quant_generic_*     any other shape or alignment: one thread per group
//                       for the metadata, one thread per code byte.
#include <algorithm>

#include "kvq_device.cuh"

namespace kvq {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;      // chunks in flight per lane (along C)
constexpr int kTileRows = 8;    // rows per thread in a [16 x 16]-thread tile
constexpr int kSliceRows = 16 * kTileRows;

template <typename InT> __device__ __forceinline__ const InT* src(const QArgs& a) {
    return static_cast<const InT*>(a.x);
}

// ======================================================================
// groups along C (per token)
// ======================================================================
template <typename InT, int BITS, bool ASYM>
__global__ void __launch_bounds__(kThreads)
quant_c_kernel(const QArgs a, int lcpr, int lanes)
{
    const QSpec& q = a.q;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int cpr = 1 << lcpr;                       // 8-element chunks per row
    const int64_t ntiles = (q.T * cpr + 31) >> 5;    // 32 chunks per warp tile
    const int64_t stride = (int64_t)gridDim.x * (kThreads / 32);
    const InT* x = src<InT>(a);
    InT* resid = static_cast<InT*>(a.resid);
    uint8_t* codes = static_cast<uint8_t*>(a.codes);
    const int64_t code_row_B = (int64_t)cpr * BITS;  // C*BITS/8
    const int gpr = cpr / lanes;                     // groups per row

    for (int64_t o = blockIdx.y; o < q.outer; o += gridDim.y) {
        for (int64_t tile0 = (int64_t)blockIdx.x * (kThreads / 32) + warp; tile0 < ntiles;
             tile0 += stride * kUnroll) {
            Raw8<InT> raw[kUnroll];
            int64_t tt[kUnroll];
            int cc[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t tile = tile0 + u * stride;
                int64_t t;
                int c;
                if (lcpr <= 5) {
                    t = (tile << (5 - lcpr)) + (lane >> lcpr);
                    c = lane & (cpr - 1);
                } else {
                    t = tile >> (lcpr - 5);
                    c = (int)((tile & ((1 << (lcpr - 5)) - 1)) << 5) + lane;
                }
                if (tile >= ntiles) t = q.T;                // mark invalid
                tt[u] = t;
                cc[u] = c;
                if (t < q.T) load_raw8(x + (((o * q.T + t) << lcpr) + c) * 8, raw[u]);
                else zero_raw8(raw[u]);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                float v[8];
                widen8(raw[u], v);
                Meta m;
                if (!ASYM) {
                    float am = 0.0f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) am = fmaxf(am, fabsf(v[j]));
                    m = meta_sym(warp_max_xor(am, lanes), q);
                } else {
                    float mn = v[0], mx = v[0];
#pragma unroll
                    for (int j = 1; j < 8; ++j) { mn = fminf(mn, v[j]); mx = fmaxf(mx, v[j]); }
                    m = meta_asym(warp_min_xor(mn, lanes), warp_max_xor(mx, lanes), q);
                }
                const int64_t t = tt[u];
                if (t >= q.T) continue;
                const int c = cc[u];
                if (t >= q.Tq) {
                    store_raw8(resid + (((o * q.R + (t - q.Tq)) << lcpr) + c) * 8, raw[u]);
                    continue;
                }
                const int64_t row = o * q.Tq + t;
                if ((lane & (lanes - 1)) == 0) write_meta(a, row * gpr + c / lanes, m);
                int qc[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) qc[j] = quant_code<ASYM>(v[j], m, q.lo, q.hi);
                *reinterpret_cast<typename CodeWord<BITS>::T*>(codes + row * code_row_B + (int64_t)c * BITS) =
                    pack8<BITS>(qc);
            }
        }
    }
}

// ======================================================================
// groups along T (per channel), g <= 128: one register tile per CTA
// ======================================================================
template <typename InT, int BITS, bool ASYM>
__global__ void __launch_bounds__(kThreads)
quant_t_tile_kernel(const QArgs a, int64_t ncb)
{
    const QSpec& q = a.q;
    __shared__ float red0[16][129];
    __shared__ float red1[16][129];
    __shared__ float ms[128], mz[128];

    const int tc = threadIdx.x & 15, tr = threadIdx.x >> 4;
    const int64_t cb = blockIdx.x % ncb;
    const int64_t tix = blockIdx.x / ncb;
    const int64_t cchunk = cb * 16 + tc;
    const int64_t c0 = cchunk * 8;
    const bool cvalid = c0 < q.C;
    const InT* x = src<InT>(a);

    for (int64_t o = blockIdx.y; o < q.outer; o += gridDim.y) {
        if (tix >= q.ngroups) {
            // residual tile: 128 tokens of the window
            InT* resid = static_cast<InT*>(a.resid);
            const int64_t r0 = (tix - q.ngroups) * kSliceRows;
#pragma unroll
            for (int k = 0; k < kTileRows; ++k) {
                const int64_t r = r0 + tr + 16 * k;
                if (cvalid && r < q.R) {
                    Raw8<InT> raw;
                    load_raw8(x + (o * q.T + q.Tq + r) * q.C + c0, raw);
                    store_raw8(resid + (o * q.R + r) * q.C + c0, raw);
                }
            }
            continue;
        }
        const int64_t t0 = tix * q.g;
        const int64_t glen = min(q.g, q.Tq - t0);
        Raw8<InT> raw[kTileRows];
#pragma unroll
        for (int k = 0; k < kTileRows; ++k) {
            const int64_t r = tr + 16 * k;
            if (cvalid && r < glen) load_raw8(x + (o * q.T + t0 + r) * q.C + c0, raw[k]);
            else zero_raw8(raw[k]);
        }
        float p0[8], p1[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) { p0[j] = ASYM ? INFINITY : 0.0f; p1[j] = -INFINITY; }
#pragma unroll
        for (int k = 0; k < kTileRows; ++k) {
            if (tr + 16 * k < glen) {
                float v[8];
                widen8(raw[k], v);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (ASYM) { p0[j] = fminf(p0[j], v[j]); p1[j] = fmaxf(p1[j], v[j]); }
                    else p0[j] = fmaxf(p0[j], fabsf(v[j]));
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            red0[tr][tc * 8 + j] = p0[j];
            if (ASYM) red1[tr][tc * 8 + j] = p1[j];
        }
        __syncthreads();
        if (threadIdx.x < 128) {
            const int ch = threadIdx.x;
            float r0 = red0[0][ch], r1 = ASYM ? red1[0][ch] : 0.0f;
#pragma unroll
            for (int i = 1; i < 16; ++i) {
                if (ASYM) { r0 = fminf(r0, red0[i][ch]); r1 = fmaxf(r1, red1[i][ch]); }
                else r0 = fmaxf(r0, red0[i][ch]);
            }
            const Meta m = ASYM ? meta_asym(r0, r1, q) : meta_sym(r0, q);
            ms[ch] = m.s;
            mz[ch] = m.z;
            const int64_t c = cb * 128 + ch;
            if (c < q.C) write_meta(a, (o * q.ngroups + tix) * q.C + c, m);
        }
        __syncthreads();
        if (cvalid) {
            Meta mm[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) { mm[j].s = ms[tc * 8 + j]; mm[j].z = mz[tc * 8 + j]; }
            uint8_t* codes = static_cast<uint8_t*>(a.codes);
            const int64_t code_row_B = q.C / 8 * BITS;
#pragma unroll
            for (int k = 0; k < kTileRows; ++k) {
                const int64_t r = tr + 16 * k;
                if (r < glen) {
                    float v[8];
                    widen8(raw[k], v);
                    int qc[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) qc[j] = quant_code<ASYM>(v[j], mm[j], q.lo, q.hi);
                    *reinterpret_cast<typename CodeWord<BITS>::T*>(
                        codes + (o * q.Tq + t0 + r) * code_row_B + cchunk * BITS) = pack8<BITS>(qc);
                }
            }
        }
        __syncthreads();   // smem reuse across the outer loop
    }
}

// ======================================================================
// groups along T longer than one tile: stats pass + apply pass
// ======================================================================
// Workspace: uint32 keys [outer][ngroups][C] for the abs-max (SYM) or the
// max (ASYM), followed by the same array of min keys (ASYM).
template <typename InT, bool ASYM>
__global__ void __launch_bounds__(kThreads)
quant_t_stats_kernel(const QArgs a, int64_t ncb, int64_t nslices, int64_t o_base)
{
    const QSpec& q = a.q;
    __shared__ float red0[16][129];
    __shared__ float red1[16][129];
    const int tc = threadIdx.x & 15, tr = threadIdx.x >> 4;
    const int64_t cb = blockIdx.x % ncb;
    const int64_t rest = blockIdx.x / ncb;
    const int64_t slice = rest % nslices;
    const int64_t gi = rest / nslices;
    const int64_t o = o_base + blockIdx.y;
    const int64_t c0 = (cb * 16 + tc) * 8;
    const bool cvalid = c0 < q.C;
    const int64_t gend = min((gi + 1) * q.g, q.Tq);
    const int64_t tbeg = gi * q.g + slice * kSliceRows;
    const InT* x = src<InT>(a);

    float p0[8], p1[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) { p0[j] = ASYM ? INFINITY : 0.0f; p1[j] = -INFINITY; }
    Raw8<InT> raw[kTileRows];
#pragma unroll
    for (int k = 0; k < kTileRows; ++k) {
        const int64_t t = tbeg + tr + 16 * k;
        if (cvalid && t < gend) load_raw8(x + (o * q.T + t) * q.C + c0, raw[k]);
    }
#pragma unroll
    for (int k = 0; k < kTileRows; ++k) {
        const int64_t t = tbeg + tr + 16 * k;
        if (cvalid && t < gend) {
            float v[8];
            widen8(raw[k], v);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (ASYM) { p0[j] = fminf(p0[j], v[j]); p1[j] = fmaxf(p1[j], v[j]); }
                else p0[j] = fmaxf(p0[j], fabsf(v[j]));
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        red0[tr][tc * 8 + j] = p0[j];
        if (ASYM) red1[tr][tc * 8 + j] = p1[j];
    }
    __syncthreads();
    if (threadIdx.x < 128) {
        const int ch = threadIdx.x;
        const int64_t c = cb * 128 + ch;
        if (c < q.C) {
            float r0 = red0[0][ch], r1 = ASYM ? red1[0][ch] : 0.0f;
            for (int i = 1; i < 16; ++i) {
                if (ASYM) { r0 = fminf(r0, red0[i][ch]); r1 = fmaxf(r1, red1[i][ch]); }
                else r0 = fmaxf(r0, red0[i][ch]);
            }
            uint32_t* kmax = static_cast<uint32_t*>(a.ws);
            const int64_t n = q.outer * q.ngroups * q.C;
            const int64_t i = (o * q.ngroups + gi) * q.C + c;
            if (ASYM) {
                atomicMax(kmax + i, float_key(r1));
                atomicMin(kmax + n + i, float_key(r0));
            } else {
                atomicMax(kmax + i, __float_as_uint(r0));   // r0 >= 0: bits are ordered
            }
        }
    }
}

template <typename InT, int BITS, bool ASYM>
__global__ void __launch_bounds__(kThreads)
quant_t_apply_kernel(const QArgs a, int64_t ncb, int64_t nslices, int64_t o_base)
{
    const QSpec& q = a.q;
    __shared__ float ms[128], mz[128];
    const int tc = threadIdx.x & 15, tr = threadIdx.x >> 4;
    const int64_t cb = blockIdx.x % ncb;
    const int64_t rest = blockIdx.x / ncb;
    const int64_t slice = rest % nslices;
    const int64_t gi = rest / nslices;
    const int64_t o = o_base + blockIdx.y;
    const int64_t cchunk = cb * 16 + tc;
    const int64_t c0 = cchunk * 8;
    const bool cvalid = c0 < q.C;
    const int64_t gend = min((gi + 1) * q.g, q.Tq);
    const int64_t tbeg = gi * q.g + slice * kSliceRows;
    const InT* x = src<InT>(a);

    Raw8<InT> raw[kTileRows];
#pragma unroll
    for (int k = 0; k < kTileRows; ++k) {
        const int64_t t = tbeg + tr + 16 * k;
        if (cvalid && t < gend) load_raw8(x + (o * q.T + t) * q.C + c0, raw[k]);
    }
    if (threadIdx.x < 128) {
        const int ch = threadIdx.x;
        const int64_t c = cb * 128 + ch;
        Meta m = {1.0f, 0.0f};
        if (c < q.C) {
            const uint32_t* kmax = static_cast<const uint32_t*>(a.ws);
            const int64_t n = q.outer * q.ngroups * q.C;
            const int64_t i = (o * q.ngroups + gi) * q.C + c;
            m = ASYM ? meta_asym(key_float(kmax[n + i]), key_float(kmax[i]), q)
                     : meta_sym(__uint_as_float(kmax[i]), q);
            if (slice == 0) write_meta(a, i, m);
        }
        ms[ch] = m.s;
        mz[ch] = m.z;
    }
    __syncthreads();
    if (!cvalid) return;
    Meta mm[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) { mm[j].s = ms[tc * 8 + j]; mm[j].z = mz[tc * 8 + j]; }
    uint8_t* codes = static_cast<uint8_t*>(a.codes);
    const int64_t code_row_B = q.C / 8 * BITS;
#pragma unroll
    for (int k = 0; k < kTileRows; ++k) {
        const int64_t t = tbeg + tr + 16 * k;
        if (t < gend) {
            float v[8];
            widen8(raw[k], v);
            int qc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) qc[j] = quant_code<ASYM>(v[j], mm[j], q.lo, q.hi);
            *reinterpret_cast<typename CodeWord<BITS>::T*>(codes + (o * q.Tq + t) * code_row_B +
                                                           cchunk * BITS) = pack8<BITS>(qc);
        }
    }
}

// ======================================================================
// generic paths (any shape / alignment)
// ======================================================================
__device__ __forceinline__ float load_x(const QArgs& a, int64_t i) {
    if (a.q.x_dt == KVQ_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(a.x)[i]);
    return static_cast<const float*>(a.x)[i];
}

// group gi -> first element, stride, member count (metadata order)
__device__ __forceinline__ void group_geometry(const QSpec& q, int64_t gidx, int64_t& first,
                                               int64_t& stride, int64_t& count) {
    if (q.axis == KVQ_GROUP_ALONG_T) {
        const int64_t c = gidx % q.C;
        const int64_t gi = (gidx / q.C) % q.ngroups;
        const int64_t o = gidx / (q.C * q.ngroups);
        const int64_t t0 = gi * q.g;
        count = min(q.g, q.Tq - t0);
        first = (o * q.T + t0) * q.C + c;
        stride = q.C;
    } else {
        const int64_t gi = gidx % q.ngroups;
        const int64_t t = (gidx / q.ngroups) % q.Tq;
        const int64_t o = gidx / (q.ngroups * q.Tq);
        const int64_t c0 = gi * q.g;
        count = min(q.g, q.C - c0);
        first = (o * q.T + t) * q.C + c0;
        stride = 1;
    }
}

__global__ void quant_generic_meta_kernel(const QArgs a, int64_t ngroups_total)
{
    const QSpec& q = a.q;
    for (int64_t gidx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gidx < ngroups_total;
         gidx += (int64_t)gridDim.x * blockDim.x) {
        int64_t first, stride, count;
        group_geometry(q, gidx, first, stride, count);
        float am = 0.0f, mn = INFINITY, mx = -INFINITY;
        for (int64_t m = 0; m < count; ++m) {
            const float v = load_x(a, first + m * stride);
            am = fmaxf(am, fabsf(v));
            mn = fminf(mn, v);
            mx = fmaxf(mx, v);
        }
        const Meta mt = q.mode == KVQ_ASYM ? meta_asym(mn, mx, q) : meta_sym(am, q);
        write_meta(a, gidx, mt);
    }
}

__global__ void quant_generic_codes_kernel(const QArgs a, int64_t nbytes)
{
    const QSpec& q = a.q;
    const int per = 8 / q.bits;
    const int64_t row_B = q.C * q.bits / 8;
    uint8_t* codes = static_cast<uint8_t*>(a.codes);
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nbytes;
         b += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = b / row_B;
        const int64_t t = row % q.Tq, o = row / q.Tq;
        uint32_t byte = 0;
        for (int j = 0; j < per; ++j) {
            const int64_t c = (b % row_B) * per + j;
            const int64_t mi = q.axis == KVQ_GROUP_ALONG_T ? (o * q.ngroups + t / q.g) * q.C + c
                                                           : (o * q.Tq + t) * q.ngroups + c / q.g;
            Meta m;
            m.s = load_meta(a.scale, q.scale_dt, mi);
            m.z = q.mode == KVQ_ASYM ? load_meta(a.zero, q.zero_dt, mi) : 0.0f;
            const float v = load_x(a, (o * q.T + t) * q.C + c);
            const int code = q.mode == KVQ_ASYM ? quant_code<true>(v, m, q.lo, q.hi)
                                                : quant_code<false>(v, m, q.lo, q.hi);
            byte |= ((uint32_t)code & ((1u << q.bits) - 1u)) << (j * q.bits);
        }
        codes[b] = (uint8_t)byte;
    }
}

// residual window copy, element by element (bytes of the source dtype)
__global__ void copy_residual_kernel(const QArgs a, int64_t n_elems, int es)
{
    const QSpec& q = a.q;
    const int64_t per_o = q.R * q.C;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_elems;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t o = i / per_o, r = i % per_o;
        const int64_t si = o * q.T * q.C + q.Tq * q.C + r;
        if (es == 2) static_cast<uint16_t*>(a.resid)[i] = static_cast<const uint16_t*>(a.x)[si];
        else static_cast<uint32_t*>(a.resid)[i] = static_cast<const uint32_t*>(a.x)[si];
    }
}

int64_t grid_for(int64_t work, int64_t per_block) {
    const int64_t cap = (int64_t)sm_count() * 16;
    return std::max<int64_t>(1, std::min<int64_t>(cap, (work + per_block - 1) / per_block));
}

template <typename InT, int BITS, bool ASYM>
cudaError_t dispatch_typed(const QArgs& a, cudaStream_t st)
{
    const QSpec& q = a.q;
    const int ymax = (int)std::min<int64_t>(q.outer, 65535);
    if (q.axis == KVQ_GROUP_ALONG_C && along_c_fast_ok(q)) {
        int lcpr = 0;
        while ((int64_t(1) << lcpr) < q.C / 8) ++lcpr;
        const int64_t ntiles = (q.T * (q.C / 8) + 31) / 32;
        const int64_t want = std::max<int64_t>(1, (int64_t)sm_count() * 8 / std::max<int64_t>(q.outer, 1));
        const int64_t gx = std::max<int64_t>(1, std::min<int64_t>(want, (ntiles + 8 * kUnroll - 1) / (8 * kUnroll)));
        quant_c_kernel<InT, BITS, ASYM><<<dim3((unsigned)gx, ymax), kThreads, 0, st>>>(a, lcpr, (int)(q.g / 8));
        return cudaGetLastError();
    }
    if (q.axis == KVQ_GROUP_ALONG_T && along_t_fast_ok(q)) {
        const int64_t ncb = (q.C + 127) / 128;
        if (q.g <= kSliceRows) {
            const int64_t nres = (q.R + kSliceRows - 1) / kSliceRows;
            const int64_t gx = ncb * (q.ngroups + nres);
            quant_t_tile_kernel<InT, BITS, ASYM><<<dim3((unsigned)gx, ymax), kThreads, 0, st>>>(a, ncb);
            return cudaGetLastError();
        }
        // long groups: chunk the outer axis so one chunk's source fits in L2
        const int64_t nslices = (q.g + kSliceRows - 1) / kSliceRows;
        const size_t n_keys = (size_t)(q.outer * q.ngroups * q.C);
        cudaError_t e = cudaMemsetAsync(a.ws, 0, n_keys * 4, st);
        if (e == cudaSuccess && ASYM)
            e = cudaMemsetAsync(static_cast<uint32_t*>(a.ws) + n_keys, 0xFF, n_keys * 4, st);
        if (e != cudaSuccess) return e;
        int dev = 0, l2 = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
        const int64_t per_o = q.T * q.C * (int64_t)sizeof(InT);
        const int64_t chunk = std::max<int64_t>(1, std::min<int64_t>(65535, (int64_t)l2 / 2 / std::max<int64_t>(per_o, 1)));
        const int64_t gx = ncb * nslices * q.ngroups;
        for (int64_t ob = 0; ob < q.outer; ob += chunk) {
            const int64_t n = std::min(chunk, q.outer - ob);
            quant_t_stats_kernel<InT, ASYM><<<dim3((unsigned)gx, (unsigned)n), kThreads, 0, st>>>(a, ncb, nslices, ob);
            quant_t_apply_kernel<InT, BITS, ASYM><<<dim3((unsigned)gx, (unsigned)n), kThreads, 0, st>>>(a, ncb, nslices, ob);
        }
    } else {
        const int64_t ng = q.axis == KVQ_GROUP_ALONG_T ? q.outer * q.ngroups * q.C
                                                       : q.outer * q.Tq * q.ngroups;
        quant_generic_meta_kernel<<<(unsigned)grid_for(ng, kThreads), kThreads, 0, st>>>(a, ng);
        const int64_t nbytes = q.outer * q.Tq * q.C * q.bits / 8;
        quant_generic_codes_kernel<<<(unsigned)grid_for(nbytes, kThreads), kThreads, 0, st>>>(a, nbytes);
    }
    if (q.R > 0) {
        const int64_t n = q.outer * q.R * q.C;
        copy_residual_kernel<<<(unsigned)grid_for(n, kThreads), kThreads, 0, st>>>(a, n, (int)sizeof(InT));
    }
    return cudaGetLastError();
}

template <typename InT>
cudaError_t dispatch_bits(const QArgs& a, cudaStream_t st)
{
    const bool asym = a.q.mode == KVQ_ASYM;
    switch (a.q.bits) {
    case 8: return asym ? dispatch_typed<InT, 8, true>(a, st) : dispatch_typed<InT, 8, false>(a, st);
    case 4: return asym ? dispatch_typed<InT, 4, true>(a, st) : dispatch_typed<InT, 4, false>(a, st);
    default: return asym ? dispatch_typed<InT, 2, true>(a, st) : dispatch_typed<InT, 2, false>(a, st);
    }
}

}  // namespace

size_t quantize_workspace(const QSpec& q)
{
    if (fast_quantize_supported(q)) return fast_quantize_workspace(q);
    if (q.axis == KVQ_GROUP_ALONG_T && along_t_fast_ok(q) && q.g > kSliceRows && q.Tq > 0)
        return (size_t)(q.outer * q.ngroups * q.C) * 4 * (q.mode == KVQ_ASYM ? 2 : 1);
    return 0;
}

cudaError_t launch_quantize(const QArgs& a, cudaStream_t st)
{
    const QSpec& q = a.q;
    if (q.outer == 0 || q.T == 0 || q.C == 0) return cudaSuccess;
    if (q.Tq == 0) {
        const int64_t n = q.outer * q.R * q.C;
        const int es = q.x_dt == KVQ_BF16 ? 2 : 4;
        copy_residual_kernel<<<(unsigned)grid_for(n, kThreads), kThreads, 0, st>>>(a, n, es);
        return cudaGetLastError();
    }
    if (fast_quantize_supported(q)) {
        cudaError_t e = fast_quantize(a, st);
        if (e != cudaSuccess || fast_quantize_copies_residual(q) || q.R == 0) return e;
        const int64_t n = q.outer * q.R * q.C;
        copy_residual_kernel<<<(unsigned)grid_for(n, kThreads), kThreads, 0, st>>>(a, n, 2);
        return cudaGetLastError();
    }
    return q.x_dt == KVQ_BF16 ? dispatch_bits<__nv_bfloat16>(a, st) : dispatch_bits<float>(a, st);
}

}  // namespace kvq
