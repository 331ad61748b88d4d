// dequant.cu -- dequantize and error-statistics kernels.
//
// Method ("KV Compression 公式到源码对照" §1.3): x_hat = (q - zero_point) *
// scale, rounded once to the output dtype; the residual window is copied back
// unchanged.  The error statistics (RMSE, max |x - x_hat|, mean |x - x_hat|
// over all N elements) re-derive x_hat in registers from the codes and
// compare it with x, so x_hat never reaches memory; residual tokens
// contribute exactly zero error and are not read.
//
// Both share one kernel template per layout; STATS selects "store x_hat" or
// "accumulate |d| and d^2".  Per chunk of 8 elements the sums are float32;
// chunk sums are folded into per-thread Kahan-compensated float32
// accumulators (FP64 throughput is far too low on this part for per-element
// binary64 work), converted to binary64 once per thread, reduced per block
// and finally over blocks in a fixed order (deterministic).
#include <algorithm>

#include "kvq_device.cuh"

namespace kvq {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int kTileRows = 8;
constexpr int kSliceRows = 16 * kTileRows;

struct Partial { double s1, s2, mx; };

// Kahan-compensated float32 sums of |d| and d^2 plus the running max |d|.
struct Acc {
    float s1 = 0.0f, e1 = 0.0f, s2 = 0.0f, e2 = 0.0f, mx = 0.0f;
    __device__ __forceinline__ static void kahan(float& s, float& e, float v) {
        const float y = __fsub_rn(v, e);
        const float t = __fadd_rn(s, y);
        e = __fsub_rn(__fsub_rn(t, s), y);
        s = t;
    }
    __device__ __forceinline__ void add_chunk(const float (&x)[8], const float (&xh)[8]) {
        float c1 = 0.0f, c2 = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float d = __fsub_rn(x[j], xh[j]);
            const float ad = fabsf(d);
            c1 = __fadd_rn(c1, ad);
            c2 = __fmaf_rn(d, d, c2);
            mx = fmaxf(mx, ad);
        }
        kahan(s1, e1, c1);
        kahan(s2, e2, c2);
    }
    __device__ __forceinline__ void add_one(float x, float xh) {
        const float d = __fsub_rn(x, xh);
        const float ad = fabsf(d);
        kahan(s1, e1, ad);
        kahan(s2, e2, __fmul_rn(d, d));
        mx = fmaxf(mx, ad);
    }
};

// Block reduction of the per-thread accumulators into partials[block].
__device__ void block_reduce_store(const Acc& A, Partial* partials)
{
    __shared__ double sh1[kThreads / 32], sh2[kThreads / 32], shm[kThreads / 32];
    double s1 = (double)A.s1 - (double)A.e1;
    double s2 = (double)A.s2 - (double)A.e2;
    double mx = (double)A.mx;
    for (int o = 16; o > 0; o >>= 1) {
        s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, o);
        s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, o);
        mx = fmax(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) { sh1[w] = s1; sh2[w] = s2; shm[w] = mx; }
    __syncthreads();
    if (threadIdx.x == 0) {
        Partial p = {0.0, 0.0, 0.0};
        for (int i = 0; i < kThreads / 32; ++i) { p.s1 += sh1[i]; p.s2 += sh2[i]; p.mx = fmax(p.mx, shm[i]); }
        partials[(int64_t)blockIdx.y * gridDim.x + blockIdx.x] = p;
    }
}

// Final reduction over all block partials, fixed order (1024 threads, so a
// launch of up to a few thousand blocks needs one or two loads per thread).
__global__ void __launch_bounds__(1024) finalize_stats_kernel(const Partial* partials, int64_t n,
                                                              double N, kvq_err* out)
{
    __shared__ double s1[1024], s2[1024], mx[1024];
    double a = 0.0, b = 0.0, m = 0.0;
    for (int64_t i = threadIdx.x; i < n; i += 1024) { a += partials[i].s1; b += partials[i].s2; m = fmax(m, partials[i].mx); }
    s1[threadIdx.x] = a; s2[threadIdx.x] = b; mx[threadIdx.x] = m;
    __syncthreads();
    for (int o = 512; o > 0; o >>= 1) {
        if (threadIdx.x < o) {
            s1[threadIdx.x] += s1[threadIdx.x + o];
            s2[threadIdx.x] += s2[threadIdx.x + o];
            mx[threadIdx.x] = fmax(mx[threadIdx.x], mx[threadIdx.x + o]);
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        out->rmse = sqrt(s2[0] / N);
        out->max_abs = mx[0];
        out->mean_abs = s1[0] / N;
    }
}

template <int BITS>
__device__ __forceinline__ void decode8(typename CodeWord<BITS>::T w, bool is_signed, int (&q)[8]) {
    if (is_signed) unpack8<BITS, true>(w, q);
    else unpack8<BITS, false>(w, q);
}

// ======================================================================
// groups along C
// ======================================================================
template <typename OutT, int BITS, bool ASYM, bool STATS>
__global__ void __launch_bounds__(kThreads)
dq_c_kernel(const QArgs a, int lcpr, int lanes, Partial* partials)
{
    const QSpec& q = a.q;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int cpr = 1 << lcpr;
    const int64_t ntiles = (q.T * cpr + 31) >> 5;
    const int64_t stride = (int64_t)gridDim.x * (kThreads / 32);
    const int64_t code_row_B = (int64_t)cpr * BITS;
    const int gpr = cpr / lanes;
    const uint8_t* codes = static_cast<const uint8_t*>(a.codes);
    OutT* out = static_cast<OutT*>(a.out);
    const OutT* x = static_cast<const OutT*>(a.x);
    const OutT* resid = static_cast<const OutT*>(a.resid);
    using W = typename CodeWord<BITS>::T;
    Acc A;

    for (int64_t o = blockIdx.y; o < q.outer; o += gridDim.y) {
        for (int64_t tile0 = (int64_t)blockIdx.x * (kThreads / 32) + warp; tile0 < ntiles;
             tile0 += stride * kUnroll) {
            W w[kUnroll];
            Meta m[kUnroll];
            Raw8<OutT> xr[kUnroll];
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
                if (tile >= ntiles) t = q.T;
                tt[u] = t;
                cc[u] = c;
                if (t < q.Tq) {
                    const int64_t row = o * q.Tq + t;
                    w[u] = *reinterpret_cast<const W*>(codes + row * code_row_B + (int64_t)c * BITS);
                    const int64_t mi = row * gpr + c / lanes;
                    m[u].s = load_meta(a.scale, q.scale_dt, mi);
                    m[u].z = ASYM ? load_meta(a.zero, q.zero_dt, mi) : 0.0f;
                    if (STATS) load_raw8(x + (((o * q.T + t) << lcpr) + c) * 8, xr[u]);
                } else if (!STATS && t < q.T) {
                    load_raw8(resid + (((o * q.R + (t - q.Tq)) << lcpr) + c) * 8, xr[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t t = tt[u];
                if (t >= q.T) continue;
                const int c = cc[u];
                if (t >= q.Tq) {
                    if (!STATS) store_raw8(out + (((o * q.T + t) << lcpr) + c) * 8, xr[u]);
                    continue;
                }
                int qc[8];
                decode8<BITS>(w[u], q.is_signed, qc);
                float v[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = dequant_value(qc[j], m[u]);
                if (STATS) {
                    float xv[8], xh[8];
                    widen8(xr[u], xv);
#pragma unroll
                    for (int j = 0; j < 8; ++j) xh[j] = as_output<OutT>(v[j]);
                    A.add_chunk(xv, xh);
                } else {
                    store8(out + (((o * q.T + t) << lcpr) + c) * 8, v);
                }
            }
        }
    }
    if (STATS) block_reduce_store(A, partials);
}

// ======================================================================
// groups along T: CTA per (channel block, group, 128-token slice)
// ======================================================================
template <typename OutT, int BITS, bool ASYM, bool STATS>
__global__ void __launch_bounds__(kThreads)
dq_t_kernel(const QArgs a, int64_t ncb, int64_t nslices, Partial* partials)
{
    const QSpec& q = a.q;
    const int tc = threadIdx.x & 15, tr = threadIdx.x >> 4;
    const int64_t cb = blockIdx.x % ncb;
    const int64_t tix = blockIdx.x / ncb;
    const int64_t cchunk = cb * 16 + tc;
    const int64_t c0 = cchunk * 8;
    const bool cvalid = c0 < q.C;
    const uint8_t* codes = static_cast<const uint8_t*>(a.codes);
    OutT* out = static_cast<OutT*>(a.out);
    const OutT* x = static_cast<const OutT*>(a.x);
    const OutT* resid = static_cast<const OutT*>(a.resid);
    const int64_t code_row_B = q.C / 8 * BITS;
    using W = typename CodeWord<BITS>::T;
    Acc A;

    for (int64_t o = blockIdx.y; o < q.outer; o += gridDim.y) {
        if (!cvalid) continue;
        if (tix >= q.ngroups * nslices) {
            if (STATS) continue;                 // residual error is exactly zero
            const int64_t r0 = (tix - q.ngroups * nslices) * kSliceRows;
#pragma unroll
            for (int k = 0; k < kTileRows; ++k) {
                const int64_t r = r0 + tr + 16 * k;
                if (r < q.R) {
                    Raw8<OutT> raw;
                    load_raw8(resid + (o * q.R + r) * q.C + c0, raw);
                    store_raw8(out + (o * q.T + q.Tq + r) * q.C + c0, raw);
                }
            }
            continue;
        }
        const int64_t gi = tix / nslices, slice = tix % nslices;
        const int64_t gend = min((gi + 1) * q.g, q.Tq);
        const int64_t tbeg = gi * q.g + slice * kSliceRows;
        Meta mm[8];
        const int64_t mi = (o * q.ngroups + gi) * q.C + c0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            mm[j].s = load_meta(a.scale, q.scale_dt, mi + j);
            mm[j].z = ASYM ? load_meta(a.zero, q.zero_dt, mi + j) : 0.0f;
        }
        W w[kTileRows];
        Raw8<OutT> xr[kTileRows];
#pragma unroll
        for (int k = 0; k < kTileRows; ++k) {
            const int64_t t = tbeg + tr + 16 * k;
            if (t < gend) {
                w[k] = *reinterpret_cast<const W*>(codes + (o * q.Tq + t) * code_row_B + cchunk * BITS);
                if (STATS) load_raw8(x + (o * q.T + t) * q.C + c0, xr[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < kTileRows; ++k) {
            const int64_t t = tbeg + tr + 16 * k;
            if (t >= gend) continue;
            int qc[8];
            decode8<BITS>(w[k], q.is_signed, qc);
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = dequant_value(qc[j], mm[j]);
            if (STATS) {
                float xv[8], xh[8];
                widen8(xr[k], xv);
#pragma unroll
                for (int j = 0; j < 8; ++j) xh[j] = as_output<OutT>(v[j]);
                A.add_chunk(xv, xh);
            } else {
                store8(out + (o * q.T + t) * q.C + c0, v);
            }
        }
    }
    if (STATS) block_reduce_store(A, partials);
}

// ======================================================================
// generic: one thread per element
// ======================================================================
__device__ __forceinline__ int64_t meta_index(const QSpec& q, int64_t o, int64_t t, int64_t c) {
    return q.axis == KVQ_GROUP_ALONG_T ? (o * q.ngroups + t / q.g) * q.C + c
                                       : (o * q.Tq + t) * q.ngroups + c / q.g;
}

template <typename OutT, bool STATS>
__global__ void __launch_bounds__(kThreads)
dq_generic_kernel(const QArgs a, int64_t n, Partial* partials)
{
    const QSpec& q = a.q;
    const uint8_t* codes = static_cast<const uint8_t*>(a.codes);
    OutT* out = static_cast<OutT*>(a.out);
    const OutT* x = static_cast<const OutT*>(a.x);
    const OutT* resid = static_cast<const OutT*>(a.resid);
    Acc A;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t c = i % q.C;
        const int64_t t = (i / q.C) % q.T;
        const int64_t o = i / (q.C * q.T);
        if (t >= q.Tq) {
            if (!STATS) out[i] = resid[(o * q.R + (t - q.Tq)) * q.C + c];
            continue;
        }
        const int64_t mi = meta_index(q, o, t, c);
        Meta m;
        m.s = load_meta(a.scale, q.scale_dt, mi);
        m.z = q.mode == KVQ_ASYM ? load_meta(a.zero, q.zero_dt, mi) : 0.0f;
        const int code = code_at(codes, q.bits, (o * q.Tq + t) * q.C + c, q.is_signed != 0);
        const float v = dequant_value(code, m);
        if (STATS) {
            float xv;
            if constexpr (sizeof(OutT) == 2) xv = __bfloat162float(x[i]);
            else xv = x[i];
            A.add_one(xv, as_output<OutT>(v));
        } else {
            if constexpr (sizeof(OutT) == 2) out[i] = __float2bfloat16_rn(v);
            else out[i] = v;
        }
    }
    if (STATS) block_reduce_store(A, partials);
}

// ======================================================================
// launch geometry (shared by dequantize, error stats and the workspace size)
// ======================================================================
struct Geometry {
    int kind;            // 0 = along C fast, 1 = along T fast, 2 = generic
    dim3 grid;
    int lcpr = 0;
    int64_t ncb = 0, nslices = 0;
};

Geometry geometry(const QSpec& q, int sms)
{
    Geometry G;
    const unsigned ymax = (unsigned)std::max<int64_t>(1, std::min<int64_t>(q.outer, 65535));
    if (q.axis == KVQ_GROUP_ALONG_C && along_c_fast_ok(q)) {
        G.kind = 0;
        while ((int64_t(1) << G.lcpr) < q.C / 8) ++G.lcpr;
        const int64_t ntiles = (q.T * (q.C / 8) + 31) / 32;
        const int64_t want = std::max<int64_t>(1, (int64_t)sms * 8 / std::max<int64_t>(q.outer, 1));
        const int64_t gx = std::max<int64_t>(1, std::min<int64_t>(want, (ntiles + 8 * kUnroll - 1) / (8 * kUnroll)));
        G.grid = dim3((unsigned)gx, ymax);
    } else if (q.axis == KVQ_GROUP_ALONG_T && along_t_fast_ok(q)) {
        G.kind = 1;
        G.ncb = (q.C + 127) / 128;
        G.nslices = (q.g + kSliceRows - 1) / kSliceRows;
        const int64_t nres = (q.R + kSliceRows - 1) / kSliceRows;
        G.grid = dim3((unsigned)(G.ncb * (q.ngroups * G.nslices + nres)), ymax);
    } else {
        G.kind = 2;
        const int64_t n = q.outer * q.T * q.C;
        const int64_t cap = (int64_t)sms * 16;
        G.grid = dim3((unsigned)std::max<int64_t>(1, std::min<int64_t>(cap, (n + kThreads - 1) / kThreads)), 1);
    }
    return G;
}

template <typename OutT, int BITS, bool ASYM, bool STATS>
void launch_typed(const QArgs& a, const Geometry& G, Partial* partials, cudaStream_t st)
{
    const QSpec& q = a.q;
    if (G.kind == 0)
        dq_c_kernel<OutT, BITS, ASYM, STATS><<<G.grid, kThreads, 0, st>>>(a, G.lcpr, (int)(q.g / 8), partials);
    else if (G.kind == 1)
        dq_t_kernel<OutT, BITS, ASYM, STATS><<<G.grid, kThreads, 0, st>>>(a, G.ncb, G.nslices, partials);
    else
        dq_generic_kernel<OutT, STATS><<<G.grid, kThreads, 0, st>>>(a, q.outer * q.T * q.C, partials);
}

template <typename OutT, bool STATS>
void launch_bits(const QArgs& a, const Geometry& G, Partial* partials, cudaStream_t st)
{
    const bool asym = a.q.mode == KVQ_ASYM;
    switch (a.q.bits) {
    case 8: asym ? launch_typed<OutT, 8, true, STATS>(a, G, partials, st) : launch_typed<OutT, 8, false, STATS>(a, G, partials, st); break;
    case 4: asym ? launch_typed<OutT, 4, true, STATS>(a, G, partials, st) : launch_typed<OutT, 4, false, STATS>(a, G, partials, st); break;
    default: asym ? launch_typed<OutT, 2, true, STATS>(a, G, partials, st) : launch_typed<OutT, 2, false, STATS>(a, G, partials, st); break;
    }
}

__global__ void copy_back_residual_kernel(const QArgs a, int64_t n, int es)
{
    const QSpec& q = a.q;
    const int64_t per_o = q.R * q.C;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t o = i / per_o, r = i % per_o;
        const int64_t di = o * q.T * q.C + q.Tq * q.C + r;
        if (es == 2) static_cast<uint16_t*>(a.out)[di] = static_cast<const uint16_t*>(a.resid)[i];
        else static_cast<uint32_t*>(a.out)[di] = static_cast<const uint32_t*>(a.resid)[i];
    }
}

}  // namespace

// Upper bound on the SM count used to size the workspace without a device
// query (the launch uses the real count, which only lowers the block count).
constexpr int kMaxSms = 1024;

// Statistics workspace: a 256-byte header (the completion counter of the
// fused final reduction) followed by one Partial per block.
constexpr size_t kStatsHeader = 256;

size_t errstats_workspace(const QSpec& q)
{
    const Geometry G = geometry(q, kMaxSms);
    const int64_t fast = fast_stats_blocks(q, kMaxSms);
    return kStatsHeader +
           std::max<size_t>((size_t)G.grid.x * G.grid.y, (size_t)std::max<int64_t>(fast, 0)) * sizeof(Partial);
}

cudaError_t launch_dequantize(const QArgs& a, int out_dt, cudaStream_t st)
{
    const QSpec& q = a.q;
    if (q.outer == 0 || q.T == 0 || q.C == 0) return cudaSuccess;
    if (q.Tq == 0) {
        const int64_t n = q.outer * q.R * q.C;
        const int64_t g = std::max<int64_t>(1, std::min<int64_t>((int64_t)sm_count() * 16, (n + 255) / 256));
        copy_back_residual_kernel<<<(unsigned)g, 256, 0, st>>>(a, n, out_dt == KVQ_BF16 ? 2 : 4);
        return cudaGetLastError();
    }
    if (fast_dequant_supported(q, out_dt)) return fast_dequantize(a, st);
    const Geometry G = geometry(q, sm_count());
    if (out_dt == KVQ_BF16) launch_bits<__nv_bfloat16, false>(a, G, nullptr, st);
    else launch_bits<float, false>(a, G, nullptr, st);
    return cudaGetLastError();
}

cudaError_t launch_error_stats(const QArgs& a, kvq_err* out_dev, cudaStream_t st)
{
    const QSpec& q = a.q;
    const Geometry G = geometry(q, sm_count());
    unsigned int* done = static_cast<unsigned int*>(a.ws);
    Partial* partials = reinterpret_cast<Partial*>(static_cast<char*>(a.ws) + kStatsHeader);
    int64_t nblocks = (int64_t)G.grid.x * G.grid.y;
    if (q.Tq > 0 && stream_stats_blocks(q, sm_count()) > 0) {
        // streaming kernel with the final reduction fused into its last block
        cudaError_t e = cudaMemsetAsync(done, 0, sizeof(unsigned int), st);
        if (e != cudaSuccess) return e;
        return stream_error_stats(a, partials, done, out_dev, st);
    }
    const int64_t fast_blocks = fast_stats_blocks(q, sm_count());
    if (q.Tq > 0 && fast_blocks > 0) {
        nblocks = fast_blocks;
        cudaError_t e = fast_error_stats(a, partials, st);
        if (e != cudaSuccess) return e;
    } else if (q.Tq == 0) {
        cudaError_t e = cudaMemsetAsync(partials, 0, (size_t)nblocks * sizeof(Partial), st);
        if (e != cudaSuccess) return e;
    } else if (q.x_dt == KVQ_BF16) {
        launch_bits<__nv_bfloat16, true>(a, G, partials, st);
    } else {
        launch_bits<float, true>(a, G, partials, st);
    }
    finalize_stats_kernel<<<1, 1024, 0, st>>>(partials, nblocks, (double)(q.outer * q.T * q.C), out_dev);
    return cudaGetLastError();
}

}  // namespace kvq
