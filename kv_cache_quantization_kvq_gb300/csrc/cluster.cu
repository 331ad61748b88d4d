// cluster.cu -- quantize, groups along T longer than one tile (bf16 sources):
// one scale per channel over hundreds to thousands of tokens, up to a whole
// layer's context.
//
// Method: "KV Compression 公式到源码对照" §1.1 (symmetric per-channel
// quantization: scale = max|x| / qmax, q = clip(round(x / scale))) and §1.2
// (asymmetric: min / max, zero point); "KV cache 压缩：把历史装得更小" group-wise
// form with K grouped per channel.  Same results as the other quantize
// kernels, bit for bit (same group constants, same exact quotient).
//
// A unit is (outer slice, group along T, block of 64 channels).  One
// thread-block cluster of NC CTAs takes a unit, so the group is read from HBM
// exactly once:
//  1. CTA r of the cluster takes rows [r*sl, (r+1)*sl) of the group (sl =
//     ceil(group length / NC)).  Groups of up to 2048 tokens: sl <= 512 rows,
//     all in shared memory (or <= 1024 where clusters of 16 cannot be
//     resident), three CTAs per SM.  Longer groups: sl <= 1024 rows, the first
//     512 in shared memory and the rest in registers (16 words of 16 bytes per
//     thread, loaded with plain coalesced loads), two CTAs per SM and at most
//     8 CTAs per cluster.  Shared-memory rows arrive by 3-D TMA boxes of 256
//     rows x 64 channels, each completing on its own mbarrier (rows past the
//     quantized tokens are zero-filled, not read);
//  2. it folds the per-channel abs-max (or min and max) of its rows as bf16
//     pairs and publishes them in its shared memory;
//  3. after a cluster barrier, one warp reads the NC partials of every CTA of
//     the cluster through distributed shared memory, derives the group
//     constants of the 64 channels and (cluster rank 0) stores the scales and
//     zero points;
//  4. every thread then quantizes its rows straight from shared memory and
//     registers and stores the codes.
// A second cluster barrier, arrived at after step 3 and waited on at exit,
// keeps each CTA resident until its peers have read its partials.  With 64 KB
// slices three CTAs share an SM, so while one cluster exchanges or quantizes
// another is loading.  For 8192-token groups the register rows halve the
// cluster (8 CTAs instead of 16), which measured 0.81x the time; for groups
// of 1024 to 2048 tokens the three-CTA form measured faster.  (Persistent
// clusters walking the units through a ring of slices measured slower: fewer
// clusters are resident, and the adjacent channel blocks read at the same
// time -- 128 bytes of every 8 KB row per unit -- then span less of each row.)
#include <algorithm>
#include <mutex>

#include <cudaTypedefs.h>

#include "kvq_bulk.cuh"
#include "kvq_elem.cuh"

namespace kvq {

namespace {

using namespace elem;

constexpr int kLCB = 64;                         // channels per unit
constexpr int kLThreads = 256;
constexpr int kLWarps = kLThreads / 32;
constexpr int kLTPR = kLCB / 8;                  // threads per row (16 bytes each)
constexpr int kLRPP = kLThreads / kLTPR;         // rows per pass of the CTA: 32
constexpr int kLBoxRows = 256;                   // rows per TMA box
constexpr uint32_t kLRowB = kLCB * 2;            // 128 bytes of bf16 per row
constexpr uint32_t kLBoxB = kLBoxRows * kLRowB;  // 32 KB
constexpr int kLMaxBoxes = 4;                    // at most 1024 rows per CTA
constexpr uint32_t kLMaxCluster = 16;
constexpr uint32_t kLSmemCap = kLMaxBoxes * kLBoxB + 128;   // dynamic shared memory (+ alignment slack)
constexpr int64_t kLMaxGroup = 8192;             // 16 CTAs x 512 rows, or 8 x 1024
constexpr int kLRegWords = 16;                   // 16-byte register words per thread: 512 rows per CTA
constexpr uint32_t kLRegSmemRows = 512;          // rows in shared memory beside them
constexpr int64_t kLRegMinGroup = 2048;          // longer groups take the register variant

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// A 32-bit word of shared memory of CTA `rank` of the cluster, at the same
// offset as `local` in this CTA.
__device__ __forceinline__ uint32_t ld_peer_u32(const void* local, uint32_t rank) {
    uint32_t addr, v;
    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(addr) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// 3-D tiled tensor copy: box at element coordinates (x, y, z) -> smem, bytes
// counted on bar.  x * 2 bytes is a multiple of 16 (x is a multiple of 64).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// One 16-byte global load that bypasses L1 (the rows are read once).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// NR = 0: every row of the CTA's slice is held in shared memory (three CTAs
// per SM).  NR > 0: the first `smax` rows are held in shared memory and up to
// kLRPP * NR more in registers, NR 16-byte words per thread loaded straight
// from global memory (two CTAs per SM, so a thread has 128 registers).
template <int BITS, bool ASYM, int NR>
__global__ void __launch_bounds__(kLThreads, NR ? 2 : 3)
wq_l_kernel(const QArgs a, const __grid_constant__ CUtensorMap tmap, uint32_t ncb, uint32_t nc, uint32_t smax)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // [rows][64] bf16, 128 B per row; TMA boxes land on 128-byte boundaries
    unsigned char* slice = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    __shared__ __align__(8) uint64_t full[kLMaxBoxes];
    __shared__ uint32_t red_mx[kLWarps][kLCB / 2], red_mn[kLWarps][kLCB / 2];
    __shared__ uint32_t part_mx[kLCB / 2], part_mn[kLCB / 2];  // read by the cluster's peers
    __shared__ __align__(16) float c_s[kLCB], c_inv[kLCB], c_zp[kLCB];
    __shared__ __align__(16) int32_t c_zoff[kLCB];
    __shared__ __align__(16) uint32_t c_flags[kLCB];           // bit 0: fast quotient, bit 1: no lower clip

    const QSpec& q = a.q;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t ng = (uint32_t)q.ngroups;
    const uint32_t unit = blockIdx.x / nc, rank = cluster_rank();
    const uint32_t cb = unit % ncb, gk = (unit / ncb) % ng, o = unit / (ncb * ng);
    const int64_t gstart = (int64_t)gk * q.g;
    const uint32_t glen = (uint32_t)min(q.g, q.Tq - gstart);
    const uint32_t sl = (glen + nc - 1) / nc;
    const uint32_t r0 = min(rank * sl, glen);
    const uint32_t nrows = min(sl, glen - r0);
    const uint32_t nsm = NR ? min(nrows, smax) : nrows;       // rows held in shared memory
    const uint32_t nbox = (nsm + kLBoxRows - 1) / kLBoxRows;
    const int64_t t0 = gstart + r0;                            // first token of this CTA's rows

    if (tid == 0) {
        for (uint32_t b = 0; b < nbox; ++b) mbar_init(&full[b], 1);
        mbar_init_fence();
        for (uint32_t b = 0; b < nbox; ++b) {
            mbar_expect_tx(&full[b], kLBoxB);
            tma_load_3d(slice + b * kLBoxB, &tmap, (int)(cb * kLCB), (int)(t0 + (int64_t)b * kLBoxRows), (int)o, &full[b]);
        }
    }
    __syncthreads();

    // ---- 2. per-thread fold over rows rr, rr + kLRPP, ... of 8 channels (c8)
    const int c8 = tid % kLTPR, rr = tid / kLTPR;
    // rows nsm + rr + kLRPP * i held in registers, all loads in flight at once
    uint4 rg[NR ? NR : 1];
    if constexpr (NR > 0) {
        const unsigned char* src = static_cast<const unsigned char*>(a.x) +
                                   (((uint64_t)o * q.T + (uint64_t)(t0 + nsm)) * q.C + (uint64_t)cb * kLCB + c8 * 8) * 2;
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const uint32_t r = nsm + rr + kLRPP * i;
            rg[i] = r < nrows ? ld_stream16(src + (uint64_t)(rr + kLRPP * i) * q.C * 2) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    uint32_t mn[4], mx[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) { mn[p] = kBfPosInf2; mx[p] = ASYM ? kBfNegInf2 : 0u; }
    auto fold = [&](const uint4& w) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            if (ASYM) { mn[p] = bmin2(mn[p], ws[p]); mx[p] = bmax2(mx[p], ws[p]); }
            else mx[p] = bmax2(mx[p], babs2(ws[p]));
        }
    };
    bool ok = true;
    for (uint32_t b = 0; b < nbox; ++b) {
        ok = mbar_wait(&full[b], 0) && ok;                     // a timeout is recorded in g_kvq_wait_timeouts
#pragma unroll
        for (int i = 0; i < kLBoxRows / kLRPP; ++i) {
            const uint32_t r = b * kLBoxRows + rr + kLRPP * i;
            if (r < nsm) {
                fold(*reinterpret_cast<const uint4*>(slice + r * kLRowB + c8 * 16));
            }
        }
    }
    if constexpr (NR > 0) {
#pragma unroll
        for (int i = 0; i < NR; ++i)
            if (nsm + rr + kLRPP * i < nrows) fold(rg[i]);
    }
    // lanes l, l^8, l^16, l^24 hold the same channels
#pragma unroll
    for (int s = kLTPR; s < 32; s <<= 1) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            if (ASYM) mn[p] = bmin2(mn[p], __shfl_xor_sync(0xFFFFFFFFu, mn[p], s));
            mx[p] = bmax2(mx[p], __shfl_xor_sync(0xFFFFFFFFu, mx[p], s));
        }
    }
    if (lane < kLTPR) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            red_mx[warp][lane * 4 + p] = mx[p];
            if (ASYM) red_mn[warp][lane * 4 + p] = mn[p];
        }
    }
    __syncthreads();
    if (warp == 0) {
        // lane = channel pair (2*lane, 2*lane + 1)
        uint32_t m = red_mx[0][lane], n = ASYM ? red_mn[0][lane] : 0u;
#pragma unroll
        for (int w = 1; w < kLWarps; ++w) {
            m = bmax2(m, red_mx[w][lane]);
            if (ASYM) n = bmin2(n, red_mn[w][lane]);
        }
        part_mx[lane] = m;
        if (ASYM) part_mn[lane] = n;
    }

    // ---- 3. the cluster's partials -> group constants
    __syncwarp();
    cluster_arrive();
    cluster_wait();
    if (warp == 0) {
        uint32_t pm[kLMaxCluster], pn[kLMaxCluster];
#pragma unroll
        for (uint32_t r = 0; r < kLMaxCluster; ++r)      // all loads in flight at once
            if (r < nc) {
                pm[r] = ld_peer_u32(&part_mx[lane], r);
                if (ASYM) pn[r] = ld_peer_u32(&part_mn[lane], r);
            }
        uint32_t m = ASYM ? kBfNegInf2 : 0u, n = kBfPosInf2;
#pragma unroll
        for (uint32_t r = 0; r < kLMaxCluster; ++r)
            if (r < nc) {
                m = bmax2(m, pm[r]);
                if (ASYM) n = bmin2(n, pn[r]);
            }
        const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float fmx = h ? hi_f(m) : lo_f(m);
            const float fmn = ASYM ? (h ? hi_f(n) : lo_f(n)) : 0.0f;
            const GroupC gc = make_group<ASYM>(fmn, fmx, q, off);
            const int ch = 2 * lane + h;
            c_s[ch] = gc.s;
            c_inv[ch] = gc.inv;
            c_zp[ch] = gc.zp;
            c_zoff[ch] = gc.zoff;
            c_flags[ch] = (gc.fast ? 1u : 0u) | (gc.lo_ok ? 2u : 0u);
            if (rank == 0) {
                Meta mt;
                mt.s = gc.s;
                mt.z = gc.zp;
                write_meta(a, ((int64_t)o * ng + gk) * q.C + (int64_t)cb * kLCB + ch, mt);
            }
        }
    }
    __syncwarp();
    cluster_arrive();          // this CTA is done with its peers' shared memory (waited on at exit)
    __syncthreads();

    // ---- 4. codes of this CTA's rows
    if (nrows) {
        const int off = q.is_signed ? (1 << (BITS - 1)) : 0;
        const int lo_c = q.qmin + off, hi_c = q.qmax + off;
        float s8[8], i8[8], z8[8];
        int32_t zo[8];
        uint32_t fl = 3u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int ch = c8 * 8 + j;
            s8[j] = c_s[ch];
            i8[j] = c_inv[ch];
            z8[j] = c_zp[ch];
            zo[j] = c_zoff[ch];
            fl &= c_flags[ch];
        }
        QuotK kq[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            kq[p].ns = pk(-s8[2 * p], -s8[2 * p + 1]);
            kq[p].inv = pk(i8[2 * p], i8[2 * p + 1]);
        }
        const uint64_t code_row_B = (uint64_t)q.C * BITS / 8;
        uint8_t* cbase = static_cast<uint8_t*>(a.codes) + ((uint64_t)o * q.Tq + (uint64_t)t0) * code_row_B +
                         ((uint64_t)cb * kLCB + (uint64_t)c8 * 8) * BITS / 8;
        auto rows = [&](auto codes_of) {
            for (uint32_t b = 0; b < nbox; ++b) {
#pragma unroll 4
                for (int i = 0; i < kLBoxRows / kLRPP; ++i) {
                    const uint32_t r = b * kLBoxRows + rr + kLRPP * i;
                    if (r < nsm) {
                        const uint4 w = *reinterpret_cast<const uint4*>(slice + r * kLRowB + c8 * 16);
                        uint32_t cc[8];
                        codes_of(w, cc);
                        store_codes<BITS>(cbase + (uint64_t)r * code_row_B, finish_word<BITS>(cc, q.is_signed));
                    }
                }
            }
            if constexpr (NR > 0) {
#pragma unroll
                for (int i = 0; i < NR; ++i) {
                    const uint32_t r = nsm + rr + kLRPP * i;
                    if (r < nrows) {
                        uint32_t cc[8];
                        codes_of(rg[i], cc);
                        store_codes<BITS>(cbase + (uint64_t)r * code_row_B, finish_word<BITS>(cc, q.is_signed));
                    }
                }
            }
        };
        if (fl & 1u) {
            if (!ASYM || (fl & 2u)) rows([&](const uint4& w, uint32_t(&cc)[8]) { codes8_fast<ASYM, false>(w, kq, zo, lo_c, hi_c, cc); });
            else rows([&](const uint4& w, uint32_t(&cc)[8]) { codes8_fast<ASYM, true>(w, kq, zo, lo_c, hi_c, cc); });
        } else {
            rows([&](const uint4& w, uint32_t(&cc)[8]) { codes8_slow<ASYM>(w, s8, z8, q, off, cc); });
        }
    }

    // after a timed-out wait, wait (bounded) again so no copy is left in flight
    if (tid == 0 && !ok)
        for (uint32_t b = 0; b < nbox; ++b) mbar_wait(&full[b], 0);
    __syncwarp();
    cluster_wait();
}

// [outer, Tq, C] bf16 rows of x (row stride C, slice stride T*C) as boxes of
// 64 channels x 256 rows x 1 slice, no swizzle; rows >= Tq are outside the map
// (zero-filled, never read from memory).
bool encode_slices_map(const QSpec& q, const void* x, CUtensorMap* map) {
    auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)q.C, (cuuint64_t)q.Tq, (cuuint64_t)q.outer};
    const cuuint64_t strides[2] = {(cuuint64_t)q.C * 2, (cuuint64_t)q.T * (cuuint64_t)q.C * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kLCB, (cuuint32_t)kLBoxRows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Resident clusters of `nc` CTAs with `smem` bytes of dynamic shared memory
// each (0: none), queried once per device and configuration.
template <typename K>
int resident_clusters(K kernel, uint32_t nc, uint32_t smem) {
    struct Entry { const void* fn; int dev; uint32_t nc, smem; int n; };
    static Entry table[64];
    static int used = 0;
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    const void* fn = reinterpret_cast<const void*>(kernel);
    for (int i = 0; i < used; ++i)
        if (table[i].fn == fn && table[i].dev == dev && table[i].nc == nc && table[i].smem == smem) return table[i].n;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = nc;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(nc);
    cfg.blockDim = dim3(kLThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 0) {
        cudaGetLastError();
        n = 0;
    }
    if (used < 64) table[used++] = Entry{fn, dev, nc, smem, n};
    return n;
}

template <int BITS, bool ASYM, int NR>
bool wq_l_launch(const QArgs& a, cudaStream_t st) {
    const QSpec& q = a.q;
    auto kernel = wq_l_kernel<BITS, ASYM, NR>;
    if (ensure_kernel_attrs(reinterpret_cast<const void*>(kernel), (int)kLSmemCap, true) != cudaSuccess) {
        cudaGetLastError();          // not handled here: the caller takes the two-pass path
        return false;
    }
    const int64_t glen = std::min(q.g, q.Tq);
    uint32_t maxr, smax;
    if (NR > 0) {
        // 512 rows in shared memory and up to 512 in registers per CTA, up
        // to 8 CTAs per cluster
        smax = kLRegSmemRows;
        maxr = smax + kLRPP * NR;
    } else {
        // 512-row slices (64 KB: three CTAs per SM) and up to 16 CTAs per
        // cluster; where 16-CTA clusters cannot be resident, 1024-row slices
        // and up to 8 CTAs
        maxr = 512;
        if ((glen + maxr - 1) / maxr > 8 && resident_clusters(kernel, (uint32_t)((glen + maxr - 1) / maxr), maxr * kLRowB + 128) < 1)
            maxr = 1024;
        smax = maxr;
    }
    const uint32_t nc = (uint32_t)((glen + maxr - 1) / maxr);
    const uint32_t ncb = (uint32_t)(q.C / kLCB);
    const int64_t units = q.outer * q.ngroups * (int64_t)ncb;
    if (units * nc >= (int64_t(1) << 31)) return false;
    CUtensorMap map;
    if (!encode_slices_map(q, a.x, &map)) return false;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = nc;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(units * nc));
    cfg.blockDim = dim3(kLThreads);
    cfg.dynamicSmemBytes = (size_t)smax * kLRowB + 128;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, a, map, ncb, nc, smax) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return true;
}

// Groups longer than one slice hold part of each CTA's rows in registers.
template <int BITS, bool ASYM>
bool wq_l_dispatch(const QArgs& a, cudaStream_t st) {
    if (std::min(a.q.g, a.q.Tq) > kLRegMinGroup) return wq_l_launch<BITS, ASYM, kLRegWords>(a, st);
    return wq_l_launch<BITS, ASYM, 0>(a, st);
}

}  // namespace

bool cluster_quantize_supported(const QSpec& q)
{
    return q.axis == KVQ_GROUP_ALONG_T && q.x_dt == KVQ_BF16 && q.aligned && q.C % kLCB == 0 && q.Tq > 0 &&
           std::min(q.g, q.Tq) <= kLMaxGroup && q.T < (int64_t(1) << 31) &&
           q.outer * q.ngroups * (q.C / kLCB) < (int64_t(1) << 31);
}

bool cluster_quantize(const QArgs& a, cudaStream_t st)
{
    if (!cluster_quantize_supported(a.q)) return false;
    const bool asym = a.q.mode == KVQ_ASYM;
    switch (a.q.bits) {
    case 8: return asym ? wq_l_dispatch<8, true>(a, st) : wq_l_dispatch<8, false>(a, st);
    case 4: return asym ? wq_l_dispatch<4, true>(a, st) : wq_l_dispatch<4, false>(a, st);
    default: return asym ? wq_l_dispatch<2, true>(a, st) : wq_l_dispatch<2, false>(a, st);
    }
}

}  // namespace kvq
