// compact.cu -- compaction gather of the kept K/V rows.
//
// Method ("KV cache 压缩：把历史装得更小", §"少存 token：合并，或淘汰": evicting
// really frees the dropped entries): out[h][j][:] = kv[h][keep[h][j]][:].
//
// Each thread moves one 16-byte piece of a row (a 256-byte bf16 row of
// head_dim 128 is 16 consecutive lanes, so a warp moves two rows with fully
// coalesced 512-byte accesses); rows that are not 16-byte multiples or not
// aligned fall back to element-size pieces.  An index outside [0, T) is never
// dereferenced: that output row is zero-filled.
#include <algorithm>

#include "kvq_device.cuh"

namespace kvq {

namespace {

constexpr int kThreads = 256;

template <typename P>
__global__ void __launch_bounds__(kThreads)
compact_kernel(const P* kv, int64_t T, int64_t pieces_per_row, const int32_t* keep, int64_t K,
               int64_t n_pieces, P* out)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_pieces;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / pieces_per_row;            // h*K + j
        const int64_t piece = i - row * pieces_per_row;
        const int64_t h = row / K;
        const int32_t idx = keep[row];
        P v;
        if (idx >= 0 && idx < T) v = kv[(h * T + idx) * pieces_per_row + piece];
        else memset(&v, 0, sizeof(P));
        out[i] = v;
    }
}

// Rows of 2^LOG_PPR 16-byte pieces (e.g. head_dim 128 bf16 = 16 pieces):
// a warp takes RPW consecutive output rows at a time; lanes 0..RPW-1 read
// the rows' keep entries and source offsets once and broadcast them, then
// every lane issues all its 16-byte loads (of K, and of V when v != nullptr)
// before its stores, so each lane keeps several loads in flight.
template <int LOG_PPR, int RPW>
__global__ void __launch_bounds__(kThreads)
compact_rows_kernel(const uint4* k, const uint4* v, int64_t T, const int32_t* keep, int64_t K, int64_t nrows,
                    uint4* ok, uint4* ov)
{
    constexpr int PPR = 1 << LOG_PPR;
    constexpr int ITEMS = RPW * PPR;
    constexpr int PER_LANE = (ITEMS + 31) / 32;
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r0 = warp0 * RPW; r0 < nrows; r0 += nwarps * RPW) {
        // source row of output row r0 + lane (-1: zero row)
        int64_t src = -1;
        if (lane < RPW && r0 + lane < nrows) {
            const int64_t row = r0 + lane;
            const int32_t idx = keep[row];
            if (idx >= 0 && idx < T) src = (row / K) * T + idx;
        }
        uint4 a[PER_LANE], b[PER_LANE];
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int item = lane + 32 * i;
            const int r = item >> LOG_PPR, piece = item & (PPR - 1);
            const int64_t sr = __shfl_sync(0xFFFFFFFFu, src, r < RPW ? r : 0);
            a[i] = b[i] = make_uint4(0, 0, 0, 0);
            if (item < ITEMS && sr >= 0) {
                a[i] = __ldcs(k + sr * PPR + piece);
                if (v) b[i] = __ldcs(v + sr * PPR + piece);
            }
        }
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) {
            const int item = lane + 32 * i;
            const int64_t row = r0 + (item >> LOG_PPR);
            if (item < ITEMS && row < nrows) {
                ok[row * PPR + (item & (PPR - 1))] = a[i];
                if (v) ov[row * PPR + (item & (PPR - 1))] = b[i];
            }
        }
    }
}

template <int LOG_PPR>
cudaError_t launch_rows(const void* k, const void* v, int64_t heads, int64_t T, const int32_t* keep, int64_t K,
                        void* ok, void* ov, cudaStream_t st)
{
    constexpr int RPW = (128 >> LOG_PPR) > 32 ? 32 : (128 >> LOG_PPR);   // 128 pieces per warp pass
    const int64_t nrows = heads * K;
    const int64_t warps = (nrows + RPW - 1) / RPW;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((warps * 32 + kThreads - 1) / kThreads,
                                                                  (int64_t)sm_count() * 8));
    compact_rows_kernel<LOG_PPR, RPW><<<(unsigned)blocks, kThreads, 0, st>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), T, keep, K, nrows, static_cast<uint4*>(ok),
        static_cast<uint4*>(ov));
    return cudaGetLastError();
}

template <typename P>
cudaError_t launch_as(const void* kv, size_t row_B, int64_t heads, int64_t T, const int32_t* keep,
                      int64_t K, void* out, cudaStream_t st)
{
    const int64_t ppr = (int64_t)(row_B / sizeof(P));
    const int64_t n = heads * K * ppr;
    const int64_t cap = (int64_t)sm_count() * 16;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(cap, (n + kThreads - 1) / kThreads));
    compact_kernel<P><<<(unsigned)grid, kThreads, 0, st>>>(static_cast<const P*>(kv), T, ppr, keep, K, n,
                                                          static_cast<P*>(out));
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_one(const void* kv, size_t elem, int64_t heads, int64_t T, int64_t D,
                       const int32_t* keep, int64_t K, void* out, cudaStream_t st);

cudaError_t launch_compact(const void* kv, size_t elem, int64_t heads, int64_t T, int64_t D,
                           const int32_t* keep, int64_t K, void* out, cudaStream_t st)
{
    return launch_compact_pair(kv, nullptr, elem, heads, T, D, keep, K, out, nullptr, st);
}

cudaError_t launch_compact_pair(const void* k, const void* v, size_t elem, int64_t heads, int64_t T, int64_t D,
                                const int32_t* keep, int64_t K, void* ok, void* ov, cudaStream_t st)
{
    if (heads == 0 || K == 0 || D == 0) return cudaSuccess;
    const size_t row_B = (size_t)D * elem;
    const uintptr_t al2 = (uintptr_t)k | (uintptr_t)ok | (v ? ((uintptr_t)v | (uintptr_t)ov) : 0);
    if (row_B % 16 == 0 && al2 % 16 == 0) {
        switch (row_B / 16) {          // rows of 64 .. 1024 bytes: the batched row kernel
        case 4: return launch_rows<2>(k, v, heads, T, keep, K, ok, ov, st);
        case 8: return launch_rows<3>(k, v, heads, T, keep, K, ok, ov, st);
        case 16: return launch_rows<4>(k, v, heads, T, keep, K, ok, ov, st);
        case 32: return launch_rows<5>(k, v, heads, T, keep, K, ok, ov, st);
        case 64: return launch_rows<6>(k, v, heads, T, keep, K, ok, ov, st);
        default: break;
        }
    }
    cudaError_t e = launch_one(k, elem, heads, T, D, keep, K, ok, st);
    if (e != cudaSuccess || !v) return e;
    return launch_one(v, elem, heads, T, D, keep, K, ov, st);
}

cudaError_t launch_one(const void* kv, size_t elem, int64_t heads, int64_t T, int64_t D,
                       const int32_t* keep, int64_t K, void* out, cudaStream_t st)
{
    const size_t row_B = (size_t)D * elem;
    const uintptr_t al = (uintptr_t)kv | (uintptr_t)out;
    if (row_B % 16 == 0 && al % 16 == 0) return launch_as<uint4>(kv, row_B, heads, T, keep, K, out, st);
    if (row_B % 4 == 0 && al % 4 == 0) return launch_as<uint32_t>(kv, row_B, heads, T, keep, K, out, st);
    if (row_B % 2 == 0 && al % 2 == 0) return launch_as<uint16_t>(kv, row_B, heads, T, keep, K, out, st);
    return launch_as<uint8_t>(kv, row_B, heads, T, keep, K, out, st);
}

}  // namespace kvq
