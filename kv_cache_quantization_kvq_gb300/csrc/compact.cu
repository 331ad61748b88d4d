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

cudaError_t launch_compact(const void* kv, size_t elem, int64_t heads, int64_t T, int64_t D,
                           const int32_t* keep, int64_t K, void* out, cudaStream_t st)
{
    if (heads == 0 || K == 0 || D == 0) return cudaSuccess;
    const size_t row_B = (size_t)D * elem;
    const uintptr_t al = (uintptr_t)kv | (uintptr_t)out;
    if (row_B % 16 == 0 && al % 16 == 0) return launch_as<uint4>(kv, row_B, heads, T, keep, K, out, st);
    if (row_B % 4 == 0 && al % 4 == 0) return launch_as<uint32_t>(kv, row_B, heads, T, keep, K, out, st);
    if (row_B % 2 == 0 && al % 2 == 0) return launch_as<uint16_t>(kv, row_B, heads, T, keep, K, out, st);
    return launch_as<uint8_t>(kv, row_B, heads, T, keep, K, out, st);
}

}  // namespace kvq
