// append.cu -- strided row copies for the online (streaming) KIVI cache.
//
// Method: "KV cache 压缩：把历史装得更小" §"带残差区的压缩预算，逐项加起来": the
// most recent tokens stay in bf16 while the older ones are quantized in groups;
// with tokens arriving one decode step at a time, a group of K (grouped per
// channel over g tokens) can only be quantized once all its g tokens are
// there, so new tokens are buffered with the residual window and flushed a
// block at a time (kvq_append in api.cu orchestrates; this file moves rows:
// new tokens into the buffer, a flushed block's codes and metadata into the
// store, the kept tokens back to the front of the buffer).  Several copies
// (K's and V's new rows; every cache's codes, metadata and kept rows of a
// flush) go in one launch, one grid row per copy.
#include <algorithm>

#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kCThreads = 256;

struct CopyBatch {
    CopyDesc d[kMaxCopies];
    uint32_t vw[kMaxCopies];     // access width of each copy: 16, 4 or 1 bytes
};

// rows x width bytes from src (pitch spitch) to dst (pitch dpitch) with
// accesses of V, by the blocks of one grid row.
template <typename V>
__device__ __forceinline__ void copy_rows(const CopyDesc& c)
{
    const uint64_t per_row = c.width / sizeof(V);
    const uint64_t n = per_row * c.rows;
    for (uint64_t i = (uint64_t)blockIdx.x * kCThreads + threadIdx.x; i < n; i += (uint64_t)gridDim.x * kCThreads) {
        const uint64_t r = i / per_row, k = i - r * per_row;
        reinterpret_cast<V*>(c.dst + r * c.dpitch)[k] = reinterpret_cast<const V*>(c.src + r * c.spitch)[k];
    }
}

// Grid row y performs copy y of the batch.
__global__ void __launch_bounds__(kCThreads)
copies_kernel(const CopyBatch b)
{
    const CopyDesc& c = b.d[blockIdx.y];
    const uint32_t vw = b.vw[blockIdx.y];
    if (vw == 16) copy_rows<uint4>(c);
    else if (vw == 4) copy_rows<uint32_t>(c);
    else copy_rows<unsigned char>(c);
}

}  // namespace

cudaError_t launch_copies(const CopyDesc* d, int n, cudaStream_t st)
{
    CopyBatch b;
    int m = 0;
    uint64_t most = 0;
    for (int i = 0; i < n && i < kMaxCopies; ++i) {
        if (d[i].width == 0 || d[i].rows == 0) continue;
        const uint64_t bits = (uint64_t)(uintptr_t)d[i].dst | (uint64_t)(uintptr_t)d[i].src | d[i].dpitch |
                              d[i].spitch | d[i].width;
        const uint32_t vw = (bits & 15) == 0 ? 16u : ((bits & 3) == 0 ? 4u : 1u);
        b.d[m] = d[i];
        b.vw[m] = vw;
        most = std::max(most, d[i].width / vw * d[i].rows);
        ++m;
    }
    if (m == 0) return cudaSuccess;
    const unsigned grid = (unsigned)std::max<uint64_t>(1, std::min<uint64_t>((most + kCThreads - 1) / kCThreads,
                                                                              (uint64_t)sm_count() * 8));
    copies_kernel<<<dim3(grid, (unsigned)m), kCThreads, 0, st>>>(b);
    return cudaGetLastError();
}

}  // namespace kvq
