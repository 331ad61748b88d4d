// append.cu -- strided row copies for the online (streaming) KIVI cache.
//
// Method: "KV cache 压缩：把历史装得更小" §"带残差区的压缩预算，逐项加起来": the
// most recent tokens stay in bf16 while the older ones are quantized in groups;
// with tokens arriving one decode step at a time, a group of K (grouped per
// channel over g tokens) can only be quantized once all its g tokens are
// there, so new tokens are buffered with the residual window and flushed a
// block at a time (kvq_append in api.cu orchestrates; this file moves rows:
// new tokens into the buffer, a flushed block's codes and metadata into the
// store, the kept tokens back to the front of the buffer).
#include <algorithm>

#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kCThreads = 256;

// rows x width bytes from src (pitch spitch) to dst (pitch dpitch); V is the
// access width (16, 4 or 1 bytes), dividing every address, pitch and width.
template <typename V>
__global__ void __launch_bounds__(kCThreads)
copy2d_kernel(unsigned char* dst, uint64_t dpitch, const unsigned char* src, uint64_t spitch, uint64_t width,
              uint64_t rows)
{
    const uint64_t per_row = width / sizeof(V);
    const uint64_t n = per_row * rows;
    for (uint64_t i = (uint64_t)blockIdx.x * kCThreads + threadIdx.x; i < n; i += (uint64_t)gridDim.x * kCThreads) {
        const uint64_t r = i / per_row, k = i - r * per_row;
        reinterpret_cast<V*>(dst + r * dpitch)[k] = reinterpret_cast<const V*>(src + r * spitch)[k];
    }
}

}  // namespace

cudaError_t launch_copy2d(void* dst, uint64_t dpitch, const void* src, uint64_t spitch, uint64_t width,
                          uint64_t rows, cudaStream_t st)
{
    if (width == 0 || rows == 0) return cudaSuccess;
    const uint64_t bits = (uint64_t)(uintptr_t)dst | (uint64_t)(uintptr_t)src | dpitch | spitch | width;
    const uint64_t vw = (bits & 15) == 0 ? 16 : ((bits & 3) == 0 ? 4 : 1);
    const uint64_t n = width / vw * rows;
    const unsigned grid = (unsigned)std::max<uint64_t>(1, std::min<uint64_t>((n + kCThreads - 1) / kCThreads,
                                                                              (uint64_t)sm_count() * 8));
    unsigned char* d = static_cast<unsigned char*>(dst);
    const unsigned char* s = static_cast<const unsigned char*>(src);
    if (vw == 16) copy2d_kernel<uint4><<<grid, kCThreads, 0, st>>>(d, dpitch, s, spitch, width, rows);
    else if (vw == 4) copy2d_kernel<uint32_t><<<grid, kCThreads, 0, st>>>(d, dpitch, s, spitch, width, rows);
    else copy2d_kernel<unsigned char><<<grid, kCThreads, 0, st>>>(d, dpitch, s, spitch, width, rows);
    return cudaGetLastError();
}

}  // namespace kvq
