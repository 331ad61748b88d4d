// noalloc.cu -- kvq_error_stats_noalloc: the error statistics without a
// caller-supplied workspace.
//
// Some callers cannot allocate device memory when they want the statistics:
// a serving loop that has handed every byte of device memory to its own pool
// up front, or code that must not call cudaMalloc on its hot path because
// cudaMalloc can synchronise the whole device.  For them this entry point
// takes its scratch (the per-block partial sums of kvq_error_stats) from a
// fixed array compiled into the library.  The array is a file-scope device
// variable: every GPU that loads the library holds KVQ_NOALLOC_SCRATCH_BYTES
// of it until the process exits.  In host code its name is only a host-side
// stand-in, so its device address is looked up with cudaGetSymbolAddress once
// per device, with that device current, on the first call made on it.
#include <mutex>

#include "kvq_internal.h"

static __device__ __align__(256) unsigned char g_stats_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
kvq_status scratch_on_current_device(void** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        kvq::set_last_error("kvq_error_stats_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
        return KVQ_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        kvq::set_last_error("kvq_error_stats_noalloc: device ordinal %d out of range", dev);
        return KVQ_EUNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress((void**)&ptr, g_stats_scratch);
        if (e != cudaSuccess || !ptr) {
            kvq::set_last_error("kvq_error_stats_noalloc: cudaGetSymbolAddress failed on device %d: %s", dev,
                                cudaGetErrorString(e));
            return KVQ_ECUDA;
        }
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_error_stats_noalloc(const void* x, kvq_dtype x_dtype, const void* codes,
                                              const void* scale, const void* zero, const void* resid,
                                              const kvq_shape* shape, const kvq_qparams* p, kvq_err* out_dev,
                                              void* stream)
{
    void* scratch = nullptr;
    kvq_status s = scratch_on_current_device(&scratch);
    if (s != KVQ_OK) return s;
    // kvq_error_stats validates everything and reports KVQ_EWORKSPACE, before
    // launching anything, when the partial sums would not fit the array.
    s = kvq_error_stats(x, x_dtype, codes, scale, zero, resid, shape, p, out_dev, scratch,
                        (size_t)KVQ_NOALLOC_SCRATCH_BYTES, stream);
    if (s == KVQ_EWORKSPACE)
        kvq::set_last_error("kvq_error_stats_noalloc: this shape needs more partial-sum scratch than the "
                            "library's fixed %d-byte array; call kvq_error_stats with a workspace instead",
                            (int)KVQ_NOALLOC_SCRATCH_BYTES);
    return s;
}
