// kvq_internal.h -- internal interface between the C-ABI layer (api.cu) and
// the kernel launchers.  Not installed; callers use include/kvq.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

// Validated, derived description of one quantized format over [outer, T, C].
struct QSpec {
    int64_t outer, T, C;
    int64_t Tq;       // quantized tokens = T - R
    int64_t R;        // residual tokens  = min(residual, T)
    int64_t g;        // effective group length (>= 1)
    int64_t ngroups;  // ALONG_T: ceil(Tq/g) groups per channel; ALONG_C: ceil(C/g) per token
    int32_t bits, mode, axis, qmin, qmax;  // SYM: qmin = -qmax
    int32_t x_dt, scale_dt, zero_dt;
    int32_t is_signed;                      // codes are two's complement
    int32_t aligned;                        // all buffers 16-byte aligned
    float lo, hi;                           // clip range as floats
    float inv_qr;                           // RN(1 / (qmax - qmin)) (asym) or RN(1 / qmax) (sym); 0: not used
};

struct QArgs {
    const void* x;   // source [outer, T, C] (quantize, error stats)
    void* codes;
    void* scale;
    void* zero;
    void* resid;
    void* out;       // dequantize output
    void* ws;        // workspace
    size_t ws_B;
    QSpec q;
};

// ---- quantize / dequantize / error stats (quant.cu, dequant.cu, errstats.cu)
size_t quantize_workspace(const QSpec& q);
size_t errstats_workspace(const QSpec& q);
cudaError_t launch_quantize(const QArgs& a, cudaStream_t st);
cudaError_t launch_dequantize(const QArgs& a, int out_dt, cudaStream_t st);
cudaError_t launch_error_stats(const QArgs& a, kvq_err* out_dev, cudaStream_t st);

// Fast paths need 16-byte aligned buffers and these shapes; the generic
// kernels handle everything else.
bool along_c_fast_ok(const QSpec& q);
bool along_t_fast_ok(const QSpec& q);

// ---- bf16 fast paths (fast.cu): used whenever they support the shape
bool fast_quantize_supported(const QSpec& q);
bool fast_quantize_copies_residual(const QSpec& q);
size_t fast_quantize_workspace(const QSpec& q);
cudaError_t fast_quantize(const QArgs& a, cudaStream_t st);
bool fast_dequant_supported(const QSpec& q, int out_dt);
cudaError_t fast_dequantize(const QArgs& a, cudaStream_t st);
int64_t fast_stats_blocks(const QSpec& q, int sms);   // -1: not supported
cudaError_t fast_error_stats(const QArgs& a, void* partials, cudaStream_t st);

// ---- quantize, groups along T longer than one tile, one thread-block
// cluster per (slice, group, 64 channels) (cluster.cu)
bool cluster_quantize_supported(const QSpec& q);
bool cluster_quantize(const QArgs& a, cudaStream_t st);         // false: not handled

// The driver's cuTensorMapEncodeTiled, looked up once (nullptr: unavailable).
void* tensor_map_encode_fn();

// ---- staged quantize and streaming dequantize / statistics (staged.cu)
bool staged_quantize_supported(const QSpec& q);
bool staged_quantize(const QArgs& a, cudaStream_t st);          // false: not handled
bool stream_dequant_supported(const QSpec& q, int out_dt);
cudaError_t stream_dequantize(const QArgs& a, cudaStream_t st);
int64_t stream_stats_blocks(const QSpec& q, int sms);           // -1: not supported
// done != nullptr: the kernel's last block also writes the final result to
// out_dev (done must be zero at launch and counts the finished blocks).
cudaError_t stream_error_stats(const QArgs& a, void* partials, unsigned int* done, kvq_err* out_dev, cudaStream_t st);

// ---- decode attention over a quantized cache (attend.cu)
struct AttendArgs {
    const float* q;                 // [outer][group][C]
    int64_t group;                  // 1, 2, 4 or 8
    const void *k_codes, *k_scale, *k_zero, *k_resid;
    const void *v_codes, *v_scale, *v_zero, *v_resid;
    QSpec k, v;                     // the two formats over the same [outer, T, C = 128]
    float* out;                     // [outer][group][C]
    void* ws;
};
int64_t attend_splits(int64_t T);
size_t attend_workspace(int64_t outer, int64_t T, int64_t group);
cudaError_t launch_attend(const AttendArgs& a, cudaStream_t st);

// ---- randomized Hadamard rotation of [rows, C] (rotate.cu); C a power of two in [32, 1024]
cudaError_t launch_rotate(const void* x, int x_dt, void* out, int out_dt, const int8_t* signs, uint64_t rows,
                          int64_t C, int inverse, cudaStream_t st);

// ---- the rotation fused into per-token quantize / dequantize (rotq.cu): bf16,
// groups along C, C in {32, 64, 128, 256}, g a power of two in [32, C]
bool rotq_supported(const QSpec& q);
cudaError_t launch_rotate_quantize(const QArgs& a, const int8_t* signs, cudaStream_t st);
cudaError_t launch_dequantize_rotate(const QArgs& a, const int8_t* signs, cudaStream_t st);

// ---- strided row copies (append.cu): rows x width bytes, pitches in bytes;
// up to kMaxCopies independent copies in one launch
struct CopyDesc {
    char* dst;
    uint64_t dpitch;
    const char* src;
    uint64_t spitch, width, rows;
};
constexpr int kMaxCopies = 8;
cudaError_t launch_copies(const CopyDesc* d, int n, cudaStream_t st);

// ---- per-token mixed precision (mixed.cu); tags 0..3 = 2/4/8/16 bits, C in {64, 128, 256}
int64_t mixed_record_bytes(int tag, int64_t C);
cudaError_t launch_mixed_quantize(const void* x, const uint8_t* tags, int64_t outer, int64_t T, int64_t C,
                                  void* stream_buf, int64_t* off, uint8_t* tags2, const QSpec& f2, const QSpec& f4,
                                  const QSpec& f8, cudaStream_t st);
cudaError_t launch_mixed_dequantize(const void* stream_buf, const int64_t* off, const uint8_t* tags2, int64_t outer,
                                    int64_t T, int64_t C, void* out, cudaStream_t st);

// ---- keep-set selection (select.cu) and compaction (compact.cu)
struct SelectArgs {
    const float* hist;
    int64_t heads, steps, T;
    int64_t row0;      // first history row summed
    int64_t nrows;     // rows summed (steps for H2O, obs_window for SnapKV)
    int32_t divide;    // SnapKV: divide the sum by nrows
    int64_t budget, window;
    int32_t* keep;
    float* scores;     // may be the workspace
    void* ws;
    size_t ws_B;
};
size_t select_workspace(int64_t heads, int64_t T);
cudaError_t launch_select(const SelectArgs& a, cudaStream_t st);

cudaError_t launch_compact(const void* kv, size_t elem, int64_t heads, int64_t T, int64_t D,
                           const int32_t* keep, int64_t K, void* out, cudaStream_t st);
// K and V with the same keep set in one launch (v, ov may be nullptr)
cudaError_t launch_compact_pair(const void* k, const void* v, size_t elem, int64_t heads, int64_t T, int64_t D,
                                const int32_t* keep, int64_t K, void* ok, void* ov, cudaStream_t st);

// number of SMs of the current device (cached per device)
int sm_count();

// Raise kernel fn's dynamic shared-memory limit to smem_bytes (and allow
// non-portable cluster sizes, or ask for the largest shared-memory carve-out
// so that several CTAs fit on an SM, when asked) on the current device: once
// per (device, kernel), under a lock, so several host threads and several
// devices in one process are safe.  Returns the error of a failed
// cudaFuncSetAttribute, which also stays the thread's last error.
cudaError_t ensure_kernel_attrs(const void* fn, int smem_bytes, bool nonportable_cluster = false,
                                bool max_carveout = false);

// set the thread's kvq_last_error() message (printf-style)
void set_last_error(const char* fmt, ...);

}  // namespace kvq
