// api.cu -- the extern "C" entry points declared in include/kvq.h.
//
// Every argument is validated here, on the host, before anything is
// launched; a rejected call has no side effect.  The size queries and the
// ratio helpers never touch the CUDA runtime.
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "kvq_internal.h"

namespace {

thread_local std::string g_last_error;

kvq_status fail(kvq_status s, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

kvq_status cuda_status(cudaError_t e, const char* what)
{
    if (e == cudaSuccess) return KVQ_OK;
    return fail(KVQ_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr int64_t kMaxElems = int64_t(1) << 50;   // keeps every index product in int64

bool mul_ok(int64_t a, int64_t b, int64_t c)
{
    if (a == 0 || b == 0 || c == 0) return true;
    return a <= kMaxElems / b && a * b <= kMaxElems / c;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Typed accesses need natural alignment; workspaces hold 32/64-bit atomics
// and partial sums.  Misaligned buffers are rejected before any launch.
kvq_status need_align(const void* p, size_t a, const char* name)
{
    if (p && a > 1 && ((uintptr_t)p % a) != 0) return fail(KVQ_EINVAL, "%s must be %zu-byte aligned", name, a);
    return KVQ_OK;
}

size_t dtype_bytes(int dt)
{
    switch (dt) {
    case KVQ_F32: return 4;
    case KVQ_BF16: return 2;
    case KVQ_I8: return 1;
    default: return 0;
    }
}

// Validate a format over a shape and derive the kernel-side description.
kvq_status make_spec(const kvq_shape* sh, int x_dt, const kvq_qparams* p, kvq::QSpec& q)
{
    if (!sh || !p) return fail(KVQ_EINVAL, "shape and qparams must not be NULL");
    if (sh->outer < 0 || sh->T < 0 || sh->C < 0) return fail(KVQ_EINVAL, "negative extent");
    if (!mul_ok(sh->outer, sh->T, sh->C)) return fail(KVQ_EINVAL, "tensor too large");
    if (x_dt != KVQ_F32 && x_dt != KVQ_BF16) return fail(KVQ_EINVAL, "source dtype must be F32 or BF16");
    if (p->bits != 2 && p->bits != 4 && p->bits != 8) return fail(KVQ_EINVAL, "bits must be 2, 4 or 8 (got %d)", p->bits);
    if ((sh->C * p->bits) % 8 != 0) return fail(KVQ_EINVAL, "C*bits must be a multiple of 8");
    if (p->axis != KVQ_GROUP_ALONG_T && p->axis != KVQ_GROUP_ALONG_C) return fail(KVQ_EINVAL, "bad axis");
    if (p->group < 0 || p->residual < 0) return fail(KVQ_EINVAL, "group and residual must be >= 0");
    if (p->scale_dtype != KVQ_F32 && p->scale_dtype != KVQ_BF16) return fail(KVQ_EINVAL, "scale dtype must be F32 or BF16");
    const int half = 1 << (p->bits - 1);
    if (p->mode == KVQ_SYM) {
        if (p->qmax < 1 || p->qmax > half - 1) return fail(KVQ_EINVAL, "symmetric qmax must be in [1, %d]", half - 1);
        if (p->zero_dtype != KVQ_NONE) return fail(KVQ_EINVAL, "symmetric formats store no zero point (zero_dtype NONE)");
    } else if (p->mode == KVQ_ASYM) {
        if (p->qmin >= p->qmax) return fail(KVQ_EINVAL, "qmin must be < qmax");
        if (p->qmin < 0) {
            if (p->qmin < -half || p->qmax > half - 1) return fail(KVQ_EINVAL, "signed code range does not fit %d bits", p->bits);
        } else if (p->qmax > (1 << p->bits) - 1) {
            return fail(KVQ_EINVAL, "unsigned code range does not fit %d bits", p->bits);
        }
        if (p->zero_dtype != KVQ_I8 && p->zero_dtype != KVQ_BF16 && p->zero_dtype != KVQ_F32)
            return fail(KVQ_EINVAL, "asymmetric zero dtype must be I8, BF16 or F32");
    } else {
        return fail(KVQ_EINVAL, "bad mode");
    }
    q.outer = sh->outer;
    q.T = sh->T;
    q.C = sh->C;
    q.R = std::min(p->residual, sh->T);
    q.Tq = sh->T - q.R;
    q.g = p->group > 0 ? p->group : (p->axis == KVQ_GROUP_ALONG_T ? q.Tq : q.C);
    if (q.g < 1) q.g = 1;
    q.ngroups = p->axis == KVQ_GROUP_ALONG_T ? (q.Tq + q.g - 1) / q.g : (q.C + q.g - 1) / q.g;
    q.bits = p->bits;
    q.mode = p->mode;
    q.axis = p->axis;
    q.qmax = p->qmax;
    q.qmin = p->mode == KVQ_SYM ? -p->qmax : p->qmin;
    q.x_dt = x_dt;
    q.scale_dt = p->scale_dtype;
    q.zero_dt = p->mode == KVQ_SYM ? KVQ_NONE : p->zero_dtype;
    q.is_signed = (p->mode == KVQ_SYM || p->qmin < 0) ? 1 : 0;
    q.lo = (float)q.qmin;
    q.hi = (float)q.qmax;
    {
        // the group constants divide by this integer; its correctly rounded
        // reciprocal drives the exact fast quotient for ranges 1..255
        const int qr = p->mode == KVQ_SYM ? q.qmax : q.qmax - q.qmin;
        q.inv_qr = (qr >= 1 && qr <= 255) ? 1.0f / (float)qr : 0.0f;
    }
    q.aligned = 1;
    return KVQ_OK;
}

struct Sizes { size_t codes, scale, zero, resid; };

Sizes sizes_of(const kvq::QSpec& q)
{
    Sizes s;
    int64_t ng = 0;
    if (q.outer > 0 && q.Tq > 0 && q.C > 0)
        ng = q.axis == KVQ_GROUP_ALONG_T ? q.outer * q.ngroups * q.C : q.outer * q.Tq * q.ngroups;
    s.codes = (size_t)(q.outer * q.Tq * q.C * q.bits / 8);
    s.scale = (size_t)ng * dtype_bytes(q.scale_dt);
    s.zero = q.mode == KVQ_ASYM ? (size_t)ng * dtype_bytes(q.zero_dt) : 0;
    s.resid = (size_t)(q.outer * q.R * q.C) * dtype_bytes(q.x_dt);
    return s;
}

size_t workspace_of(kvq::QSpec q)
{
    // the launch geometry depends on buffer alignment, unknown here: take the
    // larger of the aligned and unaligned requirements
    q.aligned = 1;
    size_t w = std::max(kvq::quantize_workspace(q), kvq::errstats_workspace(q));
    q.aligned = 0;
    w = std::max(w, std::max(kvq::quantize_workspace(q), kvq::errstats_workspace(q)));
    return w;
}

kvq_status need_ptr(const void* p, size_t bytes, const char* name)
{
    if (bytes > 0 && !p) return fail(KVQ_EINVAL, "%s must not be NULL", name);
    return KVQ_OK;
}

}  // namespace

namespace kvq {

bool along_c_fast_ok(const QSpec& q)
{
    if (!q.aligned || q.C % 8 != 0 || q.g % 8 != 0 || q.C % q.g != 0 || q.g / 8 > 32) return false;
    const int64_t cpr = q.C / 8;
    return (cpr & (cpr - 1)) == 0;
}

bool along_t_fast_ok(const QSpec& q) { return q.aligned && q.C % 8 == 0; }

void set_last_error(const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
}

int sm_count()
{
    static std::atomic<int> cache[128];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 148;
        }
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

cudaError_t ensure_kernel_attrs(const void* fn, int smem_bytes, bool nonportable_cluster, bool max_carveout)
{
    struct Entry { const void* fn; int dev; int smem; bool npc, carve; };
    static std::mutex mu;
    static std::vector<Entry> table;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    Entry* hit = nullptr;
    for (Entry& t : table)
        if (t.fn == fn && t.dev == dev) { hit = &t; break; }
    if (hit && hit->smem >= smem_bytes && (hit->npc || !nonportable_cluster) && (hit->carve || !max_carveout))
        return cudaSuccess;
    const int want = hit ? std::max(hit->smem, smem_bytes) : smem_bytes;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (e == cudaSuccess && nonportable_cluster)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess && max_carveout)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;      // also the thread's last error: the launch path reports it
    if (hit) {
        hit->smem = want;
        hit->npc = hit->npc || nonportable_cluster;
        hit->carve = hit->carve || max_carveout;
    } else {
        table.push_back(Entry{fn, dev, want, nonportable_cluster, max_carveout});
    }
    return cudaSuccess;
}

// Readers of the per-translation-unit bounded-wait counters (kvq_bulk.cuh),
// filled during static initialisation of the library.
std::vector<cudaError_t (*)(unsigned int*)>& wait_counters()
{
    static std::vector<cudaError_t (*)(unsigned int*)> v;
    return v;
}

void register_wait_counter(cudaError_t (*read)(unsigned int*)) { wait_counters().push_back(read); }

}  // namespace kvq

extern "C" {

const char* kvq_last_error(void) { return g_last_error.c_str(); }

const char* kvq_version(void) { return "kvq 0.2.0 (sm_103a)"; }

kvq_status kvq_wait_timeouts(uint64_t* count)
{
    if (!count) return fail(KVQ_EINVAL, "count must not be NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(KVQ_ECUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
    uint64_t n = 0;
    for (auto* read : kvq::wait_counters()) {
        unsigned int v = 0;
        e = read(&v);
        if (e != cudaSuccess) return fail(KVQ_ECUDA, "reading a bounded-wait counter: %s", cudaGetErrorString(e));
        n += v;
    }
    *count = n;
    return KVQ_OK;
}

kvq_status kvq_quantized_sizes(const kvq_shape* shape, kvq_dtype x_dtype, const kvq_qparams* p,
                               size_t* codes_B, size_t* scale_B, size_t* zero_B, size_t* resid_B,
                               size_t* workspace_B)
{
    kvq::QSpec q;
    kvq_status s = make_spec(shape, x_dtype, p, q);
    if (s != KVQ_OK) return s;
    const Sizes z = sizes_of(q);
    if (codes_B) *codes_B = z.codes;
    if (scale_B) *scale_B = z.scale;
    if (zero_B) *zero_B = z.zero;
    if (resid_B) *resid_B = z.resid;
    if (workspace_B) *workspace_B = workspace_of(q);
    return KVQ_OK;
}

kvq_status kvq_quantize(const void* x, kvq_dtype x_dtype, const kvq_shape* shape, const kvq_qparams* p,
                        void* codes, void* scale, void* zero, void* resid, void* workspace,
                        size_t workspace_B, void* stream)
{
    kvq::QSpec q;
    kvq_status s = make_spec(shape, x_dtype, p, q);
    if (s != KVQ_OK) return s;
    const Sizes z = sizes_of(q);
    const size_t xB = (size_t)(q.outer * q.T * q.C) * dtype_bytes(x_dtype);
    if ((s = need_ptr(x, xB, "x")) || (s = need_ptr(codes, z.codes, "codes")) ||
        (s = need_ptr(scale, z.scale, "scale")) || (s = need_ptr(zero, z.zero, "zero")) ||
        (s = need_ptr(resid, z.resid, "resid")))
        return s;
    if ((s = need_align(x, dtype_bytes(x_dtype), "x")) || (s = need_align(resid, dtype_bytes(x_dtype), "resid")) ||
        (s = need_align(scale, dtype_bytes(q.scale_dt), "scale")) ||
        (s = need_align(zero, dtype_bytes(q.zero_dt), "zero")) || (s = need_align(workspace, 16, "workspace")))
        return s;
    q.aligned = aligned16(x) && aligned16(codes) && aligned16(resid) && aligned16(scale) && aligned16(zero);
    const size_t need = kvq::quantize_workspace(q);
    if (need > 0 && (!workspace || workspace_B < need))
        return fail(KVQ_EWORKSPACE, "kvq_quantize needs %zu workspace bytes (got %zu)", need, workspace_B);
    kvq::QArgs a = {x, codes, scale, zero, resid, nullptr, workspace, workspace_B, q};
    return cuda_status(kvq::launch_quantize(a, (cudaStream_t)stream), "kvq_quantize launch");
}

kvq_status kvq_dequantize(const void* codes, const void* scale, const void* zero, const void* resid,
                          const kvq_shape* shape, const kvq_qparams* p, void* out, kvq_dtype out_dtype,
                          void* stream)
{
    kvq::QSpec q;
    kvq_status s = make_spec(shape, out_dtype, p, q);
    if (s != KVQ_OK) return s;
    const Sizes z = sizes_of(q);
    const size_t oB = (size_t)(q.outer * q.T * q.C) * dtype_bytes(out_dtype);
    if ((s = need_ptr(out, oB, "out")) || (s = need_ptr(codes, z.codes, "codes")) ||
        (s = need_ptr(scale, z.scale, "scale")) || (s = need_ptr(zero, z.zero, "zero")) ||
        (s = need_ptr(resid, z.resid, "resid")))
        return s;
    if ((s = need_align(out, dtype_bytes(out_dtype), "out")) || (s = need_align(resid, dtype_bytes(out_dtype), "resid")) ||
        (s = need_align(scale, dtype_bytes(q.scale_dt), "scale")) || (s = need_align(zero, dtype_bytes(q.zero_dt), "zero")))
        return s;
    q.aligned = aligned16(out) && aligned16(codes) && aligned16(resid) && aligned16(scale) && aligned16(zero);
    kvq::QArgs a = {nullptr, const_cast<void*>(codes), const_cast<void*>(scale), const_cast<void*>(zero),
                    const_cast<void*>(resid), out, nullptr, 0, q};
    return cuda_status(kvq::launch_dequantize(a, out_dtype, (cudaStream_t)stream), "kvq_dequantize launch");
}

kvq_status kvq_error_stats(const void* x, kvq_dtype x_dtype, const void* codes, const void* scale,
                           const void* zero, const void* resid, const kvq_shape* shape, const kvq_qparams* p,
                           kvq_err* out_dev, void* workspace, size_t workspace_B, void* stream)
{
    kvq::QSpec q;
    kvq_status s = make_spec(shape, x_dtype, p, q);
    if (s != KVQ_OK) return s;
    if (q.outer * q.T * q.C == 0) return fail(KVQ_EINVAL, "error statistics of an empty tensor are undefined");
    const Sizes z = sizes_of(q);
    const size_t xB = (size_t)(q.outer * q.T * q.C) * dtype_bytes(x_dtype);
    if ((s = need_ptr(x, xB, "x")) || (s = need_ptr(codes, z.codes, "codes")) ||
        (s = need_ptr(scale, z.scale, "scale")) || (s = need_ptr(zero, z.zero, "zero")) ||
        (s = need_ptr(out_dev, 1, "out_dev")))
        return s;
    if ((s = need_align(x, dtype_bytes(x_dtype), "x")) || (s = need_align(scale, dtype_bytes(q.scale_dt), "scale")) ||
        (s = need_align(zero, dtype_bytes(q.zero_dt), "zero")) || (s = need_align(out_dev, 8, "out_dev")) ||
        (s = need_align(workspace, 16, "workspace")))
        return s;
    (void)resid;   // residual tokens are exact by construction: not read
    q.aligned = aligned16(x) && aligned16(codes) && aligned16(scale) && aligned16(zero);
    const size_t need = kvq::errstats_workspace(q);
    if (!workspace || workspace_B < need)
        return fail(KVQ_EWORKSPACE, "kvq_error_stats needs %zu workspace bytes (got %zu)", need, workspace_B);
    kvq::QArgs a = {x, const_cast<void*>(codes), const_cast<void*>(scale), const_cast<void*>(zero),
                    const_cast<void*>(resid), nullptr, workspace, workspace_B, q};
    return cuda_status(kvq::launch_error_stats(a, out_dev, (cudaStream_t)stream), "kvq_error_stats launch");
}

kvq_status kvq_attend_workspace(const kvq_shape* shape, int64_t group, size_t* workspace_B)
{
    if (!shape || !workspace_B) return fail(KVQ_EINVAL, "shape and workspace_B must not be NULL");
    if (shape->outer < 0 || shape->T < 0 || shape->C < 0 || group < 1) return fail(KVQ_EINVAL, "negative extent or group < 1");
    if (!mul_ok(shape->outer, group, std::max<int64_t>(shape->T, 1))) return fail(KVQ_EINVAL, "tensor too large");
    *workspace_B = kvq::attend_workspace(shape->outer, shape->T, group);
    return KVQ_OK;
}

kvq_status kvq_attend_decode(const float* q, int64_t group, const void* k_codes, const void* k_scale,
                             const void* k_zero, const void* k_resid, const kvq_qparams* k_params,
                             const void* v_codes, const void* v_scale, const void* v_zero, const void* v_resid,
                             const kvq_qparams* v_params, const kvq_shape* shape, float* out, void* workspace,
                             size_t workspace_B, void* stream)
{
    kvq::AttendArgs a;
    kvq_status s = make_spec(shape, KVQ_BF16, k_params, a.k);
    if (s != KVQ_OK) return s;
    if ((s = make_spec(shape, KVQ_BF16, v_params, a.v)) != KVQ_OK) return s;
    if (shape->T == 0) return fail(KVQ_EINVAL, "attention over an empty cache is undefined (T = 0)");
    if (group < 1) return fail(KVQ_EINVAL, "group must be >= 1 (got %lld)", (long long)group);
    if (a.k.R != a.v.R) return fail(KVQ_EINVAL, "K and V must keep the same residual window");
    if (shape->C != 128) return fail(KVQ_EUNSUPPORTED, "fused attention supports head_dim 128 (got %lld)", (long long)shape->C);
    if (group != 1 && group != 2 && group != 4 && group != 8)
        return fail(KVQ_EUNSUPPORTED, "fused attention supports 1, 2, 4 or 8 query heads per KV head (got %lld)", (long long)group);
    if (a.k.axis != KVQ_GROUP_ALONG_T || a.v.axis != KVQ_GROUP_ALONG_C)
        return fail(KVQ_EUNSUPPORTED, "fused attention needs K grouped along T (per channel) and V along C (per token)");
    if (a.k.bits != a.v.bits) return fail(KVQ_EUNSUPPORTED, "fused attention needs K and V of the same bit width");
    if (a.k.Tq > 0 && a.k.ngroups > 1 && a.k.g % 32 != 0)
        return fail(KVQ_EUNSUPPORTED, "fused attention needs K groups of a multiple of 32 tokens (got %lld)", (long long)a.k.g);
    if (a.v.g != 32 && a.v.g != 64 && a.v.g != 128)
        return fail(KVQ_EUNSUPPORTED, "fused attention needs V groups of 32, 64 or 128 channels (got %lld)", (long long)a.v.g);
    const Sizes zk = sizes_of(a.k), zv = sizes_of(a.v);
    const size_t qB = (size_t)(shape->outer * group * shape->C) * 4;
    if ((s = need_ptr(q, qB, "q")) || (s = need_ptr(out, qB, "out")) ||
        (s = need_ptr(k_codes, zk.codes, "k_codes")) || (s = need_ptr(k_scale, zk.scale, "k_scale")) ||
        (s = need_ptr(k_zero, zk.zero, "k_zero")) || (s = need_ptr(k_resid, zk.resid, "k_resid")) ||
        (s = need_ptr(v_codes, zv.codes, "v_codes")) || (s = need_ptr(v_scale, zv.scale, "v_scale")) ||
        (s = need_ptr(v_zero, zv.zero, "v_zero")) || (s = need_ptr(v_resid, zv.resid, "v_resid")))
        return s;
    if ((s = need_align(q, 4, "q")) || (s = need_align(out, 4, "out")) || (s = need_align(k_codes, 16, "k_codes")) ||
        (s = need_align(v_codes, 16, "v_codes")) || (s = need_align(k_resid, 16, "k_resid")) ||
        (s = need_align(v_resid, 16, "v_resid")) || (s = need_align(k_scale, dtype_bytes(a.k.scale_dt), "k_scale")) ||
        (s = need_align(v_scale, dtype_bytes(a.v.scale_dt), "v_scale")) ||
        (s = need_align(k_zero, dtype_bytes(a.k.zero_dt), "k_zero")) ||
        (s = need_align(v_zero, dtype_bytes(a.v.zero_dt), "v_zero")) || (s = need_align(workspace, 16, "workspace")))
        return s;
    const size_t need = kvq::attend_workspace(shape->outer, shape->T, group);
    if (need && (!workspace || workspace_B < need))
        return fail(KVQ_EWORKSPACE, "kvq_attend_decode needs %zu workspace bytes (got %zu)", need, workspace_B);
    a.q = q;
    a.group = group;
    a.k_codes = k_codes;
    a.k_scale = k_scale;
    a.k_zero = a.k.mode == KVQ_ASYM ? k_zero : nullptr;
    a.k_resid = k_resid;
    a.v_codes = v_codes;
    a.v_scale = v_scale;
    a.v_zero = a.v.mode == KVQ_ASYM ? v_zero : nullptr;
    a.v_resid = v_resid;
    a.out = out;
    a.ws = workspace;
    return cuda_status(kvq::launch_attend(a, (cudaStream_t)stream), "kvq_attend_decode launch");
}

kvq_status kvq_rotate(const void* x, kvq_dtype x_dtype, const kvq_shape* shape, const int8_t* signs, int inverse,
                      void* out, kvq_dtype out_dtype, void* stream)
{
    if (!shape) return fail(KVQ_EINVAL, "shape must not be NULL");
    if (shape->outer < 0 || shape->T < 0 || shape->C < 0) return fail(KVQ_EINVAL, "negative extent");
    if (!mul_ok(shape->outer, shape->T, shape->C)) return fail(KVQ_EINVAL, "tensor too large");
    if (x_dtype != KVQ_F32 && x_dtype != KVQ_BF16) return fail(KVQ_EINVAL, "x dtype must be F32 or BF16");
    if (out_dtype != KVQ_F32 && out_dtype != KVQ_BF16) return fail(KVQ_EINVAL, "out dtype must be F32 or BF16");
    const int64_t rows = shape->outer * shape->T, C = shape->C;
    if (rows == 0 || C == 0) return KVQ_OK;
    if (C < 32 || C > 1024 || (C & (C - 1)) != 0)
        return fail(KVQ_EUNSUPPORTED, "the rotation needs C a power of two from 32 to 1024 (got %lld)", (long long)C);
    kvq_status s;
    if ((s = need_ptr(x, 1, "x")) || (s = need_ptr(out, 1, "out")) || (s = need_ptr(signs, 1, "signs")))
        return s;
    if (!aligned16(x) || !aligned16(out)) return fail(KVQ_EINVAL, "x and out must be 16-byte aligned");
    return cuda_status(kvq::launch_rotate(x, x_dtype, out, out_dtype, signs, (uint64_t)rows, C, inverse ? 1 : 0,
                                          (cudaStream_t)stream),
                       "kvq_rotate launch");
}

namespace {

// Validation shared by the two fused rotation calls: the format, the shapes
// the fused kernels take, the buffers' presence and alignment.
kvq_status rotq_checks(const kvq_shape* shape, kvq_dtype dt, const kvq_qparams* p, const void* x, const char* xname,
                       const int8_t* signs, const void* codes, const void* scale, const void* zero, const void* resid,
                       kvq::QSpec& q)
{
    kvq_status s = make_spec(shape, dt, p, q);
    if (s != KVQ_OK) return s;
    if (dt != KVQ_BF16) return fail(KVQ_EUNSUPPORTED, "the fused rotation takes bf16 tensors only");
    if (q.outer * q.T == 0) return KVQ_OK;
    if (!kvq::rotq_supported(q))
        return fail(KVQ_EUNSUPPORTED,
                    "the fused rotation needs groups along C, C in {32, 64, 128, 256} and a group of 32..C channels, "
                    "a power of two (got C = %lld, group = %lld, axis %d)", (long long)q.C, (long long)q.g, q.axis);
    const Sizes z = sizes_of(q);
    const size_t xB = (size_t)(q.outer * q.T * q.C) * 2;
    if ((s = need_ptr(x, xB, xname)) || (s = need_ptr(codes, z.codes, "codes")) ||
        (s = need_ptr(scale, z.scale, "scale")) || (s = need_ptr(zero, z.zero, "zero")) ||
        (s = need_ptr(resid, z.resid, "resid")) || (s = need_ptr(signs, 1, "signs")))
        return s;
    if (!aligned16(x) || !aligned16(codes) || (z.resid && !aligned16(resid)))
        return fail(KVQ_EINVAL, "%s, codes and resid must be 16-byte aligned", xname);
    if ((s = need_align(scale, dtype_bytes(q.scale_dt), "scale")) || (s = need_align(zero, dtype_bytes(q.zero_dt), "zero")))
        return s;
    return KVQ_OK;
}

}  // namespace

kvq_status kvq_rotate_quantize(const void* x, kvq_dtype x_dtype, const kvq_shape* shape, const int8_t* signs,
                               const kvq_qparams* p, void* codes, void* scale, void* zero, void* resid, void* stream)
{
    kvq::QSpec q;
    kvq_status s = rotq_checks(shape, x_dtype, p, x, "x", signs, codes, scale, zero, resid, q);
    if (s != KVQ_OK || q.outer * q.T == 0) return s;
    kvq::QArgs a = {x, codes, scale, zero, resid, nullptr, nullptr, 0, q};
    return cuda_status(kvq::launch_rotate_quantize(a, signs, (cudaStream_t)stream), "kvq_rotate_quantize launch");
}

kvq_status kvq_dequantize_rotate(const void* codes, const void* scale, const void* zero, const void* resid,
                                 const kvq_shape* shape, const kvq_qparams* p, const int8_t* signs, void* out,
                                 kvq_dtype out_dtype, void* stream)
{
    kvq::QSpec q;
    kvq_status s = rotq_checks(shape, out_dtype, p, out, "out", signs, codes, scale, zero, resid, q);
    if (s != KVQ_OK || q.outer * q.T == 0) return s;
    kvq::QArgs a = {nullptr, const_cast<void*>(codes), const_cast<void*>(scale), const_cast<void*>(zero),
                    const_cast<void*>(resid), out, nullptr, 0, q};
    return cuda_status(kvq::launch_dequantize_rotate(a, signs, (cudaStream_t)stream), "kvq_dequantize_rotate launch");
}

namespace {

// The store's format and the one flush of the streaming cache: the buffer
// [outer, R + block, C] quantized with residual R, into workspace buffers.
struct AppendPlan {
    kvq::QSpec store, flush;
    Sizes fz;
    size_t off_codes, off_scale, off_zero, off_resid, off_qws, qws, total;
};

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

kvq_status append_plan(const kvq_shape* shape, kvq_dtype x_dtype, const kvq_qparams* p, int64_t block,
                       AppendPlan& P)
{
    if (!shape || !p) return fail(KVQ_EINVAL, "shape and qparams must not be NULL");
    if (p->residual < 0) return fail(KVQ_EINVAL, "residual must be >= 0");
    if (block < 1) return fail(KVQ_EINVAL, "block must be >= 1 (got %lld)", (long long)block);
    kvq_qparams sp = *p;
    sp.residual = 0;
    kvq_status s = make_spec(shape, x_dtype, &sp, P.store);
    if (s != KVQ_OK) return s;
    if (p->axis == KVQ_GROUP_ALONG_T && (p->group <= 0 || block % p->group != 0))
        return fail(KVQ_EINVAL, "groups along T need block (%lld) to be a multiple of the group (%lld > 0)",
                    (long long)block, (long long)p->group);
    const kvq_shape fs = {shape->outer, p->residual + block, shape->C};
    if ((s = make_spec(&fs, x_dtype, p, P.flush)) != KVQ_OK) return s;
    P.fz = sizes_of(P.flush);
    P.qws = kvq::quantize_workspace(P.flush);
    P.off_codes = 0;
    P.off_scale = round256(P.fz.codes);
    P.off_zero = P.off_scale + round256(P.fz.scale);
    P.off_resid = P.off_zero + round256(P.fz.zero);
    P.off_qws = P.off_resid + round256(P.fz.resid);
    P.total = P.off_qws + round256(P.qws);
    return KVQ_OK;
}

}  // namespace

kvq_status kvq_append_workspace(const kvq_shape* shape, kvq_dtype x_dtype, const kvq_qparams* p, int64_t block,
                                size_t* workspace_B)
{
    AppendPlan P;
    kvq_status s = append_plan(shape, x_dtype, p, block, P);
    if (s != KVQ_OK) return s;
    if (!workspace_B) return fail(KVQ_EINVAL, "workspace_B must not be NULL");
    *workspace_B = P.total;
    return KVQ_OK;
}

namespace {

// One cache of a streaming append: its plan and the caller's buffers.
struct AppendCache {
    AppendPlan P;
    const char* src;            // x_new [outer][n][C]
    char *codes, *scale, *zero, *resid, *ws;
    size_t ws_B;
};

// The flushes an append of n rows performs from the buffer fill nres.
int64_t append_flushes(int64_t nres, int64_t n, int64_t R, int64_t cap)
{
    int64_t flushes = 0;
    for (int64_t cur = nres, rem = n; rem > 0;) {
        const int64_t m = std::min(rem, cap - cur);
        cur += m;
        rem -= m;
        if (cur == cap) { ++flushes; cur = R; }
    }
    return flushes;
}

// Counters and the store's room for the flushes.
kvq_status append_counters(const int64_t* tq, const int64_t* nres, int64_t n, int64_t R, int64_t block, int64_t Tcap,
                           int64_t& flushes)
{
    const int64_t cap = R + block;
    if (!tq || !nres) return fail(KVQ_EINVAL, "tq and nres must not be NULL");
    if (n < 0) return fail(KVQ_EINVAL, "n must be >= 0");
    if (*tq < 0 || *tq % block != 0 || *tq > Tcap)
        return fail(KVQ_EINVAL, "tq (%lld) must be a multiple of block in [0, T_cap]", (long long)*tq);
    if (*nres < 0 || *nres >= cap)
        return fail(KVQ_EINVAL, "nres (%lld) must be in [0, residual + block)", (long long)*nres);
    flushes = append_flushes(*nres, n, R, cap);
    if (*tq + flushes * block > Tcap)
        return fail(KVQ_EINVAL, "the store holds %lld tokens: %lld more would be quantized after %lld",
                    (long long)Tcap, (long long)(flushes * block), (long long)*tq);
    return KVQ_OK;
}

// Buffers of one cache: presence, sizes, alignment, workspace.
kvq_status append_buffers(const AppendCache& c, const kvq_shape* shape, kvq_dtype x_dtype, int64_t n, int64_t cap,
                          int64_t flushes, const char* who)
{
    kvq_status s;
    const size_t es = dtype_bytes(x_dtype);
    const int64_t outer = shape->outer, C = shape->C;
    const Sizes sz = sizes_of(c.P.store);
    if ((s = need_ptr(c.src, (size_t)(outer * n * C) * es, "x_new")) ||
        (s = need_ptr(c.resid, (size_t)(outer * cap * C) * es, "resid")) ||
        (flushes && ((s = need_ptr(c.codes, sz.codes, "codes")) || (s = need_ptr(c.scale, sz.scale, "scale")) ||
                     (s = need_ptr(c.zero, sz.zero, "zero")))))
        return s;
    if ((s = need_align(c.src, es, "x_new")) || (s = need_align(c.resid, es, "resid")) ||
        (s = need_align(c.scale, dtype_bytes(c.P.store.scale_dt), "scale")) ||
        (s = need_align(c.zero, dtype_bytes(c.P.store.zero_dt), "zero")) || (s = need_align(c.ws, 256, "workspace")))
        return s;
    if (flushes && (!c.ws || c.ws_B < c.P.total))
        return fail(KVQ_EWORKSPACE, "%s needs %zu workspace bytes (got %zu)", who, c.P.total, c.ws_B);
    return KVQ_OK;
}

// The append itself for nc caches sharing the counters: one copy launch per
// buffer segment (every cache's rows together); per flush one quantize per
// cache and one copy launch for every cache's codes, metadata and kept rows.
kvq_status append_run(AppendCache* cs, int nc, int64_t n, const kvq_shape* shape, kvq_dtype x_dtype, int64_t R,
                      int64_t block, int64_t* tq, int64_t* nres, cudaStream_t st, const char* who)
{
    const size_t es = dtype_bytes(x_dtype);
    const int64_t outer = shape->outer, C = shape->C, cap = R + block, Tcap = shape->T;
    const uint64_t rowx = (uint64_t)C * es;                      // bytes of one token row
    int64_t t = *tq, cur = *nres;
    for (int64_t j = 0; j < n;) {
        const int64_t m = std::min(n - j, cap - cur);
        kvq::CopyDesc d[kvq::kMaxCopies];
        for (int i = 0; i < nc; ++i)
            d[i] = kvq::CopyDesc{cs[i].resid + cur * rowx, cap * rowx, cs[i].src + j * rowx, n * rowx, m * rowx,
                                 (uint64_t)outer};
        cudaError_t e = kvq::launch_copies(d, nc, st);
        if (e != cudaSuccess) return cuda_status(e, who);
        cur += m;
        j += m;
        if (cur < cap) continue;
        // flush: the oldest `block` rows -> store tokens [t, t + block), the newest R rows -> front of the buffer
        int nd = 0;
        for (int i = 0; i < nc; ++i) {
            AppendCache& c = cs[i];
            const AppendPlan& P = c.P;
            kvq::QSpec fq = P.flush;
            fq.aligned = aligned16(c.resid) ? 1 : 0;
            kvq::QArgs a = {c.resid, c.ws + P.off_codes, c.ws + P.off_scale, c.ws + P.off_zero, c.ws + P.off_resid,
                            nullptr, c.ws + P.off_qws, P.qws, fq};
            if ((e = kvq::launch_quantize(a, st)) != cudaSuccess) return cuda_status(e, who);
            const uint64_t rowc = (uint64_t)C * P.store.bits / 8;  // bytes of one token's codes
            const size_t sb = dtype_bytes(P.store.scale_dt), zb = dtype_bytes(P.store.zero_dt);
            uint64_t mrow, mpitch, moff;                            // metadata elements per slice and flush
            if (P.store.axis == KVQ_GROUP_ALONG_T) {
                mrow = (uint64_t)(block / P.store.g) * C;
                mpitch = (uint64_t)P.store.ngroups * C;
                moff = (uint64_t)(t / P.store.g) * C;
            } else {
                mrow = (uint64_t)block * P.store.ngroups;
                mpitch = (uint64_t)Tcap * P.store.ngroups;
                moff = (uint64_t)t * P.store.ngroups;
            }
            d[nd++] = kvq::CopyDesc{c.codes + t * rowc, Tcap * rowc, c.ws + P.off_codes, block * rowc, block * rowc,
                                    (uint64_t)outer};
            d[nd++] = kvq::CopyDesc{c.scale + moff * sb, mpitch * sb, c.ws + P.off_scale, mrow * sb, mrow * sb,
                                    (uint64_t)outer};
            if (P.store.mode == KVQ_ASYM)
                d[nd++] = kvq::CopyDesc{c.zero + moff * zb, mpitch * zb, c.ws + P.off_zero, mrow * zb, mrow * zb,
                                        (uint64_t)outer};
            d[nd++] = kvq::CopyDesc{c.resid, cap * rowx, c.ws + P.off_resid, R * rowx, R * rowx, (uint64_t)outer};
        }
        if ((e = kvq::launch_copies(d, nd, st)) != cudaSuccess) return cuda_status(e, who);
        t += block;
        cur = R;
    }
    *tq = t;
    *nres = cur;
    return KVQ_OK;
}

}  // namespace

kvq_status kvq_append(const void* x_new, int64_t n, kvq_dtype x_dtype, const kvq_shape* shape, const kvq_qparams* p,
                      int64_t block, void* codes, void* scale, void* zero, void* resid, int64_t* tq, int64_t* nres,
                      void* workspace, size_t workspace_B, void* stream)
{
    AppendCache c;
    kvq_status s = append_plan(shape, x_dtype, p, block, c.P);
    if (s != KVQ_OK) return s;
    int64_t flushes = 0;
    if ((s = append_counters(tq, nres, n, p->residual, block, shape->T, flushes)) != KVQ_OK) return s;
    c.src = static_cast<const char*>(x_new);
    c.codes = static_cast<char*>(codes);
    c.scale = static_cast<char*>(scale);
    c.zero = static_cast<char*>(zero);
    c.resid = static_cast<char*>(resid);
    c.ws = static_cast<char*>(workspace);
    c.ws_B = workspace_B;
    if ((s = append_buffers(c, shape, x_dtype, n, p->residual + block, flushes, "kvq_append")) != KVQ_OK) return s;
    return append_run(&c, 1, n, shape, x_dtype, p->residual, block, tq, nres, (cudaStream_t)stream, "kvq_append");
}

kvq_status kvq_append_kv_workspace(const kvq_shape* shape, kvq_dtype x_dtype, const kvq_qparams* k_params,
                                   const kvq_qparams* v_params, int64_t block, size_t* workspace_B)
{
    AppendPlan pk, pv;
    kvq_status s = append_plan(shape, x_dtype, k_params, block, pk);
    if (s == KVQ_OK) s = append_plan(shape, x_dtype, v_params, block, pv);
    if (s != KVQ_OK) return s;
    if (!workspace_B) return fail(KVQ_EINVAL, "workspace_B must not be NULL");
    *workspace_B = pk.total + pv.total;
    return KVQ_OK;
}

kvq_status kvq_append_kv(const void* k_new, const void* v_new, int64_t n, kvq_dtype x_dtype, const kvq_shape* shape,
                         const kvq_qparams* k_params, const kvq_qparams* v_params, int64_t block, void* k_codes,
                         void* k_scale, void* k_zero, void* k_resid, void* v_codes, void* v_scale, void* v_zero,
                         void* v_resid, int64_t* tq, int64_t* nres, void* workspace, size_t workspace_B, void* stream)
{
    AppendCache c[2];
    kvq_status s = append_plan(shape, x_dtype, k_params, block, c[0].P);
    if (s == KVQ_OK) s = append_plan(shape, x_dtype, v_params, block, c[1].P);
    if (s != KVQ_OK) return s;
    if (k_params->residual != v_params->residual)
        return fail(KVQ_EINVAL, "K and V share the counters: their residual windows must match (%lld, %lld)",
                    (long long)k_params->residual, (long long)v_params->residual);
    int64_t flushes = 0;
    if ((s = append_counters(tq, nres, n, k_params->residual, block, shape->T, flushes)) != KVQ_OK) return s;
    const void* src[2] = {k_new, v_new};
    void* bufs[2][4] = {{k_codes, k_scale, k_zero, k_resid}, {v_codes, v_scale, v_zero, v_resid}};
    char* ws = static_cast<char*>(workspace);
    for (int i = 0; i < 2; ++i) {
        c[i].src = static_cast<const char*>(src[i]);
        c[i].codes = static_cast<char*>(bufs[i][0]);
        c[i].scale = static_cast<char*>(bufs[i][1]);
        c[i].zero = static_cast<char*>(bufs[i][2]);
        c[i].resid = static_cast<char*>(bufs[i][3]);
        c[i].ws = ws ? ws + (i ? c[0].P.total : 0) : nullptr;
        c[i].ws_B = i ? (workspace_B > c[0].P.total ? workspace_B - c[0].P.total : 0)
                      : std::min(workspace_B, c[0].P.total);
        if ((s = append_buffers(c[i], shape, x_dtype, n, k_params->residual + block, flushes, "kvq_append_kv")) != KVQ_OK)
            return s;
    }
    return append_run(c, 2, n, shape, x_dtype, k_params->residual, block, tq, nres, (cudaStream_t)stream,
                      "kvq_append_kv");
}

namespace {

kvq_status mixed_shape(const kvq_shape* shape)
{
    if (!shape) return fail(KVQ_EINVAL, "shape must not be NULL");
    if (shape->outer < 0 || shape->T < 0 || shape->C < 0) return fail(KVQ_EINVAL, "negative extent");
    if (!mul_ok(shape->outer, shape->T + 1, std::max<int64_t>(shape->C, 8) * 2)) return fail(KVQ_EINVAL, "tensor too large");
    if (shape->C != 64 && shape->C != 128 && shape->C != 256)
        return fail(KVQ_EUNSUPPORTED, "mixed precision supports C = 64, 128 or 256 (got %lld)", (long long)shape->C);
    return KVQ_OK;
}

// the per-token format of a tag: 2 and 4 bits symmetric, 8 bits asymmetric [0, 255], bf16 metadata
kvq::QSpec mixed_format(int bits, int64_t C)
{
    kvq_qparams p = {};
    p.bits = bits;
    p.mode = bits == 8 ? KVQ_ASYM : KVQ_SYM;
    p.qmin = bits == 8 ? 0 : -((1 << (bits - 1)) - 1);
    p.qmax = bits == 8 ? 255 : (1 << (bits - 1)) - 1;
    p.axis = KVQ_GROUP_ALONG_C;
    p.group = C;
    p.residual = 0;
    p.scale_dtype = KVQ_BF16;
    p.zero_dtype = bits == 8 ? KVQ_BF16 : KVQ_NONE;
    const kvq_shape sh = {1, 1, C};
    kvq::QSpec q;
    make_spec(&sh, KVQ_BF16, &p, q);                               // valid by construction
    return q;
}

}  // namespace

kvq_status kvq_mixed_sizes(const kvq_shape* shape, size_t* stream_B, size_t* off_B, size_t* tags2_B)
{
    kvq_status s = mixed_shape(shape);
    if (s != KVQ_OK) return s;
    if (stream_B) *stream_B = (size_t)(shape->outer * shape->T * shape->C * 2);
    if (off_B) *off_B = (size_t)(shape->outer * (shape->T + 1)) * 8;
    if (tags2_B) *tags2_B = (size_t)(shape->outer * ((shape->T + 3) / 4));
    return KVQ_OK;
}

kvq_status kvq_mixed_quantize(const void* x, const uint8_t* tags, const kvq_shape* shape, void* stream_buf,
                              int64_t* off, uint8_t* tags2, void* stream)
{
    kvq_status s = mixed_shape(shape);
    if (s != KVQ_OK) return s;
    const int64_t n = shape->outer * shape->T;
    if (n == 0) return KVQ_OK;
    if ((s = need_ptr(x, 1, "x")) || (s = need_ptr(tags, 1, "tags")) || (s = need_ptr(stream_buf, 1, "stream_buf")) ||
        (s = need_ptr(off, 1, "off")) || (s = need_ptr(tags2, 1, "tags2")))
        return s;
    if ((s = need_align(x, 2, "x")) || (s = need_align(stream_buf, 2, "stream_buf")) || (s = need_align(off, 8, "off")))
        return s;
    if (!aligned16(x) || !aligned16(stream_buf)) return fail(KVQ_EINVAL, "x and stream_buf must be 16-byte aligned");
    const kvq::QSpec f2 = mixed_format(2, shape->C), f4 = mixed_format(4, shape->C), f8 = mixed_format(8, shape->C);
    return cuda_status(kvq::launch_mixed_quantize(x, tags, shape->outer, shape->T, shape->C, stream_buf, off, tags2,
                                                  f2, f4, f8, (cudaStream_t)stream),
                       "kvq_mixed_quantize launch");
}

kvq_status kvq_mixed_dequantize(const void* stream_buf, const int64_t* off, const uint8_t* tags2,
                                const kvq_shape* shape, void* out, void* stream)
{
    kvq_status s = mixed_shape(shape);
    if (s != KVQ_OK) return s;
    if (shape->outer * shape->T == 0) return KVQ_OK;
    if ((s = need_ptr(stream_buf, 1, "stream_buf")) || (s = need_ptr(off, 1, "off")) ||
        (s = need_ptr(tags2, 1, "tags2")) || (s = need_ptr(out, 1, "out")))
        return s;
    if ((s = need_align(stream_buf, 2, "stream_buf")) || (s = need_align(off, 8, "off")) || (s = need_align(out, 2, "out")))
        return s;
    if (!aligned16(out) || !aligned16(stream_buf)) return fail(KVQ_EINVAL, "out and stream_buf must be 16-byte aligned");
    return cuda_status(kvq::launch_mixed_dequantize(stream_buf, off, tags2, shape->outer, shape->T, shape->C, out,
                                                    (cudaStream_t)stream),
                       "kvq_mixed_dequantize launch");
}

double kvq_compression_ratio(size_t orig_B, size_t codes_B, size_t scale_B, size_t zero_B, size_t resid_B)
{
    const double d = (double)codes_B + (double)scale_B + (double)zero_B + (double)resid_B;
    return d > 0 ? (double)orig_B / d : 0.0;
}

kvq_status kvq_token_compression_ratio(int64_t total_tokens, int64_t kept_tokens, double* out)
{
    if (!out) return fail(KVQ_EINVAL, "out must not be NULL");
    if (total_tokens <= 0 || kept_tokens <= 0 || kept_tokens > total_tokens)
        return fail(KVQ_EINVAL, "require 0 < kept_tokens <= total_tokens");
    *out = (double)total_tokens / (double)kept_tokens;
    return KVQ_OK;
}

kvq_status kv_select_workspace(int64_t heads, int64_t T, size_t* workspace_B)
{
    if (!workspace_B) return fail(KVQ_EINVAL, "workspace_B must not be NULL");
    if (heads < 0 || T < 0 || T > INT32_MAX || !mul_ok(heads, T, 1)) return fail(KVQ_EINVAL, "bad heads / T");
    *workspace_B = kvq::select_workspace(heads, T);
    return KVQ_OK;
}

static kvq_status select_common(const float* hist, int64_t heads, int64_t steps, int64_t T, int64_t obs,
                                bool snap, int64_t budget, int64_t window, int32_t* keep, float* scores,
                                void* workspace, size_t workspace_B, void* stream)
{
    if (heads < 0 || T < 0 || T > INT32_MAX) return fail(KVQ_EINVAL, "bad heads / T");
    if (steps < 1) return fail(KVQ_EINVAL, "steps must be >= 1");
    if (!mul_ok(heads, steps, T)) return fail(KVQ_EINVAL, "history too large");
    if (budget < 1) return fail(KVQ_EINVAL, "budget must be >= 1");
    if (window < 0 || window > budget) return fail(KVQ_EINVAL, "window must be in [0, budget]");
    if (snap && (obs < 1 || obs > steps)) return fail(KVQ_EINVAL, "obs_window must be in [1, steps]");
    kvq_status s;
    const int64_t K = std::min(budget, T);
    if ((s = need_ptr(hist, (size_t)(heads * steps * T), "hist")) || (s = need_ptr(keep, (size_t)(heads * K), "keep")))
        return s;
    if ((s = need_align(hist, 4, "hist")) || (s = need_align(keep, 4, "keep")) || (s = need_align(scores, 4, "scores")) ||
        (s = need_align(workspace, 16, "workspace")))
        return s;
    const size_t need = kvq::select_workspace(heads, T);
    if (heads * T > 0 && (!workspace || workspace_B < need))
        return fail(KVQ_EWORKSPACE, "selection needs %zu workspace bytes (got %zu)", need, workspace_B);
    kvq::SelectArgs a;
    a.hist = hist;
    a.heads = heads;
    a.steps = steps;
    a.T = T;
    a.row0 = snap ? steps - obs : 0;
    a.nrows = snap ? obs : steps;
    a.divide = snap ? 1 : 0;
    a.budget = budget;
    a.window = window;
    a.keep = keep;
    a.scores = scores;
    a.ws = workspace;
    a.ws_B = workspace_B;
    return cuda_status(kvq::launch_select(a, (cudaStream_t)stream), snap ? "kv_snapkv_select launch" : "kv_h2o_select launch");
}

kvq_status kv_h2o_select(const float* hist, int64_t heads, int64_t steps, int64_t T, int64_t budget, int64_t window,
                         int32_t* keep, float* scores, void* workspace, size_t workspace_B, void* stream)
{
    return select_common(hist, heads, steps, T, steps, false, budget, window, keep, scores, workspace, workspace_B, stream);
}

kvq_status kv_snapkv_select(const float* hist, int64_t heads, int64_t steps, int64_t T, int64_t obs_window,
                            int64_t budget, int64_t window, int32_t* keep, float* scores, void* workspace,
                            size_t workspace_B, void* stream)
{
    return select_common(hist, heads, steps, T, obs_window, true, budget, window, keep, scores, workspace,
                         workspace_B, stream);
}

kvq_status kv_compact(const void* kv, kvq_dtype dtype, int64_t heads, int64_t T, int64_t D, const int32_t* keep,
                      int64_t K, void* out, void* stream)
{
    const size_t es = dtype_bytes(dtype);
    if (es == 0) return fail(KVQ_EINVAL, "dtype must be F32, BF16 or I8");
    if (heads < 0 || T < 0 || D < 0 || T > INT32_MAX || !mul_ok(heads, T, D)) return fail(KVQ_EINVAL, "bad extents");
    if (K < 0 || K > T) return fail(KVQ_EINVAL, "require 0 <= K <= T");
    kvq_status s;
    if ((s = need_ptr(kv, (size_t)(heads * T * D), "kv")) || (s = need_ptr(keep, (size_t)(heads * K), "keep")) ||
        (s = need_ptr(out, (size_t)(heads * K * D), "out")))
        return s;
    if ((s = need_align(keep, 4, "keep"))) return s;
    return cuda_status(kvq::launch_compact(kv, es, heads, T, D, keep, K, out, (cudaStream_t)stream), "kv_compact launch");
}

kvq_status kv_compact_kv(const void* k, const void* v, kvq_dtype dtype, int64_t heads, int64_t T, int64_t D,
                         const int32_t* keep, int64_t K, void* out_k, void* out_v, void* stream)
{
    const size_t es = dtype_bytes(dtype);
    if (es == 0) return fail(KVQ_EINVAL, "dtype must be F32, BF16 or I8");
    if (heads < 0 || T < 0 || D < 0 || T > INT32_MAX || !mul_ok(heads, T, D)) return fail(KVQ_EINVAL, "bad extents");
    if (K < 0 || K > T) return fail(KVQ_EINVAL, "require 0 <= K <= T");
    kvq_status s;
    if ((s = need_ptr(k, (size_t)(heads * T * D), "k")) || (s = need_ptr(v, (size_t)(heads * T * D), "v")) ||
        (s = need_ptr(keep, (size_t)(heads * K), "keep")) || (s = need_ptr(out_k, (size_t)(heads * K * D), "out_k")) ||
        (s = need_ptr(out_v, (size_t)(heads * K * D), "out_v")))
        return s;
    if ((s = need_align(keep, 4, "keep"))) return s;
    return cuda_status(kvq::launch_compact_pair(k, v, es, heads, T, D, keep, K, out_k, out_v, (cudaStream_t)stream),
                       "kv_compact_kv launch");
}

}  // extern "C"
