// select.cu -- H2O / SnapKV keep-set selection.
//
// Method ("KV Compression 公式到源码对照" §3.1-§3.3):
//   H2O score(i)    = sum over observed steps of a_t(i)   (float32, step order)
//   SnapKV score(i) = (sum of the last w steps of a_t(i)) / w
//   keep = TopK(score over [0, T-W'), B-W') union [T-W', T),  W' = min(W, T),
//   ranked by (score descending, index ascending), written in ascending order.
//
// GPU design (one pass over the history from HBM, the rest from L2):
//   colsum_hist   each thread owns 4 adjacent columns and walks the steps in
//                 order (16-byte streaming loads), writes the scores and a
//                 per-head histogram of the top 12 bits of an
//                 order-preserving key of every candidate score.
//   select_digit  per head: the bin holding the k-th largest key.
//   refine_hist   histogram of the next digit among keys sharing the prefix
//                 (12 bits, then the last 8): after three digits the k-th key
//                 T* is exact, and so is the number of ties `need` to keep.
//   count_chunks  per 1024-column chunk: keys > T* and keys == T*.
//   emit          per chunk: offsets from the preceding chunks' counts, a
//                 block scan for the tie ranks (lowest indices win), a block
//                 scan for output positions; heavy hitters land sorted by
//                 index, followed by the recent window.  No sort is needed:
//                 scanning the kept flags in index order yields sorted output.
#include <algorithm>

#include "kvq_device.cuh"

namespace kvq {

namespace {

constexpr int kThreads = 256;
constexpr int kCols = 4 * kThreads;    // columns per chunk
constexpr int kBins1 = 4096, kBins2 = 4096, kBins3 = 256;

struct SelectLayout {
    size_t scores, hist1, hist2, hist3, state, counts, ccount, done, cand, total;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

SelectLayout layout(int64_t heads, int64_t T)
{
    SelectLayout L;
    const int64_t nchunks = (T + kCols - 1) / kCols;
    size_t off = 0;
    L.scores = off; off = align256(off + (size_t)(heads * T) * 4);
    L.hist1 = off;  off = off + (size_t)heads * kBins1 * 4;
    L.done = off;   off = align256(off + (size_t)heads * 8);           // two counters per head, zeroed with hist1
    L.hist2 = off;  off = align256(off + (size_t)heads * kBins2 * 4);
    L.hist3 = off;  off = align256(off + (size_t)heads * kBins3 * 4);
    L.state = off;  off = align256(off + (size_t)heads * 4 * 4);
    L.counts = off; off = align256(off + (size_t)(heads * nchunks) * 2 * 4);
    L.ccount = off; off = align256(off + (size_t)heads * 4);
    L.cand = off;   off = align256(off + (size_t)(heads * T) * 8);     // room for every key
    L.total = off;
    return L;
}

// candidate key: -0 folded onto +0 so that equal scores tie
__device__ __forceinline__ uint32_t score_key(float s) { return float_key(s == 0.0f ? 0.0f : s); }

// ---------------------------------------------------------------- scores

template <bool VEC, bool HIST>
__global__ void __launch_bounds__(kThreads)
colsum_hist_kernel(const SelectArgs a, int64_t rs, float* scores, uint32_t* hist1)
{
    __shared__ uint32_t sh[HIST ? kBins1 : 1];
    if (HIST) {
        for (int i = threadIdx.x; i < kBins1; i += kThreads) sh[i] = 0;
        __syncthreads();
    }
    const int64_t h = blockIdx.y;
    const int64_t T = a.T;
    const int64_t col0 = (int64_t)blockIdx.x * kCols + threadIdx.x * 4;
    const float* base = a.hist + (h * a.steps + a.row0) * T;
    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int64_t nr = a.nrows;
    if (VEC) {
        if (col0 < T) {
            const float4* p = reinterpret_cast<const float4*>(base + col0);
            const int64_t rstride = T / 4;
            int64_t t = 0;
            for (; t + 8 <= nr; t += 8) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = __ldcs(p + (t + u) * rstride);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    s[0] = __fadd_rn(s[0], v[u].x);
                    s[1] = __fadd_rn(s[1], v[u].y);
                    s[2] = __fadd_rn(s[2], v[u].z);
                    s[3] = __fadd_rn(s[3], v[u].w);
                }
            }
            for (; t < nr; ++t) {
                const float4 v = __ldcs(p + t * rstride);
                s[0] = __fadd_rn(s[0], v.x);
                s[1] = __fadd_rn(s[1], v.y);
                s[2] = __fadd_rn(s[2], v.z);
                s[3] = __fadd_rn(s[3], v.w);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t col = col0 + j;
            if (col < T)
                for (int64_t t = 0; t < nr; ++t) s[j] = __fadd_rn(s[j], base[t * T + col]);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (a.divide) s[j] = __fdiv_rn(s[j], (float)nr);
        const int64_t col = col0 + j;
        if (col < T) {
            if (!VEC) scores[h * T + col] = s[j];
            if (HIST && col < rs) atomicAdd(&sh[score_key(s[j]) >> 20], 1u);
        }
    }
    if (VEC && col0 < T) *reinterpret_cast<float4*>(scores + h * T + col0) = make_float4(s[0], s[1], s[2], s[3]);
    if (HIST) {
        __syncthreads();
        for (int i = threadIdx.x; i < kBins1; i += kThreads)
            if (sh[i]) atomicAdd(&hist1[h * kBins1 + i], sh[i]);
    }
}

// Column sums for the candidate path: the gx CTAs of head h split its columns
// evenly, in 32-column (128-byte) groups, and CTA (bx, h) walks its own range
// in steps of kCols columns.  Equal ranges make the CTAs finish together, and
// contiguous ranges starting at unrelated offsets spread the concurrent
// accesses over the memory channels (CTAs that strided through 4 KB chunks
// whose offsets differ by powers of two measured up to 1.5x slower on some
// GPUs).  Each CTA flushes its shared-memory histogram of candidate keys (top
// 12 bits) once; the last CTA of the head to finish picks the level-1 bin b1
// holding the k-th largest key (state[h] = {b1, keys above b1}).
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
colsum_bin1_kernel(const SelectArgs a, int64_t rs, int64_t k, float* scores, uint32_t* hist1, uint32_t* done,
                   uint32_t* state, uint32_t* ccount, bool want_bin)
{
    __shared__ uint32_t sh[kBins1];
    __shared__ int wsum[kThreads / 32];
    __shared__ bool s_last;
    for (int i = threadIdx.x; i < kBins1; i += kThreads) sh[i] = 0;
    __syncthreads();
    const int64_t h = blockIdx.y;
    const int64_t T = a.T;
    const int64_t nr = a.nrows;
    const float* base = a.hist + (h * a.steps + a.row0) * T;
    const int64_t g32 = (T + 31) / 32;                          // 32-column groups of the head
    const int64_t lo = (int64_t)blockIdx.x * g32 / gridDim.x * 32;
    const int64_t hi = min(T, ((int64_t)blockIdx.x + 1) * g32 / gridDim.x * 32);
    for (int64_t c0 = lo; c0 < hi; c0 += kCols) {
        const int64_t col0 = c0 + threadIdx.x * 4;
        float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (VEC) {
            if (col0 < hi) {
                const float4* p = reinterpret_cast<const float4*>(base + col0);
                const int64_t rstride = T / 4;
                int64_t t = 0;
                for (; t + 8 <= nr; t += 8) {
                    float4 v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) v[u] = __ldcs(p + (t + u) * rstride);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        s[0] = __fadd_rn(s[0], v[u].x);
                        s[1] = __fadd_rn(s[1], v[u].y);
                        s[2] = __fadd_rn(s[2], v[u].z);
                        s[3] = __fadd_rn(s[3], v[u].w);
                    }
                }
                for (; t < nr; ++t) {
                    const float4 v = __ldcs(p + t * rstride);
                    s[0] = __fadd_rn(s[0], v.x);
                    s[1] = __fadd_rn(s[1], v.y);
                    s[2] = __fadd_rn(s[2], v.z);
                    s[3] = __fadd_rn(s[3], v.w);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t col = col0 + j;
                if (col < hi)
                    for (int64_t t = 0; t < nr; ++t) s[j] = __fadd_rn(s[j], base[t * T + col]);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (a.divide) s[j] = __fdiv_rn(s[j], (float)nr);
            const int64_t col = col0 + j;
            if (col < hi) {
                if (!VEC) scores[h * T + col] = s[j];
                if (want_bin && col < rs) atomicAdd(&sh[score_key(s[j]) >> 20], 1u);
            }
        }
        if (VEC && col0 < hi) *reinterpret_cast<float4*>(scores + h * T + col0) = make_float4(s[0], s[1], s[2], s[3]);
    }
    // the selection kernel that follows may be scheduled from here on; it
    // waits for this whole grid (and its memory) before reading anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (!want_bin) return;
    __syncthreads();
    for (int i = threadIdx.x; i < kBins1; i += kThreads)
        if (sh[i]) atomicAdd(&hist1[h * kBins1 + i], sh[i]);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&done[h], 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // last CTA of the head: scan the histogram from the top bin down
    const int bpt = kBins1 / kThreads;              // 16
    const int top = kBins1 - 1 - (int)threadIdx.x * bpt;
    int cnt[kBins1 / kThreads];
    int local = 0;
#pragma unroll
    for (int j = 0; j < kBins1 / kThreads; ++j) { cnt[j] = (int)__ldcg(hist1 + h * kBins1 + top - j); local += cnt[j]; }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    if (w == 0) {
        int y = lane < kThreads / 32 ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < kThreads / 32; o <<= 1) {
            const int z = __shfl_up_sync(0xFFFFFFFFu, y, o);
            if (lane >= o) y += z;
        }
        if (lane < kThreads / 32) wsum[lane] = y;
    }
    __syncthreads();
    const int64_t incl = x + (w > 0 ? wsum[w - 1] : 0);
    const int64_t excl = incl - local;
    if (excl < k && k <= incl) {
        int64_t acc = excl;
#pragma unroll
        for (int j = 0; j < kBins1 / kThreads; ++j) {
            if (acc + cnt[j] >= k) {
                state[h * 4 + 0] = (uint32_t)(top - j);
                state[h * 4 + 1] = (uint32_t)acc;
                break;
            }
            acc += cnt[j];
        }
    }
    if (threadIdx.x == 0) ccount[h] = 0;
}

// ---------------------------------------------------------------- block scans

// exclusive prefix sum over the 256 threads of a block, in thread order
template <int NT>
__device__ __forceinline__ int block_excl_scan_n(int v, int& total)
{
    __shared__ int ws[NT / 32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) ws[w] = x;
    __syncthreads();
    if (w == 0) {
        int y = lane < NT / 32 ? ws[lane] : 0;
#pragma unroll
        for (int o = 1; o < NT / 32; o <<= 1) {
            const int z = __shfl_up_sync(0xFFFFFFFFu, y, o);
            if (lane >= o) y += z;
        }
        if (lane < NT / 32) ws[lane] = y;
    }
    __syncthreads();
    const int incl = x + (w > 0 ? ws[w - 1] : 0);
    total = ws[NT / 32 - 1];
    __syncthreads();
    return incl - v;
}

__device__ __forceinline__ int block_excl_scan(int v, int& total) { return block_excl_scan_n<kThreads>(v, total); }

// ---------------------------------------------------------------- radix select

// State per head: [0] key prefix so far, [1] rank still to find within it.
// Finds, from the top bin down, the bin where the running count reaches r.
__global__ void __launch_bounds__(1024)
select_digit_kernel(const uint32_t* hist, int nbins, int digit_bits, int level, int64_t k,
                    uint32_t* state)
{
    __shared__ int wsum[32];
    __shared__ uint32_t s_prefix;
    __shared__ int64_t s_r;
    const int64_t h = blockIdx.x;
    if (threadIdx.x == 0) {
        s_prefix = level == 1 ? 0u : state[h * 4 + 0];
        s_r = level == 1 ? k : (int64_t)state[h * 4 + 1];
    }
    __syncthreads();
    const uint32_t* hb = hist + h * nbins;
    const int bpt = (nbins + 1023) / 1024;                 // bins per thread (from the top)
    const int top = nbins - 1 - threadIdx.x * bpt;         // this thread's highest bin
    int local = 0;
    for (int j = 0; j < bpt; ++j)
        if (top - j >= 0) local += (int)hb[top - j];
    // inclusive scan in thread order (= descending bins)
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = local;
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[w] = x;
    __syncthreads();
    if (w == 0) {
        int y = wsum[lane];
        for (int o = 1; o < 32; o <<= 1) {
            const int z = __shfl_up_sync(0xFFFFFFFFu, y, o);
            if (lane >= o) y += z;
        }
        wsum[lane] = y;
    }
    __syncthreads();
    const int64_t incl = x + (w > 0 ? wsum[w - 1] : 0);
    const int64_t excl = incl - local;
    const int64_t r = s_r;
    if (excl < r && r <= incl) {
        int64_t acc = excl;
        for (int j = 0; j < bpt; ++j) {
            const int b = top - j;
            if (b < 0) break;
            if (acc + hb[b] >= r) {
                state[h * 4 + 0] = (s_prefix << digit_bits) | (uint32_t)b;
                state[h * 4 + 1] = (uint32_t)(r - acc);
                break;
            }
            acc += hb[b];
        }
    }
}

// Histogram of the next digit among candidate keys matching the prefix.
__global__ void __launch_bounds__(kThreads)
refine_hist_kernel(const float* scores, int64_t T, int64_t rs, const uint32_t* state, int level,
                   uint32_t* hist)
{
    __shared__ uint32_t sh[kBins2];
    const int nbins = level == 2 ? kBins2 : kBins3;
    for (int i = threadIdx.x; i < nbins; i += kThreads) sh[i] = 0;
    __syncthreads();
    const int64_t h = blockIdx.y;
    const uint32_t prefix = state[h * 4 + 0];
    const int64_t col0 = (int64_t)blockIdx.x * kCols + threadIdx.x * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t col = col0 + j;
        if (col < rs) {
            const uint32_t key = score_key(scores[h * T + col]);
            if (level == 2) { if ((key >> 20) == prefix) atomicAdd(&sh[(key >> 8) & 0xFFFu], 1u); }
            else if ((key >> 8) == prefix) atomicAdd(&sh[key & 0xFFu], 1u);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nbins; i += kThreads)
        if (sh[i]) atomicAdd(&hist[h * nbins + i], sh[i]);
}

// Per chunk: candidates with key > T* and key == T*.
__global__ void __launch_bounds__(kThreads)
count_chunks_kernel(const float* scores, int64_t T, int64_t rs, const uint32_t* state, int32_t* counts)
{
    const int64_t h = blockIdx.y;
    const uint32_t kth = state[h * 4 + 0];
    const int64_t col0 = (int64_t)blockIdx.x * kCols + threadIdx.x * 4;
    int gt = 0, eq = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t col = col0 + j;
        if (col < rs) {
            const uint32_t key = score_key(scores[h * T + col]);
            gt += key > kth;
            eq += key == kth;
        }
    }
    int tg, te;
    block_excl_scan(gt, tg);
    block_excl_scan(eq, te);
    if (threadIdx.x == 0) {
        counts[(h * gridDim.x + blockIdx.x) * 2 + 0] = tg;
        counts[(h * gridDim.x + blockIdx.x) * 2 + 1] = te;
    }
}

// mode 0: no heavy hitters (k = 0); 1: every candidate (k = T - W'); 2: threshold.
__global__ void __launch_bounds__(kThreads)
emit_kernel(const float* scores, int64_t T, int64_t rs, int64_t K, int64_t k, int mode,
            const uint32_t* state, const int32_t* counts, int32_t* keep)
{
    __shared__ int64_t s_gt_before, s_eq_before;
    const int64_t h = blockIdx.y;
    const int64_t chunk = blockIdx.x;
    const int64_t col0 = chunk * kCols + threadIdx.x * 4;
    int32_t* kh = keep + h * K;

    // the recent window: [rs, T) lands after the k heavy hitters
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t col = col0 + j;
        if (col >= rs && col < T) kh[k + (col - rs)] = (int32_t)col;
    }
    if (mode == 0) return;
    if (mode == 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t col = col0 + j;
            if (col < rs) kh[col] = (int32_t)col;
        }
        return;
    }
    if (chunk * kCols >= rs) return;                      // no candidates in this chunk (uniform)

    if (threadIdx.x < 32) {
        int64_t g = 0, e = 0;
        for (int64_t c = threadIdx.x; c < chunk; c += 32) {
            g += counts[(h * gridDim.x + c) * 2 + 0];
            e += counts[(h * gridDim.x + c) * 2 + 1];
        }
        for (int o = 16; o > 0; o >>= 1) {
            g += __shfl_xor_sync(0xFFFFFFFFu, g, o);
            e += __shfl_xor_sync(0xFFFFFFFFu, e, o);
        }
        if (threadIdx.x == 0) { s_gt_before = g; s_eq_before = e; }
    }
    __syncthreads();
    const uint32_t kth = state[h * 4 + 0];
    const int64_t need = (int64_t)state[h * 4 + 1];
    uint32_t key[4];
    bool cand[4];
    int eq = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t col = col0 + j;
        cand[j] = col < rs;
        key[j] = cand[j] ? score_key(scores[h * T + col]) : 0u;
        eq += cand[j] && key[j] == kth;
    }
    int tot;
    int64_t tie_rank = s_eq_before + block_excl_scan(eq, tot);
    bool sel[4];
    int nsel = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        sel[j] = false;
        if (cand[j]) {
            if (key[j] > kth) sel[j] = true;
            else if (key[j] == kth) { sel[j] = tie_rank < need; ++tie_rank; }
        }
        nsel += sel[j];
    }
    int64_t pos = s_gt_before + min(s_eq_before, need) + block_excl_scan(nsel, tot);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (sel[j]) {
            if (pos < k) kh[pos] = (int32_t)(col0 + j);   // never past the heavy-hitter slots
            ++pos;
        }
}

// ---------------------------------------------------------------- candidate select
//
// After the level-1 histogram (top 12 key bits, built by colsum_bin1) the
// k-th largest key lies in one bin b1; only keys in bins >= b1 can be kept.
//   colsum_bin1     column sums plus the level-1 histogram; the last CTA of
//                   each head picks b1 and the count of keys above it;
//   gather_kernel   one pass over the scores: candidates (bin >= b1) are
//                   appended to the head's list (one atomic per CTA);
//   finish_kernel   one CTA per head: levels 2 and 3 (12 + 8 bits) over the
//                   candidates of bin b1 give the exact k-th key T* and the
//                   number of ties to keep; the kept indices are marked in a
//                   shared-memory bitmap over [0, T) -- ties in index order --
//                   and written out by a scan of the bitmap, i.e. ascending.
constexpr int kFinThreads = 1024;
constexpr int64_t kBitmapMaxT = int64_t(1) << 19;     // two shared-memory bitmaps of T bits (128 KB)

// CTA (bx, h) takes chunks bx, bx + gridDim.x, ... (kGatherJ at most) of
// head h: all its loads are issued first, then one block scan and one atomic
// reserve the CTA's slots in the head's candidate list.
constexpr int kGatherJ = 4;

__global__ void __launch_bounds__(kThreads)
gather_kernel(const float* scores, int64_t T, int64_t rs, const uint32_t* state, uint32_t* ccount, uint2* cand,
              int64_t cap, bool vec)
{
    __shared__ uint32_t s_base;
    const uint32_t h = blockIdx.y;
    const uint32_t thr = state[h * 4 + 0] << 20;          // lowest key of bin b1
    const float* sh = scores + (uint64_t)h * (uint64_t)T;
    const uint32_t rs32 = (uint32_t)rs;                   // T < 2^31
    uint32_t key[kGatherJ][4];
    uint32_t is_cand = 0;                                 // bit 4*jj + q
    int n = 0;
#pragma unroll
    for (int jj = 0; jj < kGatherJ; ++jj) {
        const uint32_t col0 = (blockIdx.x + jj * gridDim.x) * (uint32_t)kCols + threadIdx.x * 4;
        float v[4];
        if (vec && col0 + 3 < rs32) {
            const float4 f = *reinterpret_cast<const float4*>(sh + col0);
            v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] = col0 + q < rs32 ? sh[col0 + q] : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            key[jj][q] = score_key(v[q]);
            const bool c = col0 + q < rs32 && key[jj][q] >= thr;
            is_cand |= (uint32_t)c << (4 * jj + q);
            n += c;
        }
    }
    int total;
    const int excl = block_excl_scan(n, total);
    if (total == 0) return;                               // uniform
    if (threadIdx.x == 0) s_base = atomicAdd(&ccount[h], (uint32_t)total);
    __syncthreads();
    uint32_t pos = s_base + (uint32_t)excl;
    uint2* out = cand + (uint64_t)h * (uint64_t)cap;
#pragma unroll
    for (int jj = 0; jj < kGatherJ; ++jj) {
        const uint32_t col0 = (blockIdx.x + jj * gridDim.x) * (uint32_t)kCols + threadIdx.x * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (is_cand & (1u << (4 * jj + q))) {
                if (pos < (uint64_t)cap) out[pos] = make_uint2(key[jj][q], col0 + q);
                ++pos;
            }
    }
}

// The bin, counted from the top of hist[0..nbins), where the running count
// reaches r (1 <= r <= sum of hist), and r minus the count of the bins above
// it.  Every one of the kFinThreads threads calls it and gets the result.
__device__ __forceinline__ void rank_bin(const uint32_t* hist, int nbins, uint32_t r, uint32_t& bin, uint32_t& rem)
{
    __shared__ uint32_t s_res[2];
    const int bpt = (nbins + kFinThreads - 1) / kFinThreads;      // 4 at most
    const int top = nbins - 1 - (int)threadIdx.x * bpt;
    uint32_t cnt[4] = {0u, 0u, 0u, 0u};
    int local = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (j < bpt && top - j >= 0) { cnt[j] = hist[top - j]; local += (int)cnt[j]; }
    int total;
    const int excl = block_excl_scan_n<kFinThreads>(local, total);
    if ((uint32_t)excl < r && r <= (uint32_t)(excl + local)) {
        uint32_t acc = (uint32_t)excl;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < bpt && acc + cnt[j] >= r) {
                s_res[0] = (uint32_t)(top - j);
                s_res[1] = r - acc;
                break;
            }
            acc += cnt[j];
        }
    }
    __syncthreads();
    bin = s_res[0];
    rem = s_res[1];
    __syncthreads();
}

// Calls emit(position, index) for the set bits of bm[0..nwords) in index
// order (positions 0, 1, ...).  Every one of the kFinThreads threads calls it.
template <typename F>
__device__ __forceinline__ void scan_bits(const uint32_t* bm, int nwords, F emit)
{
    const int wpt = (nwords + kFinThreads - 1) / kFinThreads;
    const int w0 = (int)threadIdx.x * wpt;
    int local = 0;
    for (int j = 0; j < wpt; ++j)
        if (w0 + j < nwords) local += __popc(bm[w0 + j]);
    int total;
    int pos = block_excl_scan_n<kFinThreads>(local, total);
    for (int j = 0; j < wpt; ++j) {
        if (w0 + j >= nwords) break;
        uint32_t w = bm[w0 + j];
        while (w) {
            const int bit = __ffs(w) - 1;
            w &= w - 1;
            emit(pos, (w0 + j) * 32 + bit);
            ++pos;
        }
    }
}

// The keep set of head h from its candidate list (kFinThreads threads).
// Kept: every candidate above bin b1, plus the best `need` of bin b1 by (key
// desc, index asc).  Radix levels 2 (12 bits) and 3 (8 bits) among the
// members of bin b1 give the exact k-th key and how many of its ties to
// keep; the ties are taken in index order; a scan of the kept bitmap writes
// the indices ascending, then the recent window follows.
__device__ __forceinline__ void finish_head(int64_t h, int64_t T, int64_t rs, int64_t k, int64_t K,
                                            const uint32_t* state, int64_t m, const uint2* ch, int32_t* keep,
                                            int64_t cache_cap)
{
    // dynamic: kept bitmap and tie bitmap (ceil(T/32) words each), then a
    // copy of the head's candidates when there are at most cache_cap of them
    extern __shared__ uint32_t bitmap[];
    __shared__ uint32_t hist[kBins2];
    const uint32_t b1 = __ldcg(&state[h * 4 + 0]);
    const int64_t above = (int64_t)__ldcg(&state[h * 4 + 1]);
    const int nwords = (int)((T + 31) / 32);
    uint32_t* ties = bitmap + nwords;
    if (m <= cache_cap) {                 // the passes below read the candidates: keep them on chip
        uint2* cs = reinterpret_cast<uint2*>(bitmap + 2 * nwords);
        for (int64_t i = threadIdx.x; i < m; i += kFinThreads) cs[i] = __ldcg(&ch[i]);
        ch = cs;
    }
    for (int i = threadIdx.x; i < nwords; i += kFinThreads) { bitmap[i] = 0; ties[i] = 0; }
    for (int b = threadIdx.x; b < kBins2; b += kFinThreads) hist[b] = 0;
    __syncthreads();
    const uint32_t need = (uint32_t)(k - above);            // >= 1: bin b1 holds the k-th key

    // level 2 among the members of bin b1
    for (int64_t i = threadIdx.x; i < m; i += kFinThreads) {
        const uint32_t key = ch[i].x;
        if ((key >> 20) == b1) atomicAdd(&hist[(key >> 8) & 0xFFFu], 1u);
    }
    __syncthreads();
    uint32_t b2, rem2;
    rank_bin(hist, kBins2, need, b2, rem2);
    const uint32_t pre = (b1 << 12) | b2;
    const uint32_t in_b2 = hist[b2];
    // kept: keys > kth, and tneed of the nties keys equal to kth (lowest indices)
    uint32_t kth, tneed, nties;
    __syncthreads();                                          // every thread has read hist[b2]
    if (in_b2 == rem2 && pre != 0u) {
        // the whole sub-bin is kept: the boundary lies just below it
        kth = (pre << 8) - 1u;
        tneed = nties = 0u;
    } else {
        // level 3 among the keys with that 24-bit prefix
        for (int b = threadIdx.x; b < kBins3; b += kFinThreads) hist[b] = 0;
        __syncthreads();
        for (int64_t i = threadIdx.x; i < m; i += kFinThreads) {
            const uint32_t key = ch[i].x;
            if ((key >> 8) == pre) atomicAdd(&hist[key & 0xFFu], 1u);
        }
        __syncthreads();
        uint32_t b3;
        rank_bin(hist, kBins3, rem2, b3, tneed);
        kth = (pre << 8) | b3;                                // the exact k-th key
        nties = hist[b3];
    }
    const bool all_ties = tneed == nties;                    // every tie is kept: no index pass

    for (int64_t i = threadIdx.x; i < m; i += kFinThreads) {
        const uint2 c = ch[i];
        if (c.x > kth || (all_ties && c.x == kth)) atomicOr(&bitmap[c.y >> 5], 1u << (c.y & 31));
        else if (c.x == kth) atomicOr(&ties[c.y >> 5], 1u << (c.y & 31));
    }
    __syncthreads();
    if (!all_ties) {
        scan_bits(ties, nwords, [&](int p, int idx) {
            if ((uint32_t)p < tneed) atomicOr(&bitmap[idx >> 5], 1u << (idx & 31));
        });
        __syncthreads();
    }
    int32_t* kh = keep + h * K;
    scan_bits(bitmap, nwords, [&](int p, int idx) {
        if (p < k) kh[p] = idx;
    });
    // the recent window follows the heavy hitters
    for (int64_t i = rs + threadIdx.x; i < T; i += kFinThreads) kh[k + (i - rs)] = (int32_t)i;
}

__global__ void __launch_bounds__(kFinThreads)
finish_kernel(int64_t T, int64_t rs, int64_t k, int64_t K, const uint32_t* state, const uint32_t* ccount,
              const uint2* cand, int64_t cap, int32_t* keep, int64_t cache_cap)
{
    const int64_t h = blockIdx.x;
    finish_head(h, T, rs, k, K, state, min((int64_t)ccount[h], cap), cand + h * cap, keep, cache_cap);
}

// Gather and finish in one launch: kGFParts CTAs per head (kFinThreads
// threads each) gather the candidates of a quarter of the head's scores --
// all loads issued first, keys kept in registers, one block scan and one
// atomic per CTA -- and the last CTA of the head to finish (done2[h], zeroed
// before the column sums) builds the head's keep set from the list.
constexpr int kGFParts = 4;
constexpr int kGFMaxJ = 8;                // 4-column groups per thread at most: rs <= 4 * 8 * 4 * kFinThreads

__global__ void __launch_bounds__(kFinThreads, 1)
gather_finish_kernel(const float* scores, int64_t T, int64_t rs, int64_t k, int64_t K, const uint32_t* state,
                     uint32_t* ccount, uint32_t* done2, uint2* cand, int64_t cap, int32_t* keep, int64_t cache_cap,
                     int jpt)
{
    __shared__ uint32_t s_base;
    __shared__ bool s_last;
    // launched as a programmatic dependent of the column sums: nothing is read
    // before that grid has completed and its writes are visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t h = blockIdx.y;
    const uint32_t thr = __ldcg(&state[h * 4 + 0]) << 20;       // lowest key of bin b1
    const float* sh = scores + (uint64_t)h * (uint64_t)T;
    const uint32_t rs32 = (uint32_t)rs;
    const uint32_t span = (uint32_t)jpt * 4u * kFinThreads;       // columns per part
    const uint32_t base = blockIdx.x * span + threadIdx.x * 4u;
    uint32_t key[kGFMaxJ][4];
    uint32_t is_cand = 0;                                         // bit 4*j + q
    int n = 0;
#pragma unroll
    for (int j = 0; j < kGFMaxJ; ++j) {
        if (j < jpt) {
            const uint32_t col0 = base + (uint32_t)j * 4u * kFinThreads;
            float v[4];
            if (col0 + 3 < rs32) {
                const float4 f = __ldcg(reinterpret_cast<const float4*>(sh + col0));
                v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) v[q] = col0 + q < rs32 ? __ldcg(sh + col0 + q) : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                key[j][q] = score_key(v[q]);
                const bool c = col0 + q < rs32 && key[j][q] >= thr;
                is_cand |= (uint32_t)c << (4 * j + q);
                n += c;
            }
        }
    }
    int total;
    const int excl = block_excl_scan_n<kFinThreads>(n, total);
    if (threadIdx.x == 0) s_base = total ? atomicAdd(&ccount[h], (uint32_t)total) : 0u;
    __syncthreads();
    uint32_t pos = s_base + (uint32_t)excl;
    uint2* out = cand + (uint64_t)h * (uint64_t)cap;
#pragma unroll
    for (int j = 0; j < kGFMaxJ; ++j) {
        if (is_cand & (0xFu << (4 * j))) {
            const uint32_t col0 = base + (uint32_t)j * 4u * kFinThreads;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (is_cand & (1u << (4 * j + q))) {
                    if (pos < (uint64_t)cap) out[pos] = make_uint2(key[j][q], col0 + q);
                    ++pos;
                }
        }
    }
    // the last part of the head builds the keep set
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&done2[h], 1u) == kGFParts - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int64_t m = min((int64_t)__ldcg(&ccount[h]), cap);
    finish_head(h, T, rs, k, K, state, m, out, keep, cache_cap);
}

}  // namespace

size_t select_workspace(int64_t heads, int64_t T) { return layout(heads, T).total; }

cudaError_t launch_select(const SelectArgs& a, cudaStream_t st)
{
    const int64_t H = a.heads, T = a.T;
    if (H == 0 || T == 0) return cudaSuccess;
    const SelectLayout L = layout(H, T);
    char* ws = static_cast<char*>(a.ws);
    float* scores = a.scores ? a.scores : reinterpret_cast<float*>(ws + L.scores);
    uint32_t* hist1 = reinterpret_cast<uint32_t*>(ws + L.hist1);
    uint32_t* hist2 = reinterpret_cast<uint32_t*>(ws + L.hist2);
    uint32_t* hist3 = reinterpret_cast<uint32_t*>(ws + L.hist3);
    uint32_t* state = reinterpret_cast<uint32_t*>(ws + L.state);
    int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);

    const int64_t Wr = std::min(a.window, T);
    const int64_t rs = T - Wr;
    const int64_t k = std::min(a.budget - Wr, rs);
    const int64_t K = std::min(a.budget, T);
    const int mode = k == 0 ? 0 : (k == rs ? 1 : 2);
    const int64_t nchunks = (T + kCols - 1) / kCols;
    const dim3 grid((unsigned)nchunks, (unsigned)H);

    const bool vec = (T % 4 == 0) && ((uintptr_t)a.hist % 16 == 0) && ((uintptr_t)scores % 16 == 0);
    // candidates path: level-1 histogram and bin in the column sum, then gather + finish
    if (T <= kBitmapMaxT) {
        uint32_t* ccount = reinterpret_cast<uint32_t*>(ws + L.ccount);
        uint32_t* done = reinterpret_cast<uint32_t*>(ws + L.done);
        uint2* cand = reinterpret_cast<uint2*>(ws + L.cand);
        const bool want_bin = mode == 2;
        if (want_bin) {       // hist1 and the per-head completion counters are adjacent
            cudaError_t e = cudaMemsetAsync(ws + L.hist1, 0, L.done + (size_t)H * 8 - L.hist1, st);
            if (e != cudaSuccess) return e;
        }
        // six CTAs per SM in one wave (at most six are resident: 40 registers,
        // 16 KB of shared memory), measured 2 % faster than four
        const int64_t per_head = std::max<int64_t>(1, std::min<int64_t>(nchunks, ((int64_t)sm_count() * 6) / H));
        const dim3 cgrid((unsigned)per_head, (unsigned)H);
        if (vec) colsum_bin1_kernel<true><<<cgrid, kThreads, 0, st>>>(a, rs, k, scores, hist1, done, state, ccount, want_bin);
        else colsum_bin1_kernel<false><<<cgrid, kThreads, 0, st>>>(a, rs, k, scores, hist1, done, state, ccount, want_bin);
        if (mode == 2) {
            const size_t bits_B = (size_t)2 * ((T + 31) / 32) * 4;
            constexpr size_t kFinDynMax = 190 * 1024;     // + ~25 KB static stays under 227 KB
            const int64_t cache_cap = std::min<int64_t>(T, (int64_t)((kFinDynMax - bits_B) / 8));
            const size_t smem = bits_B + (size_t)cache_cap * 8;
            const int64_t per_part = (rs + kGFParts - 1) / kGFParts;
            const int jpt = (int)std::max<int64_t>(1, (per_part + 4 * kFinThreads - 1) / (4 * kFinThreads));
            if (jpt <= kGFMaxJ && vec && T >= 4) {
                cudaError_t ea = ensure_kernel_attrs(reinterpret_cast<const void*>(gather_finish_kernel), (int)smem);
                if (ea != cudaSuccess) return ea;
                // programmatic dependent launch: its launch overlaps the column sums' tail
                cudaLaunchConfig_t cfg = {};
                cudaLaunchAttribute at[1];
                at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                at[0].val.programmaticStreamSerializationAllowed = 1;
                cfg.gridDim = dim3(kGFParts, (unsigned)H);
                cfg.blockDim = dim3(kFinThreads);
                cfg.dynamicSmemBytes = smem;
                cfg.stream = st;
                cfg.attrs = at;
                cfg.numAttrs = 1;
                cudaError_t el = cudaLaunchKernelEx(&cfg, gather_finish_kernel, (const float*)scores, T, rs, k, K,
                                                    (const uint32_t*)state, ccount, done + H, cand, (int64_t)T, a.keep,
                                                    cache_cap, jpt);
                if (el != cudaSuccess) return el;
            } else {
                const int64_t rchunks = (rs + kCols - 1) / kCols;
                const dim3 ggrid((unsigned)std::max<int64_t>(1, (rchunks + kGatherJ - 1) / kGatherJ), (unsigned)H);
                gather_kernel<<<ggrid, kThreads, 0, st>>>(scores, T, rs, state, ccount, cand, T, vec);
                // static + dynamic may exceed the 48 KB default
                cudaError_t ea = ensure_kernel_attrs(reinterpret_cast<const void*>(finish_kernel), (int)smem);
                if (ea != cudaSuccess) return ea;
                finish_kernel<<<(unsigned)H, kFinThreads, smem, st>>>(T, rs, k, K, state, ccount, cand, T, a.keep,
                                                                      cache_cap);
            }
        } else {
            emit_kernel<<<grid, kThreads, 0, st>>>(scores, T, rs, K, k, mode, state, counts, a.keep);
        }
        return cudaGetLastError();
    }
    cudaError_t e = cudaMemsetAsync(ws + L.hist1, 0, L.counts - L.hist1, st);
    if (e != cudaSuccess) return e;
    if (vec) colsum_hist_kernel<true, true><<<grid, kThreads, 0, st>>>(a, rs, scores, hist1);
    else colsum_hist_kernel<false, true><<<grid, kThreads, 0, st>>>(a, rs, scores, hist1);
    if (mode == 2) {
        select_digit_kernel<<<(unsigned)H, 1024, 0, st>>>(hist1, kBins1, 12, 1, k, state);
        refine_hist_kernel<<<grid, kThreads, 0, st>>>(scores, T, rs, state, 2, hist2);
        select_digit_kernel<<<(unsigned)H, 1024, 0, st>>>(hist2, kBins2, 12, 2, k, state);
        refine_hist_kernel<<<grid, kThreads, 0, st>>>(scores, T, rs, state, 3, hist3);
        select_digit_kernel<<<(unsigned)H, 1024, 0, st>>>(hist3, kBins3, 8, 3, k, state);
        count_chunks_kernel<<<grid, kThreads, 0, st>>>(scores, T, rs, state, counts);
    }
    emit_kernel<<<grid, kThreads, 0, st>>>(scores, T, rs, K, k, mode, state, counts, a.keep);
    return cudaGetLastError();
}

}  // namespace kvq
