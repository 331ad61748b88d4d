/*
 * kvq.h -- C ABI of the GB300 (sm_103a) KV-cache compression hot path.
 *
 * Everything the path computes runs in hand-written CUDA kernels launched on
 * the caller's stream.  The header needs no CUDA include: a stream is passed
 * as `void*` (a cudaStream_t; NULL is the legacy default stream).
 *
 * Sources, cited by page title and section:
 *  [FtC] "KV Compression 公式到源码对照" (formula-to-source walkthrough):
 *        §1.1 symmetric per-channel quantization, §1.2 asymmetric
 *        per-channel quantization, §1.3 dequantization and error metrics,
 *        §2 compression ratio counting scale/zero-point bytes, §3.1 H2O
 *        cumulative attention score, §3.2 recent window union heavy hitters,
 *        §3.3 SnapKV one-shot selection, §4 token compression ratio.
 *  [KVC] "KV cache 压缩：把历史装得更小":
 *        §"量化：位置都留着，每个数更短" (group-wise x ~ s*(q - z); K grouped
 *        per channel, V per token), §"4 bit 的实际压缩率由分组大小决定"
 *        (payload plus per-group bf16 scale and zero),
 *        §"带残差区的压缩预算，逐项加起来" (the most recent tokens stay in
 *        bf16), §"少存 token：合并，或淘汰" (eviction frees the dropped K/V).
 *
 * Conventions shared by every entry point
 *  - Ownership: every buffer pointer is a DEVICE pointer owned by the caller,
 *    except the small descriptor structs (kvq_shape, kvq_qparams), which are
 *    read on the host during the call and may be freed when it returns.  The
 *    library never allocates, frees or synchronises (the one exception is the
 *    diagnostic kvq_wait_timeouts, which synchronises the device); sizes of
 *    every output and workspace come from the size and workspace queries
 *    (kvq_quantized_sizes, kv_select_workspace, kvq_attend_workspace,
 *    kvq_append_workspace, kvq_mixed_sizes).  Host pointers, where an entry
 *    point takes one, say so in its comment.
 *  - Asynchrony: device work is enqueued on `stream`; outputs are valid once
 *    the stream reaches that point.  Workspace contents are scratch and must
 *    not be shared by calls that may overlap on the GPU.
 *  - Errors: arguments are checked on the host before anything is launched.
 *    A rejected call returns KVQ_EINVAL (or KVQ_EWORKSPACE / KVQ_EUNSUPPORTED)
 *    and has no side effect.  KVQ_ECUDA reports a launch failure.  The text
 *    of the last failure on the calling thread is kvq_last_error().
 *  - Tensors are row-major with the last axis contiguous.  A KV tensor is
 *    viewed as [outer, T, C]: outer = batch*heads (or layers), T tokens,
 *    C channels (head_dim, or heads*head_dim).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVQ_OK = 0,
    KVQ_EINVAL = 1,        /* invalid argument (the pages' ValueError cases) */
    KVQ_ECUDA = 2,         /* a CUDA launch or runtime call failed           */
    KVQ_EUNSUPPORTED = 3,  /* valid, but not implemented                     */
    KVQ_EWORKSPACE = 4     /* workspace missing or smaller than required     */
} kvq_status;

typedef enum { KVQ_F32 = 0, KVQ_BF16 = 1, KVQ_I8 = 2, KVQ_NONE = 3 } kvq_dtype;
typedef enum { KVQ_SYM = 0, KVQ_ASYM = 1 } kvq_mode;
typedef enum {
    KVQ_GROUP_ALONG_T = 0, /* groups of g tokens of one channel ("per channel", K in KIVI) */
    KVQ_GROUP_ALONG_C = 1  /* groups of g channels of one token ("per token", V in KIVI)  */
} kvq_axis;

typedef struct { int64_t outer, T, C; } kvq_shape;

/* Quantized format.  Fields are plain ints so the layout is fixed.
 *  bits        2, 4 or 8.
 *  mode        KVQ_SYM: q = clip(rint(x/s), -qmax, qmax), s = max|x|/qmax
 *              ([FtC] §1.1); qmin is ignored (treated as -qmax).
 *              KVQ_ASYM: s = (max-min)/(qmax-qmin), zp = rint(qmin - min/s),
 *              q = clip(rint(x/s) + zp, qmin, qmax) ([FtC] §1.2).
 *  qmin, qmax  integer code range.  SYM: 1 <= qmax <= 2^(bits-1)-1.
 *              ASYM: qmin < qmax, both in [-2^(bits-1), 2^(bits-1)-1] when
 *              qmin < 0, else in [0, 2^bits - 1].
 *  axis        grouping axis (kvq_axis).
 *  group       g >= 1 elements per group; 0 = the whole axis (all quantized
 *              tokens for ALONG_T, all C channels for ALONG_C).  A shorter
 *              last group gets its own scale.
 *  residual    R >= 0: the last min(R, T) tokens of every [outer] slice are
 *              kept unquantized in the source dtype ([KVC] residual window).
 *  scale_dtype KVQ_F32 or KVQ_BF16.
 *  zero_dtype  KVQ_NONE for SYM; KVQ_I8 (saturating), KVQ_BF16 or KVQ_F32 for
 *              ASYM.
 * Arithmetic: float32 IEEE operations rounded to nearest-even, a true
 * division, abs-max / range floored at the float32 value nearest 1e-8, and the
 * codes computed from the scale and zero point AS STORED (bf16 metadata is
 * rounded first). */
typedef struct {
    int32_t bits;
    int32_t mode;
    int32_t qmin;
    int32_t qmax;
    int32_t axis;
    int64_t group;
    int64_t residual;
    int32_t scale_dtype;
    int32_t zero_dtype;
} kvq_qparams;

/* [FtC] §1.3 error metrics, accumulated in binary64. */
typedef struct { double rmse, max_abs, mean_abs; } kvq_err;

/*
 * Layout of the quantized representation (Tq = T - min(R, T) quantized tokens):
 *  codes   uint8 [outer][Tq][C*bits/8]; element c of a token sits in byte
 *          c*bits/8 at bit (c mod (8/bits))*bits, lowest bits first, holding
 *          (q & (2^bits - 1)).  Codes are signed (two's complement) when
 *          mode is SYM or qmin < 0, else unsigned.  C*bits must be a
 *          multiple of 8.
 *  scale   ALONG_T: [outer][ceil(Tq/g)][C];  ALONG_C: [outer][Tq][ceil(C/g)].
 *  zero    same shape as scale (absent for SYM).
 *  resid   [outer][min(R,T)][C] in the source dtype.
 */

/* Sizes in bytes of every buffer kvq_quantize writes, plus the workspace that
 * kvq_quantize and kvq_error_stats need (one workspace of this size serves
 * both).  [KVC] storage table: payload bits/8 per number plus per-group
 * metadata.  Host only; no CUDA call.  Returns KVQ_EINVAL on a bad format. */
KVQ_API kvq_status kvq_quantized_sizes(const kvq_shape* shape, kvq_dtype x_dtype, const kvq_qparams* p,
                               size_t* codes_B, size_t* scale_B, size_t* zero_B,
                               size_t* resid_B, size_t* workspace_B);

/* Quantize x ([outer, T, C], KVQ_F32 or KVQ_BF16) into codes / scale / zero /
 * resid ([FtC] §1.1, §1.2; [KVC] group-wise form, KIVI axes, residual).
 * zero may be NULL for SYM and resid may be NULL when min(R,T) = 0.
 * workspace may be NULL when kvq_quantized_sizes reported 0. */
KVQ_API kvq_status kvq_quantize(const void* x, kvq_dtype x_dtype, const kvq_shape* shape,
                        const kvq_qparams* p, void* codes, void* scale, void* zero, void* resid,
                        void* workspace, size_t workspace_B, void* stream);

/* x_hat = (q - zp) * s in float32, rounded once to out_dtype (KVQ_F32 or
 * KVQ_BF16) ([FtC] §1.3); the residual tokens are copied back unchanged, so
 * when R > 0 out_dtype must be the dtype the residual was stored in. */
KVQ_API kvq_status kvq_dequantize(const void* codes, const void* scale, const void* zero, const void* resid,
                          const kvq_shape* shape, const kvq_qparams* p,
                          void* out, kvq_dtype out_dtype, void* stream);

/* RMSE, max |x - x_hat| and mean |x - x_hat| over all N = outer*T*C elements
 * ([FtC] §1.3), x_hat being what kvq_dequantize returns in x_dtype (residual
 * tokens contribute zero error).  x_hat never goes to memory.  out_dev is a
 * device pointer to one kvq_err.  N = 0 is KVQ_EINVAL.  The workspace needs
 * no initialisation: the call zeroes the part of it that must start at zero.
 * The sums are combined in a fixed order, so equal inputs give equal bits. */
KVQ_API kvq_status kvq_error_stats(const void* x, kvq_dtype x_dtype, const void* codes, const void* scale,
                           const void* zero, const void* resid, const kvq_shape* shape,
                           const kvq_qparams* p, kvq_err* out_dev,
                           void* workspace, size_t workspace_B, void* stream);

/* [FtC] §2: original bytes / (codes + scale + zero + residual bytes).  Host
 * only.  Returns 0 when the denominator is 0. */
KVQ_API double kvq_compression_ratio(size_t orig_B, size_t codes_B, size_t scale_B, size_t zero_B,
                             size_t resid_B);

/* [FtC] §4: total_tokens / kept_tokens into *out; KVQ_EINVAL unless
 * 0 < kept_tokens <= total_tokens.  Host only. */
KVQ_API kvq_status kvq_token_compression_ratio(int64_t total_tokens, int64_t kept_tokens, double* out);

/* Workspace bytes for kv_h2o_select / kv_snapkv_select on [heads, *, T]. */
KVQ_API kvq_status kv_select_workspace(int64_t heads, int64_t T, size_t* workspace_B);

/* H2O keep set ([FtC] §3.1, §3.2).  hist: float32 [heads][steps][T] attention
 * history.  Per head: score[i] = sum over t = 0..steps-1, in that order, of
 * hist[t][i] (float32 adds); W' = min(window, T); the candidates are
 * [0, T-W'); the k = min(budget-W', T-W') best by (score descending, index
 * ascending) are unioned with the recent window [T-W', T).
 * keep: int32 [heads][min(budget, T)], ascending.  scores: float32
 * [heads][T] or NULL.  budget >= 1, 0 <= window <= budget, steps >= 1,
 * T < 2^31; otherwise KVQ_EINVAL. */
KVQ_API kvq_status kv_h2o_select(const float* hist, int64_t heads, int64_t steps, int64_t T,
                         int64_t budget, int64_t window, int32_t* keep, float* scores,
                         void* workspace, size_t workspace_B, void* stream);

/* SnapKV keep set ([FtC] §3.3): as kv_h2o_select, with the observation score
 * score[i] = (sum of the last obs_window rows, in order) / obs_window.
 * 1 <= obs_window <= steps; steps = obs_window = 1 passes precomputed scores. */
KVQ_API kvq_status kv_snapkv_select(const float* hist, int64_t heads, int64_t steps, int64_t T,
                            int64_t obs_window, int64_t budget, int64_t window, int32_t* keep,
                            float* scores, void* workspace, size_t workspace_B, void* stream);

/* Compaction ([KVC] eviction frees the dropped entries):
 * out[h][j][:] = kv[h][keep[h][j]][:] for j < K, kv [heads][T][D] of dtype
 * (KVQ_F32, KVQ_BF16 or KVQ_I8 element size), keep int32 [heads][K],
 * out [heads][K][D].  0 <= K <= T.  A keep entry outside [0, T) is not
 * dereferenced: its output row is filled with zero bytes. */
KVQ_API kvq_status kv_compact(const void* kv, kvq_dtype dtype, int64_t heads, int64_t T, int64_t D,
                      const int32_t* keep, int64_t K, void* out, void* stream);

/* The same compaction for a key and a value cache that share one keep set
 * (the eviction keeps or drops a token's K and V together), in one launch:
 * out_k = kv_compact(k), out_v = kv_compact(v).  k and v have the same dtype
 * and shape [heads][T][D]; out_k and out_v are [heads][K][D].  Errors as for
 * kv_compact, checked on both tensors before anything is launched. */
KVQ_API kvq_status kv_compact_kv(const void* k, const void* v, kvq_dtype dtype, int64_t heads, int64_t T,
                                 int64_t D, const int32_t* keep, int64_t K, void* out_k, void* out_v,
                                 void* stream);

/* Decode attention over a quantized KV cache, with the dequantization fused
 * into the attention kernel.  [KVC] §"量化：位置都留着，每个数更短": the
 * attention kernel reads the low-bit cache and dequantizes it; §"让 kernel 接住
 * 收益": only a fused dequantization turns the smaller cache into fewer bytes
 * moved; §"K 的误差会改变权重，V 的误差会改变内容": logit_t = q^T k_t / sqrt(d)
 * and y = sum_t a_t v_t with a = softmax(logits).
 *
 * For every KV slice o of the cache (outer = batch * kv_heads) and each of its
 * `group` query heads j (grouped-query attention: query head o*group + j reads
 * KV slice o), with C = head_dim:
 *     y[o][j][:] = sum_t softmax_t( q[o][j][:] . k[o][t][:] / sqrt(C) ) v[o][t][:],
 * over all T tokens, where k and v are the cache rows: s * (code - zero_point)
 * for the quantized tokens t < Tq, in full float precision (nothing is rounded
 * to the cache dtype in between), and the bf16 residual rows for t >= Tq.
 *  - q: [outer][group][C] float32 (device); out: [outer][group][C] float32.
 *  - K: the buffers kvq_quantize wrote for a bf16 key cache of `shape` with
 *    k_params (groups along T, the group a multiple of 32 tokens); V likewise
 *    with v_params (groups along C of 32, 64 or 128 channels).  Both formats
 *    need the same bit width and the same residual length.  Zero-point
 *    pointers are ignored for symmetric formats.
 *  - shape: the caches' [outer, T, C]; supported: C = 128, group 1 .. 8.
 *  - workspace: at least kvq_attend_workspace(shape, group) bytes (the
 *    partial results of the splits of T); no initialisation needed.
 *  - Errors: KVQ_EINVAL (NULL or misaligned buffers, bad shape or group,
 *    formats inconsistent with each other), KVQ_EUNSUPPORTED (a valid
 *    format this kernel does not cover), KVQ_EWORKSPACE. */
KVQ_API kvq_status kvq_attend_workspace(const kvq_shape* shape, int64_t group, size_t* workspace_B);
KVQ_API kvq_status kvq_attend_decode(const float* q, int64_t group, const void* k_codes, const void* k_scale,
                                     const void* k_zero, const void* k_resid, const kvq_qparams* k_params,
                                     const void* v_codes, const void* v_scale, const void* v_zero,
                                     const void* v_resid, const kvq_qparams* v_params, const kvq_shape* shape,
                                     float* out, void* workspace, size_t workspace_B, void* stream);

/* Data-free randomized Hadamard rotation of every row (the C channels of one
 * token) of a [outer, T, C] tensor.  KV-COBRA notes (papernotes.org),
 * "关键设计" item 4: an orthogonal Walsh-Hadamard matrix with fixed random
 * sign flips mixes the coordinates, equalises their variances to the mean
 * variance and makes each coordinate nearly Gaussian before scalar
 * quantization; here without the calibrated projection (no data needed).
 *     forward:  y = (1/sqrt(C)) * H_C * (signs .* x)
 *     inverse:  x = signs .* ((1/sqrt(C)) * H_C * y)
 * H_C is the Sylvester Hadamard matrix (H_1 = [1], H_2n = [[H, H], [H, -H]]),
 * symmetric with H_C * H_C = C * I, so inverse(forward(x)) = x.
 *  - x: [outer, T, C] in x_dtype (F32 or BF16); out: the same shape in
 *    out_dtype (F32 or BF16), rounded once; out may equal x when the dtypes
 *    match (each row is read completely before it is written).
 *  - signs: device int8 [C]; a negative entry flips that channel, any other
 *    value keeps it (+1 / -1 are the intended values).
 *  - C must be a power of two from 32 to 1024 (KVQ_EUNSUPPORTED otherwise).
 *  - Errors: KVQ_EINVAL (NULL or misaligned buffers, bad dtypes), KVQ_ECUDA. */
KVQ_API kvq_status kvq_rotate(const void* x, kvq_dtype x_dtype, const kvq_shape* shape, const int8_t* signs,
                              int inverse, void* out, kvq_dtype out_dtype, void* stream);

/* The rotation above fused into per-token quantization and dequantization
 * (KV-COBRA notes, "关键设计" item 4: the rotation absorbed into the quantize
 * path), one read and one write of the tensor each:
 *  - kvq_rotate_quantize: y = the forward rotation of x rounded to bf16 (what
 *    kvq_rotate writes with out_dtype BF16), quantized with p exactly as
 *    kvq_quantize quantizes y: codes / scale / zero of the first Tq tokens,
 *    and the last min(R, T) tokens of y (rotated) in resid.
 *  - kvq_dequantize_rotate: x_hat of the buffers rounded to bf16 (what
 *    kvq_dequantize writes with out_dtype BF16; resid rows as stored), then the
 *    inverse rotation rounded to bf16 into out.
 * Each equals the two separate calls bit for bit.  The y tensor and x_hat
 * never go to memory.
 *  - x / out: [outer, T, C] bf16 only; groups along C (per token) only, C in
 *    {32, 64, 128, 256} and the group a power of two from 32 to C
 *    (KVQ_EUNSUPPORTED otherwise; other formats: kvq_rotate, then
 *    kvq_quantize).  Buffers are laid out as kvq_quantize lays them out.
 *  - signs: device int8 [C], as for kvq_rotate.
 *  - x / out, codes and resid 16-byte aligned; scale and zero aligned to their
 *    element size.  No workspace.
 *  - Errors: KVQ_EINVAL (NULL or misaligned buffers, a bad format),
 *    KVQ_EUNSUPPORTED, KVQ_ECUDA; nothing is launched on an error. */
KVQ_API kvq_status kvq_rotate_quantize(const void* x, kvq_dtype x_dtype, const kvq_shape* shape, const int8_t* signs,
                                       const kvq_qparams* p, void* codes, void* scale, void* zero, void* resid,
                                       void* stream);
KVQ_API kvq_status kvq_dequantize_rotate(const void* codes, const void* scale, const void* zero, const void* resid,
                                         const kvq_shape* shape, const kvq_qparams* p, const int8_t* signs,
                                         void* out, kvq_dtype out_dtype, void* stream);

/* Online (streaming) quantized cache: append tokens, quantize full blocks.
 * [KVC] §"带残差区的压缩预算，逐项加起来": the most recent tokens stay in bf16 and
 * the older ones are stored quantized in groups; with one token per decode step
 * a key group of g tokens (per channel) can only be quantized once all g have
 * arrived, so arriving tokens are buffered together with the residual window.
 * State, all caller-owned:
 *  - the store: codes / scale / zero laid out exactly as kvq_quantize lays out
 *    a [outer, T_cap, C] tensor quantized with p and no residual
 *    (shape = {outer, T_cap, C}); its first *tq tokens are filled;
 *  - resid: [outer][p->residual + block][C] in x_dtype; its first *nres rows
 *    are the newest tokens, oldest first;
 *  - *tq (a multiple of block) and *nres (< p->residual + block): host counters,
 *    updated by the call.
 * The call copies the n new rows x_new [outer][n][C] into the buffer; each time
 * the buffer reaches p->residual + block rows, its oldest `block` rows are
 * quantized (groups of p->group along T for keys, along C for values) into
 * store tokens [*tq, *tq + block) and leave the buffer.  Appending the T tokens
 * of a sequence in any chunks therefore leaves exactly what kvq_quantize gives
 * for the whole sequence with residual T - *tq, bit for bit.
 *  - block: tokens per flush; groups along T need block to be a multiple of
 *    p->group (> 0).
 *  - workspace: at least kvq_append_workspace bytes.
 *  - Errors: KVQ_EINVAL (bad counters, a store too small for the flushes the
 *    call needs, NULL or misaligned buffers), KVQ_EWORKSPACE; nothing is
 *    launched and the counters are unchanged then.
 *  - Cost: one copy launch per call without a flush; one quantize and one
 *    copy launch per flush; a long prompt is better quantized with
 *    kvq_quantize before appending starts. */
KVQ_API kvq_status kvq_append_workspace(const kvq_shape* shape, kvq_dtype x_dtype, const kvq_qparams* p,
                                        int64_t block, size_t* workspace_B);
KVQ_API kvq_status kvq_append(const void* x_new, int64_t n, kvq_dtype x_dtype, const kvq_shape* shape,
                              const kvq_qparams* p, int64_t block, void* codes, void* scale, void* zero,
                              void* resid, int64_t* tq, int64_t* nres, void* workspace, size_t workspace_B,
                              void* stream);

/* The key and the value cache of one layer appended together, in one call
 * that shares the counters (*tq, *nres): exactly kvq_append on K, then on V,
 * with the same n, block and counters, bit for bit.  Each decode step without a
 * flush is one kernel launch (the new K and V rows copied together); a flush
 * is one quantize per cache and one launch for both caches' codes, metadata
 * and kept rows.
 *  - k_params / v_params: the two formats (keys typically grouped along T,
 *    values along C); their residual windows must be equal (KVQ_EINVAL).
 *  - k_* / v_*: each cache's store and buffer, as for kvq_append.
 *  - workspace: at least kvq_append_kv_workspace bytes (K's part, then V's).
 *  - Errors as kvq_append; nothing is launched and the counters are unchanged
 *    on an error. */
KVQ_API kvq_status kvq_append_kv_workspace(const kvq_shape* shape, kvq_dtype x_dtype, const kvq_qparams* k_params,
                                           const kvq_qparams* v_params, int64_t block, size_t* workspace_B);
KVQ_API kvq_status kvq_append_kv(const void* k_new, const void* v_new, int64_t n, kvq_dtype x_dtype,
                                 const kvq_shape* shape, const kvq_qparams* k_params, const kvq_qparams* v_params,
                                 int64_t block, void* k_codes, void* k_scale, void* k_zero, void* k_resid,
                                 void* v_codes, void* v_scale, void* v_zero, void* v_resid, int64_t* tq,
                                 int64_t* nres, void* workspace, size_t workspace_B, void* stream);

/* Per-token mixed precision.  "大模型KV缓存自适应量化实战" §2.1: every token
 * is stored at one of four levels, 2/4/8/16 bits; §3.1: per-token
 * quantization, symmetric for 2 and 4 bits (qmax 1 and 7), asymmetric for 8
 * bits ([0, 255]), 16 bits stored as is; §3.2: 2-bit precision tags
 * (00/01/10/11 = 2/4/8/16 bits) and same-precision data kept together.  The
 * controller that picks the levels is not part of this library: the caller
 * passes tags[outer][T] (uint8, low 2 bits used).
 * Layout of slice o of a bf16 [outer, T, C] tensor:
 *  - stream: slice o's records start at byte o * T * 2C; token t's record is
 *    at byte off[o][t] of it: the packed codes (as in the uniform formats:
 *    channel c at bit (c mod 8/bits)*bits of byte c*bits/8, two's complement
 *    for the symmetric levels), then the bf16 scale (and for 8 bits the bf16
 *    zero point), or the C bf16 values for 16 bits.  Record bytes: C/4 + 2,
 *    C/2 + 2, C + 4, 2C;
 *  - off[o][0..T] (int64): exclusive prefix sums of the record sizes;
 *    off[o][T] is the number of bytes slice o uses;
 *  - tags2[o][ceil(T/4)]: the 2-bit tags, token t at bit 2*(t%4) of byte t/4.
 * Scales and zero points are rounded to bf16 before the codes are computed,
 * exactly as the uniform quantizer does.
 *  - x, out: bf16; x, out and stream_buf 16-byte aligned, off 8-byte aligned;
 *    C must be 64, 128 or 256 (KVQ_EUNSUPPORTED otherwise).
 *  - Sizes: kvq_mixed_sizes (stream bytes are those of the all-16-bit case;
 *    off[o][T] tells how many a slice really uses).
 *  - Errors: KVQ_EINVAL (NULL or misaligned buffers), KVQ_ECUDA. */
KVQ_API kvq_status kvq_mixed_sizes(const kvq_shape* shape, size_t* stream_B, size_t* off_B, size_t* tags2_B);
KVQ_API kvq_status kvq_mixed_quantize(const void* x, const uint8_t* tags, const kvq_shape* shape, void* stream_buf,
                                      int64_t* off, uint8_t* tags2, void* stream);
KVQ_API kvq_status kvq_mixed_dequantize(const void* stream_buf, const int64_t* off, const uint8_t* tags2,
                                        const kvq_shape* shape, void* out, void* stream);

/* Size of the library's fixed scratch array used by kvq_error_stats_noalloc. */
#define KVQ_NOALLOC_SCRATCH_BYTES (1 << 20)

/* kvq_error_stats without a workspace argument.  The pages have no
 * counterpart to this entry point: it exists for callers that cannot allocate
 * device memory at the moment they need the statistics -- for example a
 * serving loop whose memory pool already owns all device memory, or code that
 * must not call cudaMalloc on its hot path because cudaMalloc may synchronise
 * the device.  It computes exactly what kvq_error_stats computes, with the same
 * arguments minus the workspace, and allocates nothing: the partial sums live
 * in a fixed array of KVQ_NOALLOC_SCRATCH_BYTES (1 MiB) compiled into the
 * library, which every GPU that loads the library keeps until the process
 * exits.
 *  - Limit: shapes whose partial sums need more than that array return
 *    KVQ_EWORKSPACE (with a message) before anything is launched; use
 *    kvq_error_stats with a workspace for them.
 *  - Set-up: the first call on each device looks up the array's device
 *    address (cudaGetSymbolAddress) with that device current; make that first
 *    call before any stream capture.
 *  - Sharing: every call uses the same array and it keeps the previous call's
 *    contents (each call overwrites what it reads).  Calls that may overlap on
 *    the GPU (other streams, other host threads) race on the array: order them
 *    on one stream or synchronise between them. */
KVQ_API kvq_status kvq_error_stats_noalloc(const void* x, kvq_dtype x_dtype, const void* codes,
                                           const void* scale, const void* zero, const void* resid,
                                           const kvq_shape* shape, const kvq_qparams* p, kvq_err* out_dev,
                                           void* stream);

/* Bounded waits that gave up (a diagnostic of this library; no counterpart on
 * the pages).  Every wait of the library's kernels on an asynchronous copy
 * (an mbarrier phase) polls a bounded number of times; a wait that runs out
 * records itself in a device counter and the kernel leaves its loop, so its
 * outputs are undefined.  (The cluster kernels' barriers are hardware cluster
 * barriers that every CTA of the cluster reaches on every path, timeouts
 * included.)  This call synchronises the current device (all streams), then
 * writes to *count the number of such waits on the CURRENT DEVICE since the
 * library was loaded there, over all kernels (each device keeps its own
 * counters; call it once per device to cover several).  0 is the only value
 * a correct run produces.  Host pointer; KVQ_EINVAL if NULL, KVQ_ECUDA if the
 * synchronisation or the read of a counter reports an error (*count is then
 * not written). */
KVQ_API kvq_status kvq_wait_timeouts(uint64_t* count);

/* Message describing the last non-OK status returned on this thread. */
KVQ_API const char* kvq_last_error(void);

/* Library version string. */
KVQ_API const char* kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
