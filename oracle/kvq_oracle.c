/*
 * kvq_oracle.c -- plain, slow, scalar CPU oracle for the KV-cache compression
 * hot path (quantize, dequantize, error statistics, H2O / SnapKV keep-set
 * selection, compaction).
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the smoke check and the
 * benchmark's CPU-baseline leg are the only users of this file.  The CUDA
 * library never links or calls it, and the two share no code, header, table or
 * constant: every definition below is local to this translation unit.
 *
 * Arithmetic.  Every binary32 operation is one IEEE-754 operation rounded to
 * nearest-even (the file is compiled with -ffp-contract=off and without any
 * fast-math flag, so no multiply-add is fused).  The pages compute the
 * quantizer and the cumulative scores in float32 (their code casts to float32
 * first), so the oracle does too.  Error statistics accumulate in binary64.
 *
 * Sources, cited by page title and section:
 *  [FtC] "KV Compression 公式到源码对照"
 *        §1.1 symmetric per-channel quantization, §1.2 asymmetric per-channel
 *        quantization, §1.3 dequantization and error metrics, §2 compression
 *        ratio including scale/zero-point bytes, §3.1 H2O cumulative attention
 *        score, §3.2 recent window union heavy hitters, §3.3 SnapKV one-shot
 *        selection, §4 token compression ratio.
 *  [KVC] "KV cache 压缩：把历史装得更小"
 *        §"量化：位置都留着，每个数更短" (group-wise x ~ s*(q - z); KIVI groups
 *        K per channel and V per token), §"4 bit 的实际压缩率由分组大小决定"
 *        (payload ceil(N*bits/8) bytes plus per-group bf16 scale and zero),
 *        §"带残差区的压缩预算，逐项加起来" (most recent tokens stay bf16),
 *        §"少存 token：合并，或淘汰" (eviction really frees the dropped K/V),
 *        §"K 的误差会改变权重，V 的误差会改变内容" (logit_t = q^T k_t / sqrt(d),
 *        y = sum_t a_t v_t with a = softmax of the logits), §"让 kernel 接住收益"
 *        (the attention kernel reads the quantized cache and dequantizes it).
 *  KV-COBRA notes (papernotes.org), "关键设计" item 4: an orthogonal
 *        Walsh-Hadamard rotation with fixed random sign flips equalises the
 *        variances of the coordinates before scalar quantization.
 *
 * Readings taken where the pages are silent (each one also listed in the
 * design notes):
 *  - rounding is round-half-to-even (numpy's round), division is a true IEEE
 *    division, the range/abs-max floor is the float32 value nearest 1e-8;
 *  - the codes are computed from the scale and zero point exactly as stored
 *    (bf16 metadata is rounded before the codes are derived);
 *  - a zero point stored as int8 saturates to [-128, 127];
 *  - codes are clipped as integers (no wrap-around), q + zp is a float32 sum;
 *  - "per channel" reduces over the token axis of each [outer] slice, in
 *    groups of g tokens (g = 0: all quantized tokens); "per token" reduces
 *    over groups of g channels of one token;
 *  - the last min(R, T) tokens of every [outer] slice stay in the source
 *    dtype (the residual window), for K and V alike;
 *  - packing is along the contiguous channel axis, element c in byte
 *    c*bits/8, lowest bits first, as (q & mask) in two's complement.  The
 *    bit order is a convention the pages do not fix: parity of the bit order
 *    is unpinned by the pages (pinned by byte counts and the round trip);
 *  - keep-set selection ranks by (score descending, index ascending), the
 *    recent window is min(W, T) tokens, the heavy set has
 *    min(B - W', T - W') tokens, and W > B is rejected;
 *  - SnapKV's observation score is the float32 mean of the last obs_window
 *    history rows (sequential sum, then one division);
 *  - decode attention over a quantized cache takes its rows in full precision,
 *    s * (q - zp) in binary64 with the stored s and zp (a fused kernel rounds
 *    nothing to the cache dtype in between), the residual rows as stored, and
 *    computes the softmax attention itself in binary64;
 *  - the rotation fused into quantize / dequantize rounds the rotated values
 *    to bf16 (the dtype the unfused path stores them in) and forms them in
 *    binary32 as the fast transform, stages of channel bit 1, 2, 4, ... in
 *    that order; the stand-alone rotation is the binary64 matrix product.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype / mode / axis codes used by this oracle's own entry points */
enum { OR_F32 = 0, OR_BF16 = 1, OR_I8 = 2, OR_NONE = 3 };
enum { OR_SYM = 0, OR_ASYM = 1 };
enum { OR_ALONG_T = 0, OR_ALONG_C = 1 };
enum { OR_OK = 0, OR_EINVAL = 1 };

typedef struct {
    int64_t outer, T, C;
    int32_t bits, mode, qmin, qmax, axis;
    int64_t group, residual;
    int32_t scale_dtype, zero_dtype;
} or_params;

/* ------------------------------------------------------------------ */
/* bf16 <-> f32.  A bf16 value is the top 16 bits of a binary32.        */
/* ------------------------------------------------------------------ */

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

static float bf16_to_f32(uint16_t h) { return bits_to_f32((uint32_t)h << 16); }

/* Round a binary32 to the nearest bf16, ties to the even bf16 (the IEEE
 * default).  Written from the definition: take the two bf16 neighbours that
 * bracket f and keep the nearer one; on an exact tie keep the one whose last
 * kept bit is 0.  Past the largest finite bf16 the upper neighbour is 2^128,
 * which becomes infinity. */
static uint16_t f32_to_bf16(float f)
{
    uint32_t u = f32_to_bits(f);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t sign = u & 0x80000000u;
    uint32_t mag = u & 0x7FFFFFFFu;
    uint32_t lo = mag & 0xFFFF0000u;            /* neighbour toward zero */
    if (lo == mag) return (uint16_t)((sign | lo) >> 16);
    uint32_t hi = lo + 0x00010000u;             /* next bf16 up in magnitude */
    double dlo = (double)bits_to_f32(lo);
    double dhi = (hi >= 0x7F800000u) ? ldexp(1.0, 128) : (double)bits_to_f32(hi);
    double dm = (double)bits_to_f32(mag);
    double below = dm - dlo, above = dhi - dm;  /* both exact in binary64 */
    uint32_t pick;
    if (below < above) pick = lo;
    else if (above < below) pick = hi;
    else pick = ((lo >> 16) & 1u) ? hi : lo;    /* tie: even last bit */
    if (pick >= 0x7F800000u) pick = 0x7F800000u; /* overflow to infinity */
    return (uint16_t)((sign | pick) >> 16);
}

static double load_as_double(const void* p, int dtype, int64_t i)
{
    if (dtype == OR_BF16) return (double)bf16_to_f32(((const uint16_t*)p)[i]);
    return (double)((const float*)p)[i];
}

static float load_as_float(const void* p, int dtype, int64_t i)
{
    if (dtype == OR_BF16) return bf16_to_f32(((const uint16_t*)p)[i]);
    return ((const float*)p)[i];
}

/* Store a float in dtype (bf16: rounded to nearest-even). */
static void store_float(void* p, int dtype, int64_t i, float v)
{
    if (dtype == OR_BF16) ((uint16_t*)p)[i] = f32_to_bf16(v);
    else ((float*)p)[i] = v;
}

static size_t dtype_size(int dtype)
{
    switch (dtype) {
    case OR_F32: return 4;
    case OR_BF16: return 2;
    case OR_I8: return 1;
    default: return 0;
    }
}

/* ------------------------------------------------------------------ */
/* parameters and sizes                                                */
/* ------------------------------------------------------------------ */

static int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* quantized token count: the residual window holds the last min(R, T) tokens */
static int64_t quantized_tokens(const or_params* p) { return p->T - min64(p->residual, p->T); }

/* number of elements in one group (before clipping the last partial group) */
static int64_t group_len(const or_params* p)
{
    int64_t Tq = quantized_tokens(p);
    if (p->group > 0) return p->group;
    return p->axis == OR_ALONG_T ? Tq : p->C;
}

static int64_t group_count(const or_params* p)
{
    int64_t Tq = quantized_tokens(p);
    if (p->outer == 0 || Tq == 0 || p->C == 0) return 0;
    int64_t g = group_len(p);
    if (p->axis == OR_ALONG_T) return p->outer * ceil_div(Tq, g) * p->C;
    return p->outer * Tq * ceil_div(p->C, g);
}

static int check_params(const or_params* p, int x_dtype)
{
    if (p->outer < 0 || p->T < 0 || p->C < 0 || p->group < 0 || p->residual < 0) return OR_EINVAL;
    if (x_dtype != OR_F32 && x_dtype != OR_BF16) return OR_EINVAL;
    if (p->bits != 2 && p->bits != 4 && p->bits != 8) return OR_EINVAL;
    if ((p->C * p->bits) % 8 != 0) return OR_EINVAL;
    if (p->axis != OR_ALONG_T && p->axis != OR_ALONG_C) return OR_EINVAL;
    if (p->scale_dtype != OR_F32 && p->scale_dtype != OR_BF16) return OR_EINVAL;
    int half = 1 << (p->bits - 1);
    if (p->mode == OR_SYM) {
        if (p->qmax < 1 || p->qmax > half - 1) return OR_EINVAL;
        if (p->zero_dtype != OR_NONE) return OR_EINVAL;
    } else if (p->mode == OR_ASYM) {
        if (p->qmin >= p->qmax) return OR_EINVAL;
        if (p->qmin < 0) { if (p->qmin < -half || p->qmax > half - 1) return OR_EINVAL; }
        else if (p->qmax > (1 << p->bits) - 1) return OR_EINVAL;
        if (p->zero_dtype != OR_I8 && p->zero_dtype != OR_BF16 && p->zero_dtype != OR_F32) return OR_EINVAL;
    } else {
        return OR_EINVAL;
    }
    return OR_OK;
}

/* Byte counts of the quantized representation ([KVC] storage table:
 * payload bits/8 per number plus per-group metadata, plus the residual). */
int oracle_sizes(const or_params* p, int x_dtype, int64_t* codes_B, int64_t* scale_B,
                 int64_t* zero_B, int64_t* resid_B)
{
    if (check_params(p, x_dtype) != OR_OK) return OR_EINVAL;
    int64_t Tq = quantized_tokens(p);
    int64_t ng = group_count(p);
    *codes_B = p->outer * Tq * p->C * p->bits / 8;
    *scale_B = ng * (int64_t)dtype_size(p->scale_dtype);
    *zero_B = p->mode == OR_ASYM ? ng * (int64_t)dtype_size(p->zero_dtype) : 0;
    *resid_B = p->outer * (p->T - Tq) * p->C * (int64_t)dtype_size(x_dtype);
    return OR_OK;
}

/* [FtC] §2: original bytes over data + scale + zero-point bytes; the
 * residual window is part of the compressed footprint. */
double oracle_compression_ratio(int64_t orig_B, int64_t codes_B, int64_t scale_B,
                                int64_t zero_B, int64_t resid_B)
{
    return (double)orig_B / (double)(codes_B + scale_B + zero_B + resid_B);
}

/* [FtC] §4: T / K, defined only for 0 < K <= T. */
int oracle_token_compression_ratio(int64_t total_tokens, int64_t kept_tokens, double* out)
{
    if (total_tokens <= 0 || kept_tokens <= 0 || kept_tokens > total_tokens) return OR_EINVAL;
    *out = (double)total_tokens / (double)kept_tokens;
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* group enumeration                                                   */
/* ------------------------------------------------------------------ */

/* A group is a list of element positions.  The callback style keeps the
 * quantize / dequantize / stats loops identical in their enumeration. */
typedef struct {
    int64_t count;      /* members */
    int64_t first;      /* index of member 0 in x */
    int64_t stride;     /* distance between consecutive members in x */
    int64_t meta;       /* index into scale[] / zero[] */
} or_group;

/* Enumerate every group of the quantized region in metadata order. */
static int64_t group_at(const or_params* p, int64_t gidx, or_group* G)
{
    int64_t Tq = quantized_tokens(p);
    int64_t g = group_len(p);
    if (p->axis == OR_ALONG_T) {
        /* metadata [outer][ceil(Tq/g)][C]; members are g tokens of one channel */
        int64_t ngt = ceil_div(Tq, g);
        int64_t c = gidx % p->C;
        int64_t gi = (gidx / p->C) % ngt;
        int64_t o = gidx / (p->C * ngt);
        int64_t t0 = gi * g;
        G->count = min64(g, Tq - t0);
        G->first = (o * p->T + t0) * p->C + c;
        G->stride = p->C;
    } else {
        /* metadata [outer][Tq][ceil(C/g)]; members are g channels of one token */
        int64_t ngc = ceil_div(p->C, g);
        int64_t gi = gidx % ngc;
        int64_t t = (gidx / ngc) % Tq;
        int64_t o = gidx / (ngc * Tq);
        int64_t c0 = gi * g;
        G->count = min64(g, p->C - c0);
        G->first = (o * p->T + t) * p->C + c0;
        G->stride = 1;
    }
    G->meta = gidx;
    return G->count;
}

/* element index in x  ->  index of its code in the packed code stream */
static int64_t code_index(const or_params* p, int64_t xi)
{
    int64_t c = xi % p->C;
    int64_t t = (xi / p->C) % p->T;
    int64_t o = xi / (p->C * p->T);
    int64_t Tq = quantized_tokens(p);
    return (o * Tq + t) * p->C + c;
}

static void put_code(uint8_t* codes, int bits, int64_t ci, int32_t q)
{
    int per = 8 / bits;
    uint32_t mask = (1u << bits) - 1u;
    int64_t byte = ci / per;
    int shift = (int)(ci % per) * bits;
    codes[byte] = (uint8_t)((codes[byte] & ~(mask << shift)) | (((uint32_t)q & mask) << shift));
}

static int32_t get_code(const uint8_t* codes, int bits, int64_t ci, int is_signed)
{
    int per = 8 / bits;
    uint32_t mask = (1u << bits) - 1u;
    uint32_t field = ((uint32_t)codes[ci / per] >> ((int)(ci % per) * bits)) & mask;
    if (is_signed && (field & (1u << (bits - 1)))) return (int32_t)field - (int32_t)(1u << bits);
    return (int32_t)field;
}

static int codes_signed(const or_params* p) { return p->mode == OR_SYM || p->qmin < 0; }

/* metadata as used by the arithmetic: the stored value, widened to float */
static float load_meta(const void* buf, int dtype, int64_t i)
{
    if (dtype == OR_BF16) return bf16_to_f32(((const uint16_t*)buf)[i]);
    if (dtype == OR_I8) return (float)((const int8_t*)buf)[i];
    return ((const float*)buf)[i];
}

static const float kRangeFloor = 1e-8f;  /* [FtC] §1.1/§1.2: clip at 1e-8 */

/* ------------------------------------------------------------------ */
/* quantize ([FtC] §1.1, §1.2; [KVC] group-wise form and residual)     */
/* ------------------------------------------------------------------ */

int oracle_quantize(const void* x, int x_dtype, const or_params* p,
                    void* codes, void* scale, void* zero, void* resid)
{
    if (check_params(p, x_dtype) != OR_OK) return OR_EINVAL;
    int64_t Tq = quantized_tokens(p);
    int64_t ng = group_count(p);
    int64_t codes_B = p->outer * Tq * p->C * p->bits / 8;
    if (codes_B) memset(codes, 0, (size_t)codes_B);
    for (int64_t gidx = 0; gidx < ng; ++gidx) {
        or_group G;
        group_at(p, gidx, &G);
        /* 1. group statistics in float32 */
        float amax = 0.0f, mn = 0.0f, mx = 0.0f;
        for (int64_t m = 0; m < G.count; ++m) {
            float v = load_as_float(x, x_dtype, G.first + m * G.stride);
            float a = fabsf(v);
            if (m == 0) { amax = a; mn = v; mx = v; }
            else { if (a > amax) amax = a; if (v < mn) mn = v; if (v > mx) mx = v; }
        }
        /* 2. scale, rounded to its storage dtype before any further use */
        float s;
        if (p->mode == OR_SYM) {
            if (amax < kRangeFloor) amax = kRangeFloor;
            s = amax / (float)p->qmax;
        } else {
            float rng = mx - mn;
            if (rng < kRangeFloor) rng = kRangeFloor;
            s = rng / (float)(p->qmax - p->qmin);
        }
        store_float(scale, p->scale_dtype, G.meta, s);
        float s_use = load_meta(scale, p->scale_dtype, G.meta);
        /* 3. zero point (asymmetric), rounded then stored */
        float zp_use = 0.0f;
        if (p->mode == OR_ASYM) {
            float t = mn / s_use;
            float zp = rintf((float)p->qmin - t);
            if (p->zero_dtype == OR_I8) {
                if (zp < -128.0f) zp = -128.0f;
                if (zp > 127.0f) zp = 127.0f;
                ((int8_t*)zero)[G.meta] = (int8_t)zp;
            } else {
                store_float(zero, p->zero_dtype, G.meta, zp);
            }
            zp_use = load_meta(zero, p->zero_dtype, G.meta);
        }
        /* 4. codes: round, shift by the zero point, clip as integers */
        float lo = p->mode == OR_SYM ? -(float)p->qmax : (float)p->qmin;
        float hi = (float)p->qmax;
        for (int64_t m = 0; m < G.count; ++m) {
            int64_t xi = G.first + m * G.stride;
            float v = load_as_float(x, x_dtype, xi);
            float r = rintf(v / s_use);
            float q = p->mode == OR_SYM ? r : r + zp_use;
            if (q < lo) q = lo;
            if (q > hi) q = hi;
            put_code((uint8_t*)codes, p->bits, code_index(p, xi), (int32_t)q);
        }
    }
    /* 5. residual window: the last min(R, T) tokens, copied bit for bit */
    int64_t R = p->T - Tq;
    size_t es = dtype_size(x_dtype);
    for (int64_t o = 0; o < p->outer; ++o)
        for (int64_t r = 0; r < R; ++r)
            memcpy((char*)resid + (size_t)((o * R + r) * p->C) * es,
                   (const char*)x + (size_t)((o * p->T + Tq + r) * p->C) * es, (size_t)p->C * es);
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* dequantize ([FtC] §1.3: x_hat = (q - zero_point) * scale)            */
/* ------------------------------------------------------------------ */

/* x_hat of one quantized element, in float32 */
static float dequant_one(const or_params* p, const void* codes, const void* scale,
                         const void* zero, int64_t gmeta, int64_t xi)
{
    int32_t q = get_code((const uint8_t*)codes, p->bits, code_index(p, xi), codes_signed(p));
    float s_use = load_meta(scale, p->scale_dtype, gmeta);
    float zp_use = p->mode == OR_ASYM ? load_meta(zero, p->zero_dtype, gmeta) : 0.0f;
    return ((float)q - zp_use) * s_use;
}

/* out is [outer, T, C] in out_dtype; the residual buffer holds the last
 * min(R, T) tokens in the same dtype. */
int oracle_dequantize(const void* codes, const void* scale, const void* zero, const void* resid,
                      const or_params* p, void* out, int out_dtype)
{
    if (check_params(p, out_dtype) != OR_OK) return OR_EINVAL;
    int64_t ng = group_count(p);
    for (int64_t gidx = 0; gidx < ng; ++gidx) {
        or_group G;
        group_at(p, gidx, &G);
        for (int64_t m = 0; m < G.count; ++m) {
            int64_t xi = G.first + m * G.stride;
            store_float(out, out_dtype, xi, dequant_one(p, codes, scale, zero, G.meta, xi));
        }
    }
    int64_t Tq = quantized_tokens(p);
    int64_t R = p->T - Tq;
    size_t es = dtype_size(out_dtype);
    for (int64_t o = 0; o < p->outer; ++o)
        for (int64_t r = 0; r < R; ++r)
            memcpy((char*)out + (size_t)((o * p->T + Tq + r) * p->C) * es,
                   (const char*)resid + (size_t)((o * R + r) * p->C) * es, (size_t)p->C * es);
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* error statistics ([FtC] §1.3: RMSE, max-abs, mean-abs)               */
/* ------------------------------------------------------------------ */

/* out[0] = rmse, out[1] = max |x - x_hat|, out[2] = mean |x - x_hat|, over all
 * N = outer*T*C elements; x_hat is the value dequantize returns in x's dtype,
 * so residual tokens contribute an error of exactly zero. */
int oracle_error_stats(const void* x, int x_dtype, const void* codes, const void* scale,
                       const void* zero, const void* resid, const or_params* p, double* out)
{
    (void)resid;
    if (check_params(p, x_dtype) != OR_OK) return OR_EINVAL;
    int64_t N = p->outer * p->T * p->C;
    if (N == 0) return OR_EINVAL;
    double s1 = 0.0, s2 = 0.0, mxd = 0.0;
    int64_t ng = group_count(p);
    for (int64_t gidx = 0; gidx < ng; ++gidx) {
        or_group G;
        group_at(p, gidx, &G);
        for (int64_t m = 0; m < G.count; ++m) {
            int64_t xi = G.first + m * G.stride;
            float xh = dequant_one(p, codes, scale, zero, G.meta, xi);
            double xhd = x_dtype == OR_BF16 ? (double)bf16_to_f32(f32_to_bf16(xh)) : (double)xh;
            double d = load_as_double(x, x_dtype, xi) - xhd;
            double a = fabs(d);
            s2 += d * d;
            s1 += a;
            if (a > mxd) mxd = a;
        }
    }
    out[0] = sqrt(s2 / (double)N);
    out[1] = mxd;
    out[2] = s1 / (double)N;
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* keep-set selection ([FtC] §3.1-§3.3)                                  */
/* ------------------------------------------------------------------ */

typedef struct { float score; int32_t index; } or_cand;

/* rank: higher score first, lower index first among equal scores */
static int cand_cmp(const void* a, const void* b)
{
    const or_cand* x = (const or_cand*)a;
    const or_cand* y = (const or_cand*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->index > y->index) - (x->index < y->index);
}

static int cmp_i32(const void* a, const void* b)
{
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* keep = sort(TopK(score over [0, T-W'), min(B-W', T-W')) union [T-W', T)),
 * W' = min(W, T); writes min(B, T) indices. */
static void select_one_head(const float* score, int64_t T, int64_t budget, int64_t window,
                            int32_t* keep, or_cand* scratch)
{
    int64_t Wr = min64(window, T);
    int64_t rs = T - Wr;
    int64_t k = min64(budget - Wr, rs);
    for (int64_t i = 0; i < rs; ++i) { scratch[i].score = score[i]; scratch[i].index = (int32_t)i; }
    qsort(scratch, (size_t)rs, sizeof(or_cand), cand_cmp);
    int64_t n = 0;
    for (int64_t j = 0; j < k; ++j) keep[n++] = scratch[j].index;
    qsort(keep, (size_t)n, sizeof(int32_t), cmp_i32);
    for (int64_t i = rs; i < T; ++i) keep[n++] = (int32_t)i;
}

static int check_select(int64_t heads, int64_t steps, int64_t T, int64_t budget, int64_t window)
{
    if (heads < 0 || steps < 1 || T < 0 || budget < 1 || window < 0 || window > budget) return OR_EINVAL;
    if (T > INT32_MAX) return OR_EINVAL;
    return OR_OK;
}

/* H2O: score[i] = sum over all steps t (in order) of a_t(i), float32.
 * hist is [heads, steps, T]; keep is [heads, min(B, T)]; scores ([heads, T])
 * may be NULL. */
int oracle_h2o_select(const float* hist, int64_t heads, int64_t steps, int64_t T,
                      int64_t budget, int64_t window, int32_t* keep, float* scores)
{
    if (check_select(heads, steps, T, budget, window) != OR_OK) return OR_EINVAL;
    int64_t K = min64(budget, T);
    float* sc = (float*)malloc(sizeof(float) * (size_t)(T ? T : 1));
    or_cand* scratch = (or_cand*)malloc(sizeof(or_cand) * (size_t)(T ? T : 1));
    for (int64_t h = 0; h < heads; ++h) {
        for (int64_t i = 0; i < T; ++i) sc[i] = 0.0f;
        for (int64_t t = 0; t < steps; ++t) {
            const float* row = hist + (h * steps + t) * T;
            for (int64_t i = 0; i < T; ++i) sc[i] = sc[i] + row[i];
        }
        if (scores) memcpy(scores + h * T, sc, sizeof(float) * (size_t)T);
        select_one_head(sc, T, budget, window, keep + h * K, scratch);
    }
    free(sc);
    free(scratch);
    return OR_OK;
}

/* SnapKV: observation score = (sum of the last obs_window rows) / obs_window. */
int oracle_snapkv_select(const float* hist, int64_t heads, int64_t steps, int64_t T,
                         int64_t obs_window, int64_t budget, int64_t window,
                         int32_t* keep, float* scores)
{
    if (check_select(heads, steps, T, budget, window) != OR_OK) return OR_EINVAL;
    if (obs_window < 1 || obs_window > steps) return OR_EINVAL;
    int64_t K = min64(budget, T);
    float* sc = (float*)malloc(sizeof(float) * (size_t)(T ? T : 1));
    or_cand* scratch = (or_cand*)malloc(sizeof(or_cand) * (size_t)(T ? T : 1));
    for (int64_t h = 0; h < heads; ++h) {
        for (int64_t i = 0; i < T; ++i) sc[i] = 0.0f;
        for (int64_t t = steps - obs_window; t < steps; ++t) {
            const float* row = hist + (h * steps + t) * T;
            for (int64_t i = 0; i < T; ++i) sc[i] = sc[i] + row[i];
        }
        for (int64_t i = 0; i < T; ++i) sc[i] = sc[i] / (float)obs_window;
        if (scores) memcpy(scores + h * T, sc, sizeof(float) * (size_t)T);
        select_one_head(sc, T, budget, window, keep + h * K, scratch);
    }
    free(sc);
    free(scratch);
    return OR_OK;
}

/* Compaction ([KVC] eviction frees the dropped entries):
 * out[h][j][:] = kv[h][keep[h][j]][:] for j < K. */
int oracle_compact(const void* kv, int64_t elem_size, int64_t heads, int64_t T, int64_t D,
                   const int32_t* keep, int64_t K, void* out)
{
    if (heads < 0 || T < 0 || D < 0 || K < 0 || K > T || elem_size <= 0) return OR_EINVAL;
    size_t row = (size_t)(D * elem_size);
    for (int64_t h = 0; h < heads; ++h)
        for (int64_t j = 0; j < K; ++j) {
            int32_t i = keep[h * K + j];
            if (i < 0 || i >= T) return OR_EINVAL;
            memcpy((char*)out + (size_t)(h * K + j) * row, (const char*)kv + (size_t)(h * T + i) * row, row);
        }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* decode attention over the dequantized cache                          */
/* ------------------------------------------------------------------ */

/* The cache rows in binary64: s * (q - zp) with the stored scale and zero
 * point for the quantized tokens (exact: the difference of two small integers
 * times a 24-bit scale fits 53 bits), the residual rows widened from the
 * source dtype x_dtype.  out is [outer, T, C]. */
int oracle_dequantize_f64(const void* codes, const void* scale, const void* zero, const void* resid,
                          const or_params* p, int x_dtype, double* out)
{
    if (check_params(p, x_dtype) != OR_OK) return OR_EINVAL;
    int64_t ng = group_count(p);
    for (int64_t gidx = 0; gidx < ng; ++gidx) {
        or_group G;
        group_at(p, gidx, &G);
        for (int64_t m = 0; m < G.count; ++m) {
            int64_t xi = G.first + m * G.stride;
            int32_t q = get_code((const uint8_t*)codes, p->bits, code_index(p, xi), codes_signed(p));
            double s_use = (double)load_meta(scale, p->scale_dtype, G.meta);
            double zp_use = p->mode == OR_ASYM ? (double)load_meta(zero, p->zero_dtype, G.meta) : 0.0;
            out[xi] = s_use * ((double)q - zp_use);
        }
    }
    int64_t Tq = quantized_tokens(p);
    int64_t R = p->T - Tq;
    for (int64_t o = 0; o < p->outer; ++o)
        for (int64_t r = 0; r < R; ++r)
            for (int64_t c = 0; c < p->C; ++c)
                out[(o * p->T + Tq + r) * p->C + c] = load_as_double(resid, x_dtype, (o * R + r) * p->C + c);
    return OR_OK;
}

/* y[o][j][:] = sum_t softmax_t( q[o][j][:] . k[o][t][:] / sqrt(C) ) v[o][t][:]
 * in binary64; query head j of slice o reads KV slice o (group query heads
 * per KV slice).  q, out: [outer][group][C]; k, v: [outer][T][C]. */
int oracle_attend(const double* q, int64_t group, const double* k, const double* v, int64_t outer,
                  int64_t T, int64_t C, double* out)
{
    if (outer < 0 || T < 1 || C < 1 || group < 1) return OR_EINVAL;
    double* logit = (double*)malloc((size_t)T * sizeof(double));
    if (!logit) return OR_EINVAL;
    const double inv_sqrt = 1.0 / sqrt((double)C);
    for (int64_t o = 0; o < outer; ++o)
        for (int64_t j = 0; j < group; ++j) {
            const double* qv = q + (o * group + j) * C;
            double mx = -INFINITY;
            for (int64_t t = 0; t < T; ++t) {
                const double* kt = k + (o * T + t) * C;
                double dot = 0.0;
                for (int64_t c = 0; c < C; ++c) dot += qv[c] * kt[c];
                logit[t] = dot * inv_sqrt;
                if (logit[t] > mx) mx = logit[t];
            }
            double z = 0.0;
            for (int64_t t = 0; t < T; ++t) {
                logit[t] = exp(logit[t] - mx);
                z += logit[t];
            }
            double* y = out + (o * group + j) * C;
            for (int64_t c = 0; c < C; ++c) y[c] = 0.0;
            for (int64_t t = 0; t < T; ++t) {
                const double* vt = v + (o * T + t) * C;
                for (int64_t c = 0; c < C; ++c) y[c] += logit[t] * vt[c];
            }
            for (int64_t c = 0; c < C; ++c) y[c] /= z;
        }
    free(logit);
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* randomized Hadamard rotation (KV-COBRA notes, "关键设计" item 4)      */
/* ------------------------------------------------------------------ */

/* y = (1/sqrt(C)) H (signs .* x) per row (forward), or
 * x = signs .* ((1/sqrt(C)) H y) (inverse), in binary64.  H is built by the
 * Sylvester recursion H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]] and applied
 * as a plain matrix-vector product.  A negative sign entry flips its channel.
 * x, out: [rows][C]; C a power of two. */
int oracle_rotate(const double* x, int64_t rows, int64_t C, const int8_t* signs, int inverse, double* out)
{
    if (rows < 0 || C < 1 || (C & (C - 1)) != 0) return OR_EINVAL;
    signed char* H = (signed char*)malloc((size_t)(C * C));
    double* u = (double*)malloc((size_t)C * sizeof(double));
    if (!H || !u) { free(H); free(u); return OR_EINVAL; }
    H[0] = 1;
    for (int64_t n = 1; n < C; n *= 2)            /* H_n in the top-left n x n block -> H_2n */
        for (int64_t i = 0; i < n; ++i)
            for (int64_t j = 0; j < n; ++j) {
                signed char h = H[i * C + j];
                H[i * C + j + n] = h;
                H[(i + n) * C + j] = h;
                H[(i + n) * C + j + n] = (signed char)(-h);
            }
    const double scale = 1.0 / sqrt((double)C);
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * C;
        double* yr = out + r * C;
        for (int64_t c = 0; c < C; ++c) u[c] = (!inverse && signs[c] < 0) ? -xr[c] : xr[c];
        for (int64_t i = 0; i < C; ++i) {
            double acc = 0.0;
            for (int64_t c = 0; c < C; ++c) acc += (double)H[i * C + c] * u[c];
            acc *= scale;
            yr[i] = (inverse && signs[i] < 0) ? -acc : acc;
        }
    }
    free(H);
    free(u);
    return OR_OK;
}

/* The same rotation evaluated in binary32 as the fast Walsh-Hadamard
 * transform, for the rotation fused into quantize / dequantize: there the
 * rotated values are rounded to bf16 and quantized, so the codes are decided
 * on binary32 results and both sides must form them the same way.  The
 * Sylvester recursion read as an algorithm: y = H_2n u is H_n applied to each
 * half of u, then the halves combined as (top + bottom, top - bottom).
 * Unrolled, for h = 1, 2, 4, ..., C/2 in that order, every channel pair
 * (j, j + h) with bit h of j clear becomes (v_j + v_{j+h}, v_j - v_{j+h}),
 * each one IEEE binary32 operation; then every value is multiplied by the
 * binary32 nearest to 1/sqrt(C) (taken as 1/sqrt(C) in binary64, then rounded
 * to binary32).  Forward flips the signed channels of x first, inverse flips
 * the outputs.  x: [rows][C] in x_dtype (F32 or BF16); out: [rows][C] in
 * out_dtype (F32, or BF16 rounded to nearest-even). */
int oracle_rotate_fwht32(const void* x, int x_dtype, int64_t rows, int64_t C, const int8_t* signs, int inverse,
                         void* out, int out_dtype)
{
    if (rows < 0 || C < 1 || (C & (C - 1)) != 0) return OR_EINVAL;
    if ((x_dtype != OR_F32 && x_dtype != OR_BF16) || (out_dtype != OR_F32 && out_dtype != OR_BF16)) return OR_EINVAL;
    float* v = (float*)malloc((size_t)C * sizeof(float));
    if (!v) return OR_EINVAL;
    const float scale = (float)(1.0 / sqrt((double)C));
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < C; ++c) {
            const float xc = load_as_float(x, x_dtype, r * C + c);
            v[c] = (!inverse && signs[c] < 0) ? -xc : xc;
        }
        for (int64_t h = 1; h < C; h *= 2)
            for (int64_t j = 0; j < C; ++j)
                if ((j & h) == 0) {
                    const float a = v[j], b = v[j + h];
                    v[j] = a + b;
                    v[j + h] = a - b;
                }
        for (int64_t c = 0; c < C; ++c) {
            float y = v[c] * scale;
            if (inverse && signs[c] < 0) y = -y;
            store_float(out, out_dtype, r * C + c, y);
        }
    }
    free(v);
    return OR_OK;
}

