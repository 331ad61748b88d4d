// Exhaustive check of the fast-path arithmetic in kvq_fast.cuh against CUDA's
// IEEE operations:
//  1. quot1 / quot2 (reciprocal + one FMA remainder correction) == __fdiv_rn
//     bit for bit for every bf16 x and bf16 scale s (|x|, |x/s| >= 2^-100)
//     inside the fast domain, and the rounded codes agree for every x;
//  2. the same for every bf16 x and the float32 scales RN(a / qmax) of every
//     bf16 abs-max a and every qmax used by the formats (1, 3, 7, 15, 127, 255);
//  3. 2^30 random float32 pairs (counter-based hash) inside the fast domain;
//  4. bits(y + 1.5*2^23) - 0x4B400000 == rintf(y) for every float |y| < 2^21;
//  5. the group-range division: quot1(r, n, RN(1/n)) == __fdiv_rn(r, n) for
//     every float r in [2^-100, 2^127] and every integer n in 1..255.
// Prints the mismatch counts; exit status 0 only if all are zero.
#include <cstdio>
#include <cstdint>
#include "kvq_fast.cuh"

using namespace kvq;

__device__ unsigned long long g_bad[5];
__device__ unsigned int g_nex;
__device__ float g_ex[64][5];   // first failing pairs: x, s, quotient, __fdiv_rn, slot
__device__ unsigned long long g_checked[5];

__device__ __forceinline__ bool bf16_finite(uint32_t b) { return ((b >> 7) & 0xFF) != 0xFF; }

// In the fast domain the quotient must be bit-identical to __fdiv_rn whenever
// |x| and |x / s| are at least 2^-100 (below that the remainder or the
// quotient itself underflows, and x / s is far below 1/2, so only the rounded
// code matters); the rounded code (bits of q + 1.5*2^23) must be identical
// for every pair.
__device__ __forceinline__ void check_pair(float x, float s, int slot, unsigned long long& bad, unsigned long long& n) {
    const float inv = __frcp_rn(s);
    if (!quot_ok(s, inv, fabsf(x))) return;
    const float want = __fdiv_rn(x, s), wantn = __fdiv_rn(-x, s);
    const float got1 = quot1(x, s, inv);
    QuotK k;
    k.ns = pk(-s, -s);
    k.inv = pk(inv, inv);
    const u64 got2 = quot2(pk(x, -x), k);
    ++n;
    const bool exact_required = fabsf(x) >= 0x1p-100f && fabsf(want) >= 0x1p-100f;
    bool ok;
    if (exact_required)
        ok = __float_as_uint(got1) == __float_as_uint(want) && __float_as_uint(lo_of(got2)) == __float_as_uint(want) &&
             __float_as_uint(hi_of(got2)) == __float_as_uint(wantn);
    else
        ok = true;
    const u64 rg = rint_bits2(got2), rw = rint_bits2(pk(want, wantn));
    ok = ok && rg == rw && __float_as_uint(__fadd_rn(got1, kMagic)) == lo_bits(rw);
    if (!ok) {
        ++bad;
        const unsigned int e = atomicAdd(&g_nex, 1u);
        if (e < 64) {
            g_ex[e][0] = x; g_ex[e][1] = s; g_ex[e][2] = got1; g_ex[e][3] = want; g_ex[e][4] = (float)slot;
        }
    }
}

// 1. all bf16 x  x  all positive bf16 s
__global__ void bf16_pairs() {
    unsigned long long bad = 0, n = 0;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (1ull << 32); i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t xb = (uint32_t)(i >> 16), sb = (uint32_t)(i & 0x7FFF);     // s > 0
        if ((i & 0xFFFF) >= 0x8000 || !bf16_finite(xb) || !bf16_finite(sb) || sb == 0) continue;
        check_pair(__uint_as_float(xb << 16), __uint_as_float(sb << 16), 0, bad, n);
    }
    atomicAdd(&g_bad[0], bad);
    atomicAdd(&g_checked[0], n);
}

// 2. bf16 x  x  float32 scales RN(a / qmax)
__global__ void bf16_x_f32_scales(float qmax) {
    unsigned long long bad = 0, n = 0;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (1ull << 31); i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t xb = (uint32_t)(i >> 15), ab = (uint32_t)(i & 0x7FFF);
        if (!bf16_finite(xb) || !bf16_finite(ab) || ab == 0) continue;
        const float s = __fdiv_rn(fmaxf(__uint_as_float(ab << 16), 1e-8f), qmax);
        check_pair(__uint_as_float(xb << 16), s, 1, bad, n);
    }
    atomicAdd(&g_bad[1], bad);
    atomicAdd(&g_checked[1], n);
}

__device__ __forceinline__ uint32_t mix(uint64_t v) {
    v ^= v >> 33; v *= 0xff51afd7ed558ccdull; v ^= v >> 33; v *= 0xc4ceb9fe1a85ec53ull; v ^= v >> 33;
    return (uint32_t)v;
}

// 3. random float32 pairs
__global__ void f32_random() {
    unsigned long long bad = 0, n = 0;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (1ull << 30); i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t a = mix(2 * i), b = mix(2 * i + 1);
        // x: any finite float; s: positive, exponent within the fast domain
        const float x = __uint_as_float(a);
        const float s = __uint_as_float((b & 0x007FFFFFu) | ((100u + (b >> 24) % 55u) << 23));
        if (!isfinite(x)) continue;
        check_pair(x, s, 2, bad, n);
    }
    atomicAdd(&g_bad[2], bad);
    atomicAdd(&g_checked[2], n);
}

// 4. magic rounding for every float with |y| < 2^21
__global__ void magic_round() {
    unsigned long long bad = 0, n = 0;
    const uint32_t lim = 0x4A000000u;   // 2^21
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < 2ull * lim; i += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t mag = (uint32_t)(i >> 1);
        const float y = __uint_as_float(mag | ((uint32_t)(i & 1) << 31));
        const u64 r = rint_bits2(pk(y, -y));
        const int want = (int)rintf(y);
        ++n;
        if ((int)(lo_bits(r) - kMagicBits) != want || (int)(hi_bits(r) - kMagicBits) != -want) ++bad;
    }
    atomicAdd(&g_bad[3], bad);
    atomicAdd(&g_checked[3], n);
}

// 5. range / integer divisor, every float r in [2^-100, 2^127], divisor n
__global__ void range_div(float n) {
    unsigned long long bad = 0, cnt = 0;
    const float inv = __frcp_rn(n);
    const uint32_t lo = 0x0D800000u, hi = 0x7F000000u;   // 2^-100 .. 2^127
    for (uint64_t i = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i <= hi; i += (uint64_t)gridDim.x * blockDim.x) {
        const float r = __uint_as_float((uint32_t)i);
        ++cnt;
        if (__float_as_uint(quot1(r, n, inv)) != __float_as_uint(__fdiv_rn(r, n))) {
            ++bad;
            const unsigned int e = atomicAdd(&g_nex, 1u);
            if (e < 64) { g_ex[e][0] = r; g_ex[e][1] = n; g_ex[e][2] = quot1(r, n, inv); g_ex[e][3] = __fdiv_rn(r, n); g_ex[e][4] = 5.0f; }
        }
    }
    atomicAdd(&g_bad[4], bad);
    atomicAdd(&g_checked[4], cnt);
}

int main() {
    const unsigned long long zero[5] = {0, 0, 0, 0, 0};
    cudaMemcpyToSymbol(g_bad, zero, sizeof(zero));
    cudaMemcpyToSymbol(g_checked, zero, sizeof(zero));
    const unsigned int z0 = 0;
    cudaMemcpyToSymbol(g_nex, &z0, sizeof(z0));
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    const int grid = sms * 8, block = 256;
    bf16_pairs<<<grid, block>>>();
    const float qmaxes[6] = {1.0f, 3.0f, 7.0f, 15.0f, 127.0f, 255.0f};
    for (float qm : qmaxes) bf16_x_f32_scales<<<grid, block>>>(qm);
    f32_random<<<grid, block>>>();
    magic_round<<<grid, block>>>();
    for (int n = 1; n <= 255; ++n) range_div<<<grid, block>>>((float)n);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { printf("CUDA error: %s\n", cudaGetErrorString(e)); return 2; }
    unsigned long long bad[5], n[5];
    cudaMemcpyFromSymbol(bad, g_bad, sizeof(bad));
    cudaMemcpyFromSymbol(n, g_checked, sizeof(n));
    const char* names[5] = {"bf16 x / bf16 s", "bf16 x / f32 RN(a/qmax)", "random f32 pairs", "magic rint |y|<2^21",
                            "range / n, n = 1..255"};
    unsigned int nex = 0;
    float ex[64][5];
    cudaMemcpyFromSymbol(&nex, g_nex, sizeof(nex));
    cudaMemcpyFromSymbol(ex, g_ex, sizeof(ex));
    for (unsigned int i = 0; i < nex && i < 64; ++i)
        printf("mismatch slot %d: x=%a s=%a quotient=%a fdiv=%a\n", (int)ex[i][4], ex[i][0], ex[i][1], ex[i][2], ex[i][3]);
    int rc = 0;
    for (int i = 0; i < 5; ++i) {
        printf("%-26s checked %llu mismatches %llu\n", names[i], n[i], bad[i]);
        if (bad[i] || !n[i]) rc = 1;
    }
    return rc;
}
