// kvq_div.cuh -- division of 32-bit integers by a divisor fixed per launch,
// by a multiply-high and shifts (Granlund and Montgomery, "Division by
// invariant integers using multiplication", 1994, section 4): with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (t + ((n - t) >> 1)) >> (l - 1), t = mulhi(m, n), for every 32-bit
// n; d = 1 is taken apart.
#pragma once

#include <stdint.h>

namespace kvq {

struct DivU32 {
    uint32_t d, m, sh;
};

inline DivU32 make_div(uint32_t d) {
    DivU32 v{d, 0u, 0u};
    if (d > 1) {
        uint32_t l = 0;
        while ((1ull << l) < d) ++l;
        v.m = (uint32_t)(((1ull << 32) * ((1ull << l) - d)) / d + 1);
        v.sh = l - 1;
    }
    return v;
}

__device__ __forceinline__ uint32_t div_u32(uint32_t n, const DivU32& v) {
    if (v.d == 1) return n;
    const uint32_t t = __umulhi(v.m, n);
    return (t + ((n - t) >> 1)) >> v.sh;
}

}  // namespace kvq
