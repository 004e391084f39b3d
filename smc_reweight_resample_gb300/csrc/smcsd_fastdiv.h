// smcsd_fastdiv.h -- division by a divisor that is fixed for a whole launch (Granlund and
// Montgomery, "Division by invariant integers using multiplication", PLDI 1994): for d >= 1,
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, the quotient is
// q = (n + mulhi(n, m)) >> l for every n < 2^31. Host and device; used to decode the flat chunk
// index of the streaming pass without a hardware-less integer division per chunk.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define SMCSD_FD_HD __host__ __device__ __forceinline__
#else
#define SMCSD_FD_HD static inline
#endif

namespace smcsd {

struct FastDiv {
    uint32_t d, m;
    int l;
};

inline FastDiv make_fastdiv(uint32_t d) {
    int l = 0;
    while ((1ull << l) < (unsigned long long)d) ++l;
    const unsigned long long m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
    return FastDiv{d, (uint32_t)m, l};
}

SMCSD_FD_HD uint32_t fast_div(uint32_t n, const FastDiv& f) {
#ifdef __CUDA_ARCH__
    const uint32_t t = __umulhi(n, f.m);
#else
    const uint32_t t = (uint32_t)(((unsigned long long)n * f.m) >> 32);
#endif
    return (n + t) >> f.l;
}

}  // namespace smcsd
