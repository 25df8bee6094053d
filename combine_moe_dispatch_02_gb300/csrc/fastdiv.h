// fastdiv.h -- division by a divisor fixed at launch, with a multiply-high.
//
// Granlund and Montgomery, "Division by invariant integers using
// multiplication" (PLDI 1994), unsigned N-bit division with the round-up
// multiplier of N + 1 bits kept as its low N bits: for a divisor d >= 1 let
// l = ceil(log2 d) and m = floor(2^N (2^l - d) / d) + 1 (< 2^N); then for
// every 0 <= n < 2^N
//     t = floor(m n / 2^N),   n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0).
// Here N = 32 and d <= 2^31.  Plain C++ on the host (a test builds it with
// the host compiler alone), the hardware multiply-high on the device.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define MOE_FASTDIV_HD __host__ __device__
#else
#define MOE_FASTDIV_HD
#endif

namespace moe {

struct FastDiv {
    uint32_t d;      // the divisor
    uint32_t m;      // low 32 bits of the multiplier
    uint32_t s1;     // min(l, 1)
    uint32_t s2;     // max(l - 1, 0)
};

// d in [1, 2^31].
inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t l = 0;
    while ((uint64_t{1} << l) < d) ++l;
    const uint64_t m = ((uint64_t{1} << 32) * ((uint64_t{1} << l) - d)) / d + 1;
    FastDiv f;
    f.d = d;
    f.m = static_cast<uint32_t>(m);
    f.s1 = l < 1 ? l : 1u;
    f.s2 = l > 0 ? l - 1 : 0u;
    return f;
}

MOE_FASTDIV_HD inline uint32_t fastdiv(uint32_t n, const FastDiv& f) {
#if defined(__CUDA_ARCH__)
    const uint32_t t = __umulhi(f.m, n);
#else
    const uint32_t t = static_cast<uint32_t>((static_cast<uint64_t>(f.m) * n) >> 32);
#endif
    return (t + ((n - t) >> f.s1)) >> f.s2;
}

}  // namespace moe
