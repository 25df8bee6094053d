// Host check of csrc/fastdiv.h against the C++ division operator: every
// divisor 1..4096 and a few large ones, against numerators near 0, near
// every multiple boundary of small quotients, random ones, and the top of
// the 32-bit range.  Prints the number of mismatches (0 expected) and the
// number of pairs checked.
#include <cstdint>
#include <cstdio>

#include "fastdiv.h"

int main() {
    uint64_t bad = 0, n_checked = 0;
    uint64_t state = 0x9e3779b97f4a7c15ull;
    auto next = [&]() {   // xorshift64*
        state ^= state >> 12; state ^= state << 25; state ^= state >> 27;
        return static_cast<uint32_t>((state * 0x2545f4914f6cdd1dull) >> 32);
    };
    auto check = [&](uint32_t n, const moe::FastDiv& f) {
        ++n_checked;
        if (moe::fastdiv(n, f) != n / f.d) {
            if (bad < 8) std::printf("mismatch n=%u d=%u got=%u want=%u\n", n, f.d, moe::fastdiv(n, f), n / f.d);
            ++bad;
        }
    };
    uint32_t divisors[4096 + 8];
    int nd = 0;
    for (uint32_t d = 1; d <= 4096; ++d) divisors[nd++] = d;
    const uint32_t big[] = {65535u, 65536u, 65537u, 1000003u, 0x7fffffffu, 0x80000000u, 12345679u, 3u << 29};
    for (uint32_t d : big) divisors[nd++] = d;
    for (int i = 0; i < nd; ++i) {
        const moe::FastDiv f = moe::make_fastdiv(divisors[i]);
        const uint32_t d = divisors[i];
        for (uint32_t n = 0; n < 4096; ++n) check(n, f);
        for (uint32_t q = 1; q < 2048; ++q) {              // both sides of q * d
            const uint64_t b = static_cast<uint64_t>(q) * d;
            if (b + 1 > 0xffffffffull) break;
            check(static_cast<uint32_t>(b - 1), f);
            check(static_cast<uint32_t>(b), f);
            check(static_cast<uint32_t>(b + 1), f);
        }
        for (int k = 0; k < 2000; ++k) check(next(), f);
        for (uint32_t n = 0xffffffffu - 4096u; n != 0; ++n) check(n, f);    // the top of the range
    }
    std::printf("%llu %llu\n", static_cast<unsigned long long>(bad), static_cast<unsigned long long>(n_checked));
    return bad == 0 ? 0 : 1;
}
